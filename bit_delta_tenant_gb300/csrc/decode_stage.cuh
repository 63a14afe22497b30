// decode_stage.cuh -- the shared-memory stage layout and the per-stage
// arithmetic of the two HBM-streaming fused-linear kernels: decode_tma.cu
// (one tile per CTA, K split over a thread-block cluster) and decode_batch.cu
// (a list of linears split evenly over the resident CTAs).
//
// Arithmetic: the distributive form y = x.W_base^T + alpha * (x.S^T) of
// "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU" (Hanzo blog),
// section "Le fondement mathématique", on mma.m16n8k16 with W rows on the M
// side and tokens on the N side: W_base enters as stored, the signs enter as
// exact bf16 +-1 pairs built in registers, and alpha is applied once to the
// fp32 sign sum, so no W_eff value is ever rounded.
#pragma once

#include "bd_device.cuh"

namespace bd {
namespace dstage {

constexpr int kStepK = 128;  // K columns per stage

// Stage layout for R row groups (rows = 16R) and NT token tiles (MP = 8NT):
// [W box k0..63: rows x 128 B][W box k64..127][bits: rows x 16 B, padded to
// 1 KB][x box k0..63: MP x 128 B][x box k64..127]; every box starts on a
// 1024-byte boundary (the 128-byte swizzle pattern repeats there).
struct StageLayout {
    uint32_t w_box, bits_off, bits_bytes, x_off, x_box, stage, tx;
};
__host__ __device__ constexpr StageLayout stage_layout(int rg, int nt) {
    StageLayout L{};
    const uint32_t rows = 16u * rg;
    L.w_box = rows * 128u;
    L.bits_off = 2u * L.w_box;
    L.bits_bytes = rows * 16u;
    L.x_off = L.bits_off + (L.bits_bytes + 1023u) / 1024u * 1024u;
    L.x_box = 1024u * nt;
    L.stage = L.x_off + 2u * L.x_box;
    L.tx = 2u * L.w_box + L.bits_bytes + 2u * L.x_box;  // bytes the copies deliver
    return L;
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// Swizzled byte offsets of the two 16-byte chunks (2t, 2t+1) lane (g, t) reads
// from rows r with r & 7 == r0 & 7 (W rows r0, r0 + 8 and token rows 8i + g).
struct LaneSwizzle {
    uint32_t sw0, sw1;
};
__device__ __forceinline__ LaneSwizzle lane_swizzle(int t, int r0) {
    return {static_cast<uint32_t>(((2 * t) ^ (r0 & 7)) << 4), static_cast<uint32_t>(((2 * t + 1) ^ (r0 & 7)) << 4)};
}

// One stage for a consumer warp: rows r0, r0 + 8 of its row group, the 64
// columns of K half kh.  accb += x.W_base^T, accs += x.S^T over those columns
// for NT tiles of 8 tokens.  Lane (g, t) takes columns 16t..16t+15 of the
// half; the k-slots of the four MMAs map to those columns in order,
// identically for W and the activations.
template <int NT>
__device__ __forceinline__ void consume_stage(const uint8_t *st, const StageLayout &L, int kh, int r0, int g, int t,
                                              const LaneSwizzle &sw, float (&accb)[NT][4], float (&accs)[NT][4]) {
    const uint8_t *box = st + kh * L.w_box;
    const uint4 wa0 = lds128(box + r0 * 128 + sw.sw0);
    const uint4 wa1 = lds128(box + r0 * 128 + sw.sw1);
    const uint4 wb0 = lds128(box + (r0 + 8) * 128 + sw.sw0);
    const uint4 wb1 = lds128(box + (r0 + 8) * 128 + sw.sw1);
    const uint8_t *bt = st + L.bits_off;
    const uint32_t ba = *reinterpret_cast<const uint16_t *>(bt + r0 * 16 + kh * 8 + 2 * t);
    const uint32_t bb = *reinterpret_cast<const uint16_t *>(bt + (r0 + 8) * 16 + kh * 8 + 2 * t);
    const uint32_t ba0 = ba & 0xFFu, ba1 = ba >> 8, bb0 = bb & 0xFFu, bb1 = bb >> 8;
    // signs of columns 16t + 0..15 of this half, as bf16 +-1 pairs
    const uint32_t sa[8] = {sign_pair_bf16<0>(ba0), sign_pair_bf16<1>(ba0), sign_pair_bf16<2>(ba0),
                            sign_pair_bf16<3>(ba0), sign_pair_bf16<0>(ba1), sign_pair_bf16<1>(ba1),
                            sign_pair_bf16<2>(ba1), sign_pair_bf16<3>(ba1)};
    const uint32_t sb[8] = {sign_pair_bf16<0>(bb0), sign_pair_bf16<1>(bb0), sign_pair_bf16<2>(bb0),
                            sign_pair_bf16<3>(bb0), sign_pair_bf16<0>(bb1), sign_pair_bf16<1>(bb1),
                            sign_pair_bf16<2>(bb1), sign_pair_bf16<3>(bb1)};
    const uint32_t wa[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w};
    const uint32_t wb[8] = {wb0.x, wb0.y, wb0.z, wb0.w, wb1.x, wb1.y, wb1.z, wb1.w};
    const uint8_t *xrow = st + L.x_off + kh * L.x_box + g * 128;
    uint32_t xv[NT][8];
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
        const uint4 p0 = lds128(xrow + tt * 1024 + sw.sw0);
        const uint4 p1 = lds128(xrow + tt * 1024 + sw.sw1);
        xv[tt][0] = p0.x, xv[tt][1] = p0.y, xv[tt][2] = p0.z, xv[tt][3] = p0.w;
        xv[tt][4] = p1.x, xv[tt][5] = p1.y, xv[tt][6] = p1.z, xv[tt][7] = p1.w;
    }
    // k-slice outer, tiles inner: consecutive MMAs never share an accumulator
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            mma_bf16_16816(accb[tt], wa[2 * j], wb[2 * j], wa[2 * j + 1], wb[2 * j + 1], xv[tt][2 * j],
                           xv[tt][2 * j + 1]);
            mma_bf16_16816(accs[tt], sa[2 * j], sb[2 * j], sa[2 * j + 1], sb[2 * j + 1], xv[tt][2 * j],
                           xv[tt][2 * j + 1]);
        }
    }
}

// part = accb + alpha * accs for this lane's accumulator elements (rows r, r + 8).
template <int NT>
__device__ __forceinline__ void fold_alpha(const float (&accb)[NT][4], const float (&accs)[NT][4], float al0,
                                           float al1, float (&part)[NT][4]) {
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
        part[tt][0] = accb[tt][0] + al0 * accs[tt][0];
        part[tt][1] = accb[tt][1] + al0 * accs[tt][1];
        part[tt][2] = accb[tt][2] + al1 * accs[tt][2];
        part[tt][3] = accb[tt][3] + al1 * accs[tt][3];
    }
}

// The two K halves meet in red[token][row] (rows = 16R): the upper half
// writes, then (after a barrier of the consumer warps) the lower half adds
// its own and keeps the sum.  Lane (g, t) of the MMA holds tokens 8tt + 2t,
// 8tt + 2t + 1 of rows r0 and r0 + 8.
template <int NT>
__device__ __forceinline__ void halves_store(float *red, int rows, int r0, int t, const float (&part)[NT][4]) {
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
        const int c = 8 * tt + 2 * t;
        red[c * rows + r0] = part[tt][0];
        red[(c + 1) * rows + r0] = part[tt][1];
        red[c * rows + r0 + 8] = part[tt][2];
        red[(c + 1) * rows + r0 + 8] = part[tt][3];
    }
}
template <int NT>
__device__ __forceinline__ void halves_add(float *red, int rows, int r0, int t, const float (&part)[NT][4]) {
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
        const int c = 8 * tt + 2 * t;
        red[c * rows + r0] += part[tt][0];
        red[(c + 1) * rows + r0] += part[tt][1];
        red[c * rows + r0 + 8] += part[tt][2];
        red[(c + 1) * rows + r0 + 8] += part[tt][3];
    }
}

}  // namespace dstage
}  // namespace bd
