// decode_tma.cu -- the HBM-streaming fused BitDelta linear for small token
// counts, fed by TMA.  Same arithmetic as decode.cu (distributive form
// y = x.W_base^T + alpha * (x.S^T) on mma.m16n8k16, signs built in registers),
// but W_base, the packed bits and the activations arrive through a multi-stage
// ring of shared-memory tiles filled by one producer warp with cp.async.bulk.tensor,
// so each SM keeps tens of KB of HBM reads in flight for a handful of
// instructions, and two CTAs fit on an SM.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": one fused kernel reads
// the base weights and the delta bits together and rebuilds the effective
// weight on chip, never writing W_eff to HBM (conceptual fused_bitdelta_linear
// listing).
//
// CTA: 8 consumer warps + 1 producer warp; 64 W rows; a stage is a 128-column
// K step: two 64x64 bf16 W boxes (128-byte swizzle), one 64x16-byte box of
// packed bits and two (8*NT tokens x 64 columns) activation boxes (128-byte
// swizzle; rows beyond m arrive as zeros).  Consumer warp w owns row group w%4 (16 rows, the M side of the
// MMA) and 64-column half w/4 of every stage.  Lane (g, t) reads 16-byte
// chunks 2t and 2t+1 of rows g and g+8 -- with the swizzle the eight lanes of a
// shared-memory phase hit eight different bank groups -- so its 16 columns are
// 16t..16t+15 of the half, and the k-slots of the four MMAs per half map to
// those columns in order, identically for the activations.  A cluster of C
// CTAs splits K; partials are added across the two halves in shared memory and
// across the cluster through distributed shared memory, in a fixed order.
// Launches allow programmatic dependent launch: the next kernel on the stream
// may start its prologue while this one drains.  Every global read comes after
// griddepcontrol.wait, so data written by the previous kernel is seen -- except,
// when the caller enabled weight prefetch, the first stages' W_base and bits
// boxes, which are issued before the wait.
#include <cooperative_groups.h>

#include <cstdlib>

#include "bd_device.cuh"
#include "bd_internal.h"

namespace cg = cooperative_groups;

namespace bd {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // 288
constexpr int kRows = 64;                            // W rows per CTA
constexpr int kStepK = 128;                          // K columns per stage
constexpr uint32_t kBoxBytes = 64 * 64 * 2;          // one 64-row x 64-column bf16 box
constexpr uint32_t kBitsBytes = kRows * 16;          // 64 rows x 16 packed bytes (128 columns)

// Per token-tile count NT (8 tokens each): ring depth, and the stage layout
// [W box k0..63][W box k64..127][bits][x box k0..63][x box k64..127]; every box
// starts on a 1024-byte boundary (the 128-byte swizzle pattern repeats there).
template <int NT> struct Ring {
    static constexpr int kStages = NT == 1 ? 5 : NT == 2 ? 4 : NT == 4 ? 7 : 6;
    static constexpr uint32_t kXBox = 8 * NT * 128;  // MP tokens x 64 columns
    static constexpr uint32_t kStageBytes = 2 * kBoxBytes + kBitsBytes + 2 * kXBox;
    static constexpr uint32_t kRedBytes = 8 * NT * kRows * 4;
    static constexpr size_t kSmem = 1024 + kStages * kStageBytes + kRedBytes + 2 * kStages * 8 + 16;
};

struct TmaDecodeArgs {
    const float *alpha;
    uint16_t *y;
    int64_t m, n_out, n_in;
    int64_t ks;
    int32_t mode;
    int32_t cluster;
    int32_t prefetch_weights;  // issue the first stages' W and bits boxes before griddepcontrol.wait
    unsigned *status;
    uint64_t wait_ns;
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

__device__ __forceinline__ void give_up(volatile int *abort_flag, unsigned *status) {
    *abort_flag = 1;
    flag_status(status, kDevTimeout);
}

template <int NT>
__global__ void __launch_bounds__(kThreads, NT <= 2 ? 2 : 1)
    decode_tma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ TmaDecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int MP = 8 * NT;
    constexpr int kStages = Ring<NT>::kStages;
    constexpr uint32_t kStageBytes = Ring<NT>::kStageBytes;
    constexpr uint32_t kXBox = Ring<NT>::kXBox;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *red = reinterpret_cast<float *>(smem + kStages * kStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes + Ring<NT>::kRedBytes);
    uint64_t *empty = full + kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kStages);

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t row_block = blockIdx.x / a.cluster;
    const int row0 = static_cast<int>(row_block * kRows);
    const int64_t k_lo = static_cast<int64_t>(rank) * a.ks;
    const int64_t k_hi = min(k_lo + a.ks, a.n_in);
    const int n_steps = k_hi > k_lo ? static_cast<int>((k_hi - k_lo + kStepK - 1) / kStepK) : 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    pdl_trigger();
    const int n_pre = a.prefetch_weights ? min(n_steps, kStages) : 0;
    if (warp == kConsumerWarps && lane == 0 && n_pre > 0) {
        // Weights are not written by the preceding kernel (the caller's
        // promise): start streaming them before that kernel completes.
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_b);
        for (int i = 0; i < n_pre; ++i) {
            const int kc = static_cast<int>(k_lo) + i * kStepK;
            uint8_t *st = smem + i * kStageBytes;
            mbar_arrive_expect_tx(&full[i], kStageBytes);
            tma_load_2d(st, &tm_w, &full[i], kc, row0);
            tma_load_2d(st + kBoxBytes, &tm_w, &full[i], kc + 64, row0);
            tma_load_2d(st + 2 * kBoxBytes, &tm_b, &full[i], kc / 8, row0);
        }
    }
    pdl_wait();

    float accb[NT][4], accs[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) accb[i][j] = accs[i][j] = 0.0f;

    const int g = lane >> 2, t = lane & 3;
    const int rg = warp & 3;       // row group
    const int kh = warp >> 2;      // 64-column half of each stage
    const int r0 = rg * 16 + g;    // tile rows r0, r0 + 8

    if (warp == kConsumerWarps) {
        // ---- producer ----
        if (lane == 0) {
            tma_prefetch_desc(&tm_w);
            tma_prefetch_desc(&tm_b);
            tma_prefetch_desc(&tm_x);
            for (int i = 0; i < n_pre; ++i) {  // the activations of the prefetched stages
                const int kc = static_cast<int>(k_lo) + i * kStepK;
                uint8_t *st = smem + i * kStageBytes;
                tma_load_2d(st + 2 * kBoxBytes + kBitsBytes, &tm_x, &full[i], kc, 0);
                tma_load_2d(st + 2 * kBoxBytes + kBitsBytes + kXBox, &tm_x, &full[i], kc + 64, 0);
            }
            int issued = n_pre;
            for (int i = n_pre; i < n_steps; ++i) {
                const int s = i % kStages;
                const uint32_t ph = (i / kStages) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, a.wait_ns, abort_flag)) {
                    give_up(abort_flag, a.status);
                    break;
                }
                const int kc = static_cast<int>(k_lo) + i * kStepK;
                uint8_t *st = smem + s * kStageBytes;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                tma_load_2d(st, &tm_w, &full[s], kc, row0);
                tma_load_2d(st + kBoxBytes, &tm_w, &full[s], kc + 64, row0);
                tma_load_2d(st + 2 * kBoxBytes, &tm_b, &full[s], kc / 8, row0);
                tma_load_2d(st + 2 * kBoxBytes + kBitsBytes, &tm_x, &full[s], kc, 0);
                tma_load_2d(st + 2 * kBoxBytes + kBitsBytes + kXBox, &tm_x, &full[s], kc + 64, 0);
                issued = i + 1;
            }
            if (*abort_flag) {
                for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
                    mbar_wait(&full[i % kStages], (i / kStages) & 1, kDrainLimitNs, nullptr);
            }
        }
    } else {
        // ---- consumers ----
        // Token rows of the x boxes use the same swizzle term as W rows: (8*tt + g) & 7 == r0 & 7 == g.
        const uint32_t sw0 = static_cast<uint32_t>(((2 * t) ^ (r0 & 7)) << 4);
        const uint32_t sw1 = static_cast<uint32_t>(((2 * t + 1) ^ (r0 & 7)) << 4);  // rows r0, r0+8 share r&7
        for (int i = 0; i < n_steps; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (i / kStages) & 1;
            const bool got = mbar_wait(&full[s], ph, a.wait_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up(abort_flag, a.status);
                break;
            }
            const uint8_t *st = smem + s * kStageBytes;
            const uint8_t *box = st + kh * kBoxBytes;
            const uint4 wa0 = lds128(box + r0 * 128 + sw0);
            const uint4 wa1 = lds128(box + r0 * 128 + sw1);
            const uint4 wb0 = lds128(box + (r0 + 8) * 128 + sw0);
            const uint4 wb1 = lds128(box + (r0 + 8) * 128 + sw1);
            const uint8_t *bt = st + 2 * kBoxBytes;
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
            const uint8_t *xrow = st + 2 * kBoxBytes + kBitsBytes + kh * kXBox + g * 128;
            uint32_t xv[NT][8];
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                const uint4 p0 = lds128(xrow + tt * 1024 + sw0);
                const uint4 p1 = lds128(xrow + tt * 1024 + sw1);
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
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // ---- fold alpha, add the two halves ----
        const int64_t grow0 = static_cast<int64_t>(row0) + r0;
        const bool v0 = grow0 < a.n_out, v1 = grow0 + 8 < a.n_out;
        const float al0 = v0 ? (a.mode ? a.alpha[grow0] : a.alpha[0]) : 0.0f;
        const float al1 = v1 ? (a.mode ? a.alpha[grow0 + 8] : a.alpha[0]) : 0.0f;
        float part[NT][4];
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            part[tt][0] = accb[tt][0] + al0 * accs[tt][0];
            part[tt][1] = accb[tt][1] + al0 * accs[tt][1];
            part[tt][2] = accb[tt][2] + al1 * accs[tt][2];
            part[tt][3] = accb[tt][3] + al1 * accs[tt][3];
        }
        // red[token][row]: the upper half writes, the lower half adds its own and keeps the sum.
        if (kh == 1) {
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                const int c = 8 * tt + 2 * t;
                red[c * kRows + r0] = part[tt][0];
                red[(c + 1) * kRows + r0] = part[tt][1];
                red[c * kRows + r0 + 8] = part[tt][2];
                red[(c + 1) * kRows + r0 + 8] = part[tt][3];
            }
        }
        consumer_sync();
        if (kh == 0) {
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                const int c = 8 * tt + 2 * t;
                red[c * kRows + r0] += part[tt][0];
                red[(c + 1) * kRows + r0] += part[tt][1];
                red[c * kRows + r0 + 8] += part[tt][2];
                red[(c + 1) * kRows + r0 + 8] += part[tt][3];
            }
        }
    }
    cluster.sync();

    // ---- rank c sums rows [c*share, (c+1)*share) of the block over the cluster ----
    const int share = (kRows + a.cluster - 1) / a.cluster;
    const int m_here = static_cast<int>(a.m < MP ? a.m : MP);
    for (int i = threadIdx.x; i < share * m_here; i += kThreads) {
        const int tok = i / share;
        const int lr = rank * share + (i - tok * share);
        const int64_t row = static_cast<int64_t>(row0) + lr;
        if (lr < kRows && row < a.n_out) {
            float s = 0.0f;
            for (int q = 0; q < a.cluster; ++q) s += cluster.map_shared_rank(red, q)[tok * kRows + lr];
            __nv_bfloat16 h = __float2bfloat16_rn(s);
            a.y[static_cast<int64_t>(tok) * a.n_out + row] = *reinterpret_cast<uint16_t *>(&h);
        }
    }
    cluster.sync();
}

struct TmaPlan {
    int nt, cluster;
    int64_t ks, row_blocks;
};

int env_int(const char *name, int dflt) {
    const char *e = std::getenv(name);
    if (!e) return dflt;
    const int v = std::atoi(e);
    return v > 0 ? v : dflt;
}

bool make_tma_plan(int64_t m, int64_t n_out, int64_t n_in, int num_sms, TmaPlan &p) {
    if (m < 1 || m > kDecodeMaxM) return false;
    p.nt = m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8;
    p.row_blocks = (n_out + kRows - 1) / kRows;
    // Split K over a cluster only when the 64-row blocks alone leave SMs idle:
    // each split adds a reduction, an activation re-read and cluster placement
    // constraints.  Measured on GB300: one split when row blocks >= SMs; about
    // 1.5 CTAs per SM otherwise (4096 rows -> 4 splits).
    int c = 1;
    if (p.row_blocks < num_sms)
        c = static_cast<int>((3 * static_cast<int64_t>(num_sms) / 2 + p.row_blocks - 1) / p.row_blocks);
    c = env_int("BD_DECODE_CLUSTER", c);
    if (c < 1) c = 1;
    if (c > 8) c = 8;
    const int64_t steps = (n_in + kStepK - 1) / kStepK;
    if (c > steps) c = static_cast<int>(steps);
    const int64_t per = (steps + c - 1) / c;
    p.ks = per * kStepK;
    p.cluster = static_cast<int>((steps + per - 1) / per);  // no empty ranks
    return true;
}

template <int NT>
cudaError_t launch_nt(const CUtensorMap &tw, const CUtensorMap &tb, const CUtensorMap &tx, const TmaDecodeArgs &a,
                      const TmaPlan &p, const DevCtx &ctx, cudaStream_t stream) {
    static bool attr_set[128] = {false};
    if (ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e = cudaFuncSetAttribute(decode_tma_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(Ring<NT>::kSmem));
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.row_blocks * p.cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Ring<NT>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, decode_tma_kernel<NT>, tw, tb, tx, a);
}

}  // namespace

bool decode_tma_supported(int64_t m, int64_t n_out, int64_t n_in, const void *w_base, const uint8_t *bits,
                          int num_sms) {
    if (n_in % kStepK != 0) return false;  // packed-bit rows must be 16-byte multiples for TMA
    if ((reinterpret_cast<uintptr_t>(w_base) & 15) || (reinterpret_cast<uintptr_t>(bits) & 15)) return false;
    if (n_in >= (int64_t(1) << 31) - kStepK) return false;
    TmaPlan p;
    return make_tma_plan(m, n_out, n_in, num_sms, p);
}

cudaError_t launch_decode_tma(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                              int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                              cudaStream_t stream) {
    TmaPlan p;
    if (!make_tma_plan(m, n_out, n_in, ctx.num_sms, p)) return cudaErrorNotSupported;
    if (p.row_blocks * p.cluster > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    CUtensorMap tw, tb;
    if (!encode_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_base, n_in, n_out, n_in * 2, 64, kRows,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!encode_tensor_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, bits, n_in / 8, n_out, n_in / 8, 16, kRows,
                              CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    const int mp = 8 * p.nt;
    CUtensorMap tx;
    if (!encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, n_in, m, n_in * 2, 64,
                              static_cast<uint32_t>(mp), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    TmaDecodeArgs a;
    a.alpha = alpha;
    a.y = static_cast<uint16_t *>(y);
    a.m = m;
    a.n_out = n_out;
    a.n_in = n_in;
    a.ks = p.ks;
    a.mode = alpha_mode;
    a.cluster = p.cluster;
    a.prefetch_weights = ctx.weight_prefetch ? 1 : 0;
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;
    switch (p.nt) {
        case 1: return launch_nt<1>(tw, tb, tx, a, p, ctx, stream);
        case 2: return launch_nt<2>(tw, tb, tx, a, p, ctx, stream);
        case 4: return launch_nt<4>(tw, tb, tx, a, p, ctx, stream);
        default: return launch_nt<8>(tw, tb, tx, a, p, ctx, stream);
    }
}

}  // namespace bd
