// grouped_decode.cu -- the multi-tenant fused linear for small batches (m <= 64
// tokens, up to 16 variants): one HBM pass over the shared W_base and over
// every variant's packed bits, fed by TMA.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": the variants share one
// resident W_base and each request's delta is applied on the fly, never
// writing W_eff to HBM.
//
// Arithmetic (exact distributive form, fp32 alpha): for token t of variant v,
//     y[t, j] = sum_k x[t,k] W_base[j,k]  +  alpha_v(j) * sum_k x[t,k] s^v_jk.
// The base sum is one product over all tokens (in variant-sorted order, tiles
// of 8 tokens); the sign sum runs per variant over 8-token tiles of that
// variant's tokens, with the variant's signs built in registers (two integer
// ops per pair); alpha, constant along k, multiplies the full fp32 sign sum.  Both run on
// mma.m16n8k16 (W rows on the M side), like the single-variant streaming kernel.
//
// CTA: 16 warps, each also issuing part of the TMA; 64 W rows.  A ring stage is a
// 128-column K step: two 64x64 W boxes, two (tokens x 64) activation boxes
// (128-byte swizzle) and one 64x16-byte packed-bit box per variant.  For the
// base product warp w owns row group w%4 and every fourth token tile (w/4);
// for the sign products it owns sign tiles w and w + 16, each over all four row
// groups, so a tile's activation fragment is loaded once per half step and
// feeds four independent accumulator chains.  Lane (g, t) reads 16-byte chunks
// 2t, 2t+1 of its rows and of the activation rows, so the MMA k-slots map to
// columns 16t..16t+15 of the half.  A cluster of C CTAs splits K; each token's base
// and sign parts meet in shared memory and the cluster's K slices are summed
// through distributed shared memory, then written to the original token rows.
#include <cooperative_groups.h>

#include <cstdlib>

#include "bd_device.cuh"
#include "bd_internal.h"

namespace cg = cooperative_groups;

namespace bd {
namespace {

constexpr int kConsumerWarps = 16;  // 4 row groups x 4 token-tile quarters
constexpr int kThreads = kConsumerWarps * 32;  // lane 0 of every warp also issues TMA boxes
constexpr int kRows = 64;
constexpr int kStepK = 128;
constexpr int kMaxVar = 16;
constexpr int kMaxS = 24;  // sign tiles of 8 tokens: m/8 + (variants present) <= 8 + 16
constexpr uint32_t kBoxBytes = 64 * 64 * 2;
constexpr uint32_t kBitsBox = kRows * 16;

// SIGN = true: the sign products only (the shared base product comes from the
// tensor-core kernel as fp32 and is added in the epilogue), so stages carry no W.
template <int NTB, bool SIGN>
struct GdRing {
    static constexpr uint32_t kXBox = NTB * 1024;  // 8*NTB token rows x 128 bytes
    static constexpr uint32_t kWBytes = SIGN ? 0 : 2 * kBoxBytes;
    static constexpr uint32_t kStageBytes = kWBytes + 2 * kXBox + kMaxVar * kBitsBox;
    static constexpr int kStages = SIGN ? 6 : NTB >= 4 ? 4 : 5;
    static constexpr uint32_t kRedBytes = 8 * NTB * kRows * 4;
    static constexpr uint32_t kTableBytes = kMaxVar * kRows * 4 + 3 * kMaxS * 4 + 16;
    static constexpr size_t kSmem = 1024 + kStages * kStageBytes + kRedBytes + kTableBytes + 2 * kStages * 8 + 24;
};

struct GdMaps {
    CUtensorMap w;
    CUtensorMap x;
    CUtensorMap b[kMaxVar];
};

struct GdArgs {
    const float *alpha[kMaxVar];
    int32_t mode[kMaxVar];
    int32_t nv;
    const int32_t *s_tiles;    // [kMaxS][3]: variant, first sorted row, rows (<= 8)
    const int32_t *n_s_tiles;
    const int32_t *perm;       // sorted row -> original token
    const int32_t *n_valid;    // tokens with a valid id
    uint16_t *y;
    const float *ybase;        // sign-only kernel: x . W_base^T in fp32, [sorted row][n_out]
    int64_t m, n_out, n_in, ks;
    int32_t cluster;
    unsigned *status;
    uint64_t wait_ns;
    uint32_t sign_mul[4];      // 2^(15-2I) + 2^(30-2I), I = 0..3
    int32_t test_stall;        // the first full-barrier wait is on a barrier nothing completes (tests)
};

__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// Sign pairs of 16 packed bits read as two bytes (byte loads zero-extend for
// free).  Pair I of a byte is ((byte * mul_I) & 0x80008000) ^ 0xBF80BF80 with
// mul_I = 2^(15-2I) + 2^(30-2I) (the two shifted copies never overlap).  The
// multipliers arrive as kernel parameters: a literal constant lets the
// compiler turn the product into shifts and adds on the integer ALU, which
// the sign expansion already saturates; a runtime multiplier keeps it a
// single multiply-add on the FMA pipe.
__device__ __forceinline__ uint32_t sign_pair_mul(uint32_t byte, uint32_t mul) {
    return ((byte * mul) & 0x80008000u) ^ 0xBF80BF80u;
}

__device__ __forceinline__ void signs8(const uint8_t *p, const uint32_t (&mul)[4], uint32_t (&s)[8]) {
    const uint32_t b0 = p[0], b1 = p[1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s[i] = sign_pair_mul(b0, mul[i]);
        s[4 + i] = sign_pair_mul(b1, mul[i]);
    }
}

template <int NTB, bool SIGN>
__global__ void __launch_bounds__(kThreads, 1)
    gdecode_kernel(const __grid_constant__ GdMaps maps, const __grid_constant__ GdArgs a) {
    using R = GdRing<NTB, SIGN>;
    constexpr int MP = 8 * NTB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *red = reinterpret_cast<float *>(smem + R::kStages * R::kStageBytes);
    float *alpha_s = red + R::kRedBytes / 4;                       // [kMaxVar][kRows]
    int32_t *tiles_s = reinterpret_cast<int32_t *>(alpha_s + kMaxVar * kRows);  // [kMaxS][3]
    int32_t *n_tiles_s = tiles_s + 3 * kMaxS;
    uint64_t *full = reinterpret_cast<uint64_t *>(
        smem + R::kStages * R::kStageBytes + R::kRedBytes + R::kTableBytes);
    uint64_t *empty = full + R::kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + R::kStages);
    uint64_t *never = empty + R::kStages + 1;  // completed by no one

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
        for (int s = 0; s < R::kStages; ++s) {
            mbar_init(&full[s], kConsumerWarps);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    pdl_trigger_and_wait();
    // Per-variant alpha of this CTA's rows and the sign-tile table, in shared memory.
    for (int i = threadIdx.x; i < a.nv * kRows; i += kThreads) {
        const int v = i / kRows, r = i - v * kRows;
        const int64_t row = static_cast<int64_t>(row0) + r;
        alpha_s[i] = row < a.n_out ? (a.mode[v] ? a.alpha[v][row] : a.alpha[v][0]) : 0.0f;
    }
    {
        const int n_valid_tiles = min(*a.n_s_tiles, kMaxS);
        // entries past the last tile become empty tiles (no tokens) so pairs need no branch
        if (threadIdx.x < 3 * kMaxS) tiles_s[threadIdx.x] = threadIdx.x < 3 * n_valid_tiles ? a.s_tiles[threadIdx.x] : 0;
        if (threadIdx.x == 0) *n_tiles_s = n_valid_tiles;
    }
    __syncthreads();
    const int n_st = *n_tiles_s;

    const int g = lane >> 2, t = lane & 3;
    const int rg = warp & 3, tq = warp >> 2;  // row group, token-tile quarter
    const int r0 = rg * 16 + g;
    constexpr int NB = (NTB + 3) / 4;                              // base tiles tt = 4i + tq
    constexpr int NS = (kMaxS + kConsumerWarps - 1) / kConsumerWarps;  // sign tiles q = 16i + warp

    float accb[NB][4], accs[NS][4][4];  // accs[tile][row group][fragment]
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) accb[i][j] = 0.0f;
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int j = 0; j < 4; ++j) accs[i][r][j] = 0.0f;

    // ---- TMA issue, spread over the warps ----
    // A step's boxes are W(k), W(k+64), x(k), x(k+64) and one bits box per
    // variant; lane 0 of warp w issues boxes w and w + 16 and arrives on the
    // slot's full barrier (16 arrivals) with their byte count.  Step j goes to
    // slot j % kStages once all warps released that slot's previous step.  A
    // warp blocks only for the step it is about to consume; otherwise it
    // refills between its own steps without waiting.
    constexpr int nW = SIGN ? 0 : 2;  // W boxes first (none for the sign-only kernel), then x, then bits
    const int n_boxes = nW + 2 + a.nv;
    auto box_bytes = [&](int bx) -> uint32_t { return bx < nW ? kBoxBytes : bx < nW + 2 ? R::kXBox : kBitsBox; };
    const uint32_t my_tx = (warp < n_boxes ? box_bytes(warp) : 0u) + (warp + 16 < n_boxes ? box_bytes(warp + 16) : 0u);
    int issued = 0;
    auto issue_box = [&](int bx, int kc, uint8_t *st, uint64_t *bar) {
        if (bx < nW)
            tma_load_2d(st + bx * kBoxBytes, &maps.w, bar, kc + 64 * bx, row0);
        else if (bx < nW + 2)
            tma_load_2d(st + R::kWBytes + (bx - nW) * R::kXBox, &maps.x, bar, kc + 64 * (bx - nW), 0);
        else
            tma_load_2d(st + R::kWBytes + 2 * R::kXBox + (bx - nW - 2) * kBitsBox, &maps.b[bx - nW - 2], bar, kc / 8,
                        row0);
    };
    auto issue = [&](int j) {  // lane 0 only
        const int s = j % R::kStages;
        const int kc = static_cast<int>(k_lo) + j * kStepK;
        uint8_t *st = smem + s * R::kStageBytes;
        mbar_arrive_expect_tx(&full[s], my_tx);
        if (warp < n_boxes) issue_box(warp, kc, st, &full[s]);
        if (warp + 16 < n_boxes) issue_box(warp + 16, kc, st, &full[s]);
    };
    if (lane == 0) {
        if (warp == 0) {
            if (!SIGN) tma_prefetch_desc(&maps.w);
            tma_prefetch_desc(&maps.x);
        }
        if (warp >= nW + 2 && warp < n_boxes) tma_prefetch_desc(&maps.b[warp - nW - 2]);
        for (; issued < n_steps && issued < R::kStages; ++issued) issue(issued);
    }
    {
    // Constants of this warp's sign tiles q = 16i + warp (the same in every K step).  A warp
    // takes a tile over all four row groups, so the tile's activations are read once per
    // half-step and feed four independent accumulator chains.
    const uint32_t sw0 = static_cast<uint32_t>(((2 * t) ^ g) << 4);      // rows with (row & 7) == g
    const uint32_t sw1 = static_cast<uint32_t>(((2 * t + 1) ^ g) << 4);
    const int n_mine = n_st > warp ? (n_st - warp + kConsumerWarps - 1) / kConsumerWarps : 0;
    // A token row past its tile only feeds MMA column g, which the epilogue
    // drops, so it reads some in-box row instead of being zeroed.
    int x_off[NS], b_off[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int q = min(kConsumerWarps * i + warp, kMaxS - 1);  // the table's last entry past its end
        const int v = tiles_s[3 * q], start = tiles_s[3 * q + 1];
        const int xr = min(start + g, MP - 1);
        x_off[i] = xr * 128 + (((2 * t) ^ (xr & 7)) << 4);
        b_off[i] = v * kBitsBox + g * 16 + 2 * t;  // row group r adds 256 (16 rows of 16 bytes)
    }

    bool ok = true;
    for (int i = 0; i < n_steps; ++i) {
        const int s = i % R::kStages;
        if (lane == 0) {
            while (issued <= i) {  // this warp's part of the step is not in flight yet: wait for its slot
                if (!mbar_wait(&empty[issued % R::kStages], ((issued / R::kStages) & 1) ^ 1, a.wait_ns,
                               abort_flag)) {
                    *abort_flag = 1;
                    flag_status(a.status, kDevTimeout);
                    break;
                }
                issue(issued);
                ++issued;
            }
        }
        // The other lanes wait for lane 0's copies here, not on the full barrier: a lane spinning on
        // a barrier that only its own warp's lane 0 can complete may hold that lane back for long.
        __syncwarp();
        const bool got = mbar_wait(a.test_stall && i == 0 ? never : &full[s], (i / R::kStages) & 1, a.wait_ns,
                                   abort_flag);
        if (!__all_sync(0xFFFFFFFFu, got)) {
            if (lane == 0) {
                *abort_flag = 1;
                flag_status(a.status, kDevTimeout);
            }
            ok = false;
            break;
        }
        const uint8_t *st = smem + s * R::kStageBytes;
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
            const uint8_t *xbox = st + R::kWBytes + kh * R::kXBox;
            const uint8_t *bits = st + R::kWBytes + 2 * R::kXBox + kh * 8;
            if constexpr (!SIGN) {
            const uint8_t *box = st + kh * kBoxBytes;
            const uint4 wa0 = lds128(box + r0 * 128 + sw0), wa1 = lds128(box + r0 * 128 + sw1);
            const uint4 wb0 = lds128(box + (r0 + 8) * 128 + sw0), wb1 = lds128(box + (r0 + 8) * 128 + sw1);
            const uint32_t wa[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w};
            const uint32_t wb[8] = {wb0.x, wb0.y, wb0.z, wb0.w, wb1.x, wb1.y, wb1.z, wb1.w};
            // base: this warp's 8-token tiles of all tokens (sorted order)
#pragma unroll
            for (int ib = 0; ib < NB; ++ib) {
                const int tt = 4 * ib + tq;
                if (tt < NTB) {
                    const uint4 p0 = lds128(xbox + (8 * tt + g) * 128 + sw0);
                    const uint4 p1 = lds128(xbox + (8 * tt + g) * 128 + sw1);
                    const uint32_t xv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_bf16_16816(accb[ib], wa[2 * j], wb[2 * j], wa[2 * j + 1], wb[2 * j + 1], xv[2 * j],
                                       xv[2 * j + 1]);
                }
            }
            }
            // signs: this warp's tiles, each over the four row groups (rows 16r + g and 16r + g + 8)
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                if (i < n_mine) {
                    const uint4 p0 = lds128(xbox + x_off[i]);
                    const uint4 p1 = lds128(xbox + (x_off[i] ^ 16));  // chunk 2t+1: flip the chunk's low bit
                    const uint32_t xv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        uint32_t sa[8], sb[8];
                        signs8(bits + b_off[i] + 256 * r, a.sign_mul, sa);
                        signs8(bits + b_off[i] + 256 * r + 128, a.sign_mul, sb);  // row + 8
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_bf16_16816(accs[i][r], sa[2 * j], sb[2 * j], sa[2 * j + 1], sb[2 * j + 1], xv[2 * j],
                                           xv[2 * j + 1]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (lane == 0) {  // refill every slot already released, without waiting
            while (issued < n_steps &&
                   mbar_test_wait(&empty[issued % R::kStages], ((issued / R::kStages) & 1) ^ 1)) {
                issue(issued);
                ++issued;
            }
        }
    }
    if (lane == 0 && *abort_flag) {  // drain this warp's copies still in flight
        for (int i = (issued > R::kStages ? issued - R::kStages : 0); i < issued; ++i)
            mbar_wait(&full[i % R::kStages], (i / R::kStages) & 1, kDrainLimitNs, nullptr);
    }
    (void)ok;

    // ---- red[sorted token][row] = base + alpha * signs (each token in one base and one sign tile;
    //      the sign-only kernel adds its base in the cluster sum below) ----
    if constexpr (!SIGN) {
#pragma unroll
    for (int ib = 0; ib < NB; ++ib) {
        const int tt = 4 * ib + tq;
        if (tt < NTB) {
            float *p = red + (8 * tt + 2 * t) * kRows + r0;
            p[0] = accb[ib][0], p[kRows] = accb[ib][1], p[8] = accb[ib][2], p[kRows + 8] = accb[ib][3];
        }
    }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NS; ++i) {  // alpha is constant along k: applied once to the full sign sums
        const int q = kConsumerWarps * i + warp;
        if (q < n_st) {
            const int v = tiles_s[3 * q], start = tiles_s[3 * q + 1], cnt = tiles_s[3 * q + 2];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = 16 * r + g;
                const float al0 = alpha_s[v * kRows + row], al1 = alpha_s[v * kRows + row + 8];
                if (2 * t < cnt) {
                    float *p = red + (start + 2 * t) * kRows + row;
                    p[0] = (SIGN ? 0.0f : p[0]) + al0 * accs[i][r][0];
                    p[8] = (SIGN ? 0.0f : p[8]) + al1 * accs[i][r][2];
                }
                if (2 * t + 1 < cnt) {
                    float *p = red + (start + 2 * t + 1) * kRows + row;
                    p[0] = (SIGN ? 0.0f : p[0]) + al0 * accs[i][r][1];
                    p[8] = (SIGN ? 0.0f : p[8]) + al1 * accs[i][r][3];
                }
            }
        }
    }
    }
    cluster.sync();

    // ---- rank c sums rows [c*share, (c+1)*share) over the cluster; scatter to original tokens ----
    const int share = (kRows + a.cluster - 1) / a.cluster;
    const int n_tok = min(*a.n_valid, MP);
    for (int i = threadIdx.x; i < share * n_tok; i += kThreads) {
        const int tok = i / share;
        const int lr = rank * share + (i - tok * share);
        const int64_t row = static_cast<int64_t>(row0) + lr;
        if (lr < kRows && row < a.n_out) {
            float s = SIGN ? a.ybase[static_cast<int64_t>(tok) * a.n_out + row] : 0.0f;
            for (int q = 0; q < a.cluster; ++q) s += cluster.map_shared_rank(red, q)[tok * kRows + lr];
            __nv_bfloat16 h = __float2bfloat16_rn(s);
            const int64_t t = in_bounds(tok < a.m, a.status) ? a.perm[tok] : -1;
            if (in_bounds(t >= 0 && t < a.m, a.status))
                a.y[t * a.n_out + row] = *reinterpret_cast<uint16_t *>(&h);
        }
    }
    cluster.sync();
}

template <int NTB, bool SIGN>
cudaError_t launch_ntb(const GdMaps &maps, const GdArgs &a, int64_t row_blocks, const DevCtx &ctx,
                       cudaStream_t stream) {
    static bool attr_set[128] = {false};
    if (ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e = cudaFuncSetAttribute(gdecode_kernel<NTB, SIGN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(GdRing<NTB, SIGN>::kSmem));
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(row_blocks * a.cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = GdRing<NTB, SIGN>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gdecode_kernel<NTB, SIGN>, maps, a);
}

template <bool SIGN>
cudaError_t launch_sel(int ntb, const GdMaps &maps, const GdArgs &a, int64_t row_blocks, const DevCtx &ctx,
                       cudaStream_t stream) {
    switch (ntb) {
        case 1: return launch_ntb<1, SIGN>(maps, a, row_blocks, ctx, stream);
        case 2: return launch_ntb<2, SIGN>(maps, a, row_blocks, ctx, stream);
        case 4: return launch_ntb<4, SIGN>(maps, a, row_blocks, ctx, stream);
        default: return launch_ntb<8, SIGN>(maps, a, row_blocks, ctx, stream);
    }
}

}  // namespace

bool grouped_decode_supported(int64_t m, int32_t n_variants, int64_t n_in, const void *w_base,
                              const GroupedVariants &vars) {
    if (m < 1 || m > 64 || n_variants > kMaxVar || n_in % kStepK != 0) return false;
    if (m / 8 + (m < n_variants ? m : n_variants) + 1 > kMaxS) return false;
    if (reinterpret_cast<uintptr_t>(w_base) & 15) return false;
    for (int v = 0; v < vars.count; ++v)
        if (reinterpret_cast<uintptr_t>(vars.bits[v]) & 15) return false;
    return true;
}

cudaError_t launch_grouped_decode(const void *x_sorted, int64_t m, const void *w_base, const GroupedVariants &vars,
                                  int64_t n_out, int64_t n_in, void *y, const int32_t *s_tiles,
                                  const int32_t *n_s_tiles, const int32_t *perm, const int32_t *n_valid,
                                  const float *ybase, const DevCtx &ctx, cudaStream_t stream) {
    const int ntb = m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8;
    GdMaps maps;
    if (!encode_tensor_map_2d(&maps.w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_base, n_in, n_out, n_in * 2, 64, kRows,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!encode_tensor_map_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x_sorted, n_in, m, n_in * 2, 64,
                              static_cast<uint32_t>(8 * ntb), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GdArgs a = {};
    for (int v = 0; v < vars.count; ++v) {
        if (!encode_tensor_map_2d(&maps.b[v], CU_TENSOR_MAP_DATA_TYPE_UINT8, vars.bits[v], n_in / 8, n_out, n_in / 8,
                                  16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        a.alpha[v] = vars.alpha[v];
        a.mode[v] = vars.mode[v];
    }
    a.nv = vars.count;
    a.s_tiles = s_tiles;
    a.n_s_tiles = n_s_tiles;
    a.perm = perm;
    a.n_valid = n_valid;
    a.y = static_cast<uint16_t *>(y);
    a.ybase = ybase;
    a.m = m;
    a.n_out = n_out;
    a.n_in = n_in;
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;
    a.test_stall = ctx.test_stall ? 1 : 0;
    for (int i = 0; i < 4; ++i) a.sign_mul[i] = (1u << (15 - 2 * i)) + (1u << (30 - 2 * i));
    // K split over a cluster of c CTAs (one CTA per SM here): the c in 1..8 that minimises
    // waves x (K steps per CTA + a CTA's fixed cost of about 3 steps),
    // ceil(blocks * c / SMs) * (ceil(steps / c) + 3), the smallest on ties, with clusters above
    // four CTAs only when they fit in one wave (their scheduling costs more).  Fitted to GB300
    // measurements at 64 tokens, 14 variants: 14336 x 4096 164 us with c = 2 against 195 us
    // with c = 1; 4096 x 4096 61 us (c = 2) against 81 us (c = 3); 8192 x 8192 186 us (c = 1)
    // against 195 / 206 / 255 us (c = 2 / 4 / 8).  Clusters of 8 (one CTA per SM) cost more than
    // the model says: 1024 x 4096 takes 39.7 us with c = 8 against 30.2 us with c = 6, so c <= 6.
    const int64_t row_blocks = (n_out + kRows - 1) / kRows;
    const int64_t steps = n_in / kStepK;
    int64_t c = 1, best = -1;
    for (int64_t cc = 1; cc <= 6 && cc <= steps; ++cc) {
        if (cc > 4 && row_blocks * cc > ctx.num_sms) continue;  // clusters above 4 only in a single wave
        const int64_t cost = (row_blocks * cc + ctx.num_sms - 1) / ctx.num_sms * ((steps + cc - 1) / cc + 3);
        if (best < 0 || cost < best) best = cost, c = cc;
    }
    if (c > 8) c = 8;
    if (c > steps) c = steps;
    const int64_t per = (steps + c - 1) / c;
    a.ks = per * kStepK;
    a.cluster = static_cast<int32_t>((steps + per - 1) / per);
    if (row_blocks * a.cluster > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    return ybase != nullptr ? launch_sel<true>(ntb, maps, a, row_blocks, ctx, stream)
                            : launch_sel<false>(ntb, maps, a, row_blocks, ctx, stream);
}

}  // namespace bd
