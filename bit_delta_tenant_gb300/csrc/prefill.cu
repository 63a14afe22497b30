// prefill.cu -- fused BitDelta linear for large token counts on the 5th
// generation tensor cores: y = x . (W_base + alpha*S)^T with W_eff rebuilt
// tile by tile in shared memory and never written to HBM.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": the effective weight is
// rebuilt on the fly by a fused kernel that reads the base weights and the
// delta bits together, in registers or shared memory, and the reconstruction
// is fused with the matrix multiply (conceptual fused_bitdelta_linear
// listing: unpack to {-1,+1}, W_eff = W_base + alpha*unpacked, linear).
//
// One CTA computes a 128 (W rows) x 256 (tokens) tile of y^T:
//   warp 0      TMA producer: per 64-wide K block, the W_base tile
//               [128 x 64] and the x tile [256 x 64], both K-major with the
//               128-byte swizzle, into a 4-stage ring.
//   warps 2..9  reconstruction: two threads per tile row, each with half of
//               the row's 8 packed bytes for the K block (prefetched two
//               blocks ahead); each rebuilds its four 16-byte chunks of the
//               swizzled W tile as bf16(fp32(W_base) + alpha_r * s) -- one
//               chunk is exactly one packed byte.  After the K loop the same
//               warps are the epilogue (warp w reads TMEM lanes 32*(w%4)..+31,
//               two warps per lane quarter splitting the token columns).
//   warp 1      allocates TMEM (256 accumulator columns, plus 32 columns per
//               stage for the rebuilt A tile); lane 0 issues tcgen05.mma
//               kind::f16 (M=128, N=tokens<=256, K=16, bf16 in, fp32
//               accumulate in TMEM) and commits each stage back to the producer.
// The rebuilt tile goes from registers to tensor memory (tcgen05.st) and the
// MMA takes A from there, so shared memory carries only the TMA fills, the
// rebuild reads and the activation (B) operand; with BD_PREFILL_TMEM_A=0 the
// tile is instead written back in place and read by the MMA from shared memory.
// Every wait is bounded; a role that gives up records a timeout in the status
// word, tells the other roles through a shared flag, drains its own copies
// and MMAs in flight, and the CTA frees its TMEM and returns.
#include <cstdlib>

#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {
namespace {

constexpr int kBM = 128;  // W rows per tile (MMA M)
constexpr int kBN = 256;  // tokens per tile (MMA N)
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr uint32_t kWBytes = kBM * kBK * 2;
constexpr uint32_t kXBytes = kBN * kBK * 2;
constexpr uint32_t kStageTx = kWBytes + kXBytes;
constexpr int kRebuildWarps = 8;
constexpr int kThreads = (2 + kRebuildWarps) * 32;  // producer, MMA issuer, rebuild/epilogue
constexpr uint32_t kAccCols = 256;  // fp32 accumulator columns (one per token)
constexpr size_t kSmemBytes = 1024 + kStages * (kWBytes + kXBytes) + 256;
constexpr int kMaxVariants = 64;

struct PrefillArgs {
    const uint8_t *bits;
    const float *alpha;
    uint16_t *y;
    int64_t m, n_out, n_in;
    int32_t mode;
    int32_t num_kb;
    int32_t row_tiles, tok_tiles, group;
    int32_t bits_vec8;  // rows of packed bits are 8-byte aligned
    unsigned *status;
    uint64_t wait_ns;
    // Multi-tenant mode only: token tiles come from a device-built table of
    // (variant, first row in the variant-sorted activations, row count), and
    // output rows are scattered back to the original token order through perm.
    const int32_t *tiles;
    const int32_t *n_tiles;
    const int32_t *perm;
    int32_t max_slots;
    const uint8_t *vbits[kMaxVariants];
    const float *valpha[kMaxVariants];
    int32_t vmode[kMaxVariants];
};

// One bf16 pair of W_eff = bf16(fp32(W_base) + alpha * s): the sign bit of
// -alpha is cleared where the packed bit is 1 (+alpha) and kept where it is 0.
template <int I>
__device__ __forceinline__ uint32_t rebuild_pair(uint32_t w, uint32_t byte, uint32_t neg_alpha_bits) {
    const uint32_t s_lo = ((byte << (31 - 2 * I)) & 0x80000000u) ^ neg_alpha_bits;
    const uint32_t s_hi = ((byte << (30 - 2 * I)) & 0x80000000u) ^ neg_alpha_bits;
    const float lo = bf16lo_to_f32(w) + __uint_as_float(s_lo);
    const float hi = bf16hi_to_f32(w) + __uint_as_float(s_hi);
    return pack_bf16x2(lo, hi);
}

__device__ __forceinline__ void give_up(volatile int *abort_flag, unsigned *status) {
    *abort_flag = 1;
    flag_status(status, kDevTimeout);
}

template <bool kGrouped, bool kTmemA>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // With kTmemA the rebuilt W tile goes to tensor memory (columns 256 + 32*stage)
    // and the MMA reads A from there; otherwise it is written back in place.
    constexpr uint32_t kTmemCols = kTmemA ? 512 : 256;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sW = smem;
    uint8_t *sX = smem + kStages * kWBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sX + kStages * kXBytes);
    uint64_t *full = bars;
    uint64_t *rebuilt = bars + kStages;
    uint64_t *empty = bars + 2 * kStages;
    uint64_t *acc_full = bars + 3 * kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    int m0, n0, count;
    const uint8_t *bits;
    const float *alpha;
    int32_t mode;
    if constexpr (kGrouped) {
        // Consecutive CTAs take every token tile of one W row tile, so the W
        // tile is read from HBM once per wave and reused from L2.
        const int row_tile = blockIdx.x / a.max_slots;
        const int slot = blockIdx.x - row_tile * a.max_slots;
        if (slot >= *a.n_tiles) return;  // uniform across the CTA, before any barrier or TMEM use
        const int v = a.tiles[3 * slot];
        m0 = row_tile * kBM;
        n0 = a.tiles[3 * slot + 1];
        count = a.tiles[3 * slot + 2];
        bits = a.vbits[v];
        alpha = a.valpha[v];
        mode = a.vmode[v];
    } else {
        // Grouped rasterisation: consecutive CTAs cycle over `group` token tiles
        // for one W tile, so a wave touches a compact block of W and x in L2.
        const int tile = blockIdx.x;
        const int per_group = a.group * a.row_tiles;
        const int grp = tile / per_group;
        const int rem = tile - grp * per_group;
        const int gsize = min(a.group, a.tok_tiles - grp * a.group);
        const int tok_tile = grp * a.group + rem % gsize;
        const int row_tile = rem / gsize;
        m0 = row_tile * kBM;
        n0 = tok_tile * kBN;
        count = static_cast<int>(min(static_cast<int64_t>(kBN), a.m - n0));
        bits = a.bits;
        alpha = a.alpha;
        mode = a.mode;
    }
    // MMA N: the tile's token count rounded up to the 16-column granule of M=128.
    const int n_mma = (count + 15) & ~15;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nkb = a.num_kb;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&rebuilt[s], kRebuildWarps);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_x);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kStages;
                const uint32_t ph = (kb / kStages) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, a.wait_ns, abort_flag)) {
                    give_up(abort_flag, a.status);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], kStageTx);
                tma_load_2d(sW + s * kWBytes, &tm_w, &full[s], kb * kBK, m0);
                tma_load_2d(sX + s * kXBytes, &tm_x, &full[s], kb * kBK, n0);
                issued = kb + 1;
            }
            if (*abort_flag) {
                // Drain: the loads of the last stages issued must land before the CTA exits.
                for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
                    mbar_wait(&full[kb % kStages], (kb / kStages) & 1, kDrainLimitNs, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, n_mma);
            bool ok = true;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kStages;
                const uint32_t ph = (kb / kStages) & 1;
                if (!mbar_wait(&rebuilt[s], ph, a.wait_ns, abort_flag)) {
                    give_up(abort_flag, a.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sW + s * kWBytes);
                const uint32_t b_addr = smem_u32(sX + s * kXBytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    if constexpr (kTmemA)
                        tc_mma_f16_ts(tmem, tmem + kAccCols + s * (kBK / 2) + kk * 8,
                                      sw128_kmajor_desc(b_addr + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
                    else
                        tc_mma_f16_ss(tmem, sw128_kmajor_desc(a_addr + kk * 32),
                                      sw128_kmajor_desc(b_addr + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
                }
                tc_commit(&empty[s]);
            }
            // Always wait for this thread's MMAs before the CTA may free TMEM, even if
            // the epilogue gave up early (its wait can run out while MMAs still run).
            tc_commit(acc_full);
            (void)ok;
            mbar_wait(acc_full, 0, kDrainLimitNs, nullptr);
        }
    } else {
        // ---- rebuild (then epilogue) warps ------------------------------------------
        // Thread q owns tile row r = 32*(warp%4) + lane and chunk pair h (0..3):
        // the 16-byte chunks 2h, 2h+1 of the row in every K block (two packed
        // bytes).  Warp w may read TMEM lanes 32*(w%4)..+31 only, so the same
        // row mapping serves the epilogue, where h picks a quarter of the tokens.
        constexpr int kParts = kRebuildWarps / 4;        // threads per row
        constexpr int kChunks = 8 / kParts;              // chunks per thread per K block
        const int sub = warp & 3;
        const int h = (warp - 2) >> 2;
        const int r = sub * 32 + lane;
        const int64_t row = static_cast<int64_t>(m0) + r;
        const bool row_ok = row < a.n_out;
        const float al = row_ok ? (mode ? alpha[row] : alpha[0]) : 0.0f;
        const uint32_t neg_al = __float_as_uint(-al);
        const int64_t bpr = a.n_in / 8;
        const uint8_t *brow = bits + (row_ok ? row : 0) * bpr + kChunks * h;

        auto load_bits = [&](int kb) -> uint32_t {
            uint32_t v = 0;
            if (row_ok && kb < nkb) {
                const int64_t c0 = static_cast<int64_t>(kb) * 8 + kChunks * h;  // first packed byte
                if (a.bits_vec8 && c0 + kChunks <= bpr) {
                    const uint8_t *q = brow + static_cast<int64_t>(kb) * 8;
                    if constexpr (kChunks == 4) v = __ldg(reinterpret_cast<const uint32_t *>(q));
                    else if constexpr (kChunks == 2) v = __ldg(reinterpret_cast<const uint16_t *>(q));
                    else v = __ldg(q);
                } else {
                    for (int c = 0; c < kChunks; ++c)
                        if (c0 + c < bpr)
                            v |= static_cast<uint32_t>(__ldg(brow + static_cast<int64_t>(kb) * 8 + c)) << (8 * c);
                }
            }
            return v;
        };

        uint32_t b_cur = load_bits(0);
        uint32_t b_nxt = load_bits(1);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % kStages;
            const uint32_t ph = (kb / kStages) & 1;
            const uint32_t b_nn = load_bits(kb + 2);
            const bool got = mbar_wait(&full[s], ph, a.wait_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up(abort_flag, a.status);
                ok = false;
                break;
            }
            uint8_t *rowp = sW + s * kWBytes + r * 128;
            uint4 *p[kChunks];
            uint4 w[kChunks];
#pragma unroll
            for (int cc = 0; cc < kChunks; ++cc) {
                p[cc] = reinterpret_cast<uint4 *>(rowp + (((kChunks * h + cc) ^ (r & 7)) << 4));
                w[cc] = *p[cc];
            }
#pragma unroll
            for (int cc = 0; cc < kChunks; ++cc) {
                const uint32_t byte = (b_cur >> (8 * cc)) & 0xFFu;
                w[cc].x = rebuild_pair<0>(w[cc].x, byte, neg_al);
                w[cc].y = rebuild_pair<1>(w[cc].y, byte, neg_al);
                w[cc].z = rebuild_pair<2>(w[cc].z, byte, neg_al);
                w[cc].w = rebuild_pair<3>(w[cc].w, byte, neg_al);
                if constexpr (!kTmemA) *p[cc] = w[cc];
            }
            if constexpr (kTmemA) {
                static_assert(kChunks == 4, "one 16-column TMEM store per thread and K block");
                const uint32_t v[16] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w,
                                        w[2].x, w[2].y, w[2].z, w[2].w, w[3].x, w[3].y, w[3].z, w[3].w};
                tmem_st_32x32b_x16(tmem + (static_cast<uint32_t>(sub * 32) << 16) + kAccCols + s * (kBK / 2) +
                                       16 * h,
                                   v);
                tmem_st_wait();
                tc_fence_before();
            } else {
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&rebuilt[s]);
            b_cur = b_nxt;
            b_nxt = b_nn;
        }

        if (ok) {
            const bool got = mbar_wait(acc_full, 0, a.wait_ns, abort_flag);
            if (__all_sync(0xFFFFFFFFu, got)) {
                tc_fence_after();
                const uint32_t lane_addr = tmem + (static_cast<uint32_t>(sub * 32) << 16);
                uint16_t *ycol = a.y + row;
#pragma unroll 1
                for (int c0 = h * (kBN / kParts); c0 < (h + 1) * (kBN / kParts); c0 += 32) {
                    if (c0 >= count) break;  // warp-uniform
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(lane_addr + c0, v);
                    tmem_ld_wait();
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            if (c0 + i < count) {
                                const int64_t t = kGrouped ? static_cast<int64_t>(a.perm[n0 + c0 + i])
                                                           : static_cast<int64_t>(n0) + c0 + i;
                                __nv_bfloat16 hv = __float2bfloat16_rn(__uint_as_float(v[i]));
                                ycol[t * a.n_out] = *reinterpret_cast<uint16_t *>(&hv);
                            }
                        }
                    }
                }
            } else if (lane == 0) {
                give_up(abort_flag, a.status);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace {

template <bool kGrouped, bool kTmemA>
cudaError_t set_smem_attr(const DevCtx &ctx) {
    static bool attr_set[128] = {false};
    if (ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<kGrouped, kTmemA>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    return cudaSuccess;
}

// The rebuilt W tile feeds the MMA from tensor memory by default (measured
// ~19% faster on GB300 than writing it back to shared memory, which then
// carries only the TMA fills, the rebuild reads and the activation operand);
// BD_PREFILL_TMEM_A=0 selects the shared-memory form.
bool use_tmem_a() {
    static const bool v = [] {
        const char *e = std::getenv("BD_PREFILL_TMEM_A");
        return !(e != nullptr && e[0] == '0');
    }();
    return v;
}

void fill_common(PrefillArgs &a, int64_t m, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx) {
    a.y = static_cast<uint16_t *>(y);
    a.m = m;
    a.n_out = n_out;
    a.n_in = n_in;
    a.num_kb = static_cast<int32_t>((n_in + kBK - 1) / kBK);
    a.row_tiles = static_cast<int32_t>((n_out + kBM - 1) / kBM);
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;
}

bool make_maps(CUtensorMap &tm_w, CUtensorMap &tm_x, const void *w_base, const void *x, int64_t x_rows,
               int64_t n_out, int64_t n_in) {
    return encode_tensor_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_base, n_in, n_out, n_in * 2, kBK, kBM,
                                CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, n_in, x_rows, n_in * 2, kBK, kBN,
                                CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

cudaError_t launch_prefill(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                           int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                           cudaStream_t stream) {
    const bool tmem_a = use_tmem_a();
    cudaError_t e = tmem_a ? set_smem_attr<false, true>(ctx) : set_smem_attr<false, false>(ctx);
    if (e != cudaSuccess) return e;
    CUtensorMap tm_w, tm_x;
    if (!make_maps(tm_w, tm_x, w_base, x, m, n_out, n_in)) return cudaErrorInvalidValue;
    PrefillArgs a = {};
    fill_common(a, m, n_out, n_in, y, ctx);
    a.bits = bits;
    a.alpha = alpha;
    a.mode = alpha_mode;
    a.tok_tiles = static_cast<int32_t>((m + kBN - 1) / kBN);
    a.group = a.tok_tiles < 8 ? a.tok_tiles : 8;
    a.bits_vec8 = ((n_in / 8) % 8 == 0 && (reinterpret_cast<uintptr_t>(bits) & 7) == 0) ? 1 : 0;
    const int64_t tiles = static_cast<int64_t>(a.row_tiles) * a.tok_tiles;
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    if (tmem_a)
        prefill_kernel<false, true><<<static_cast<unsigned>(tiles), kThreads, kSmemBytes, stream>>>(tm_w, tm_x, a);
    else
        prefill_kernel<false, false><<<static_cast<unsigned>(tiles), kThreads, kSmemBytes, stream>>>(tm_w, tm_x, a);
    return cudaGetLastError();
}

cudaError_t launch_prefill_grouped(const void *x_sorted, int64_t m, const void *w_base, const GroupedVariants &vars,
                                   int64_t n_out, int64_t n_in, void *y, const GroupTable &tab, const DevCtx &ctx,
                                   cudaStream_t stream) {
    const bool tmem_a = use_tmem_a();
    cudaError_t e = tmem_a ? set_smem_attr<true, true>(ctx) : set_smem_attr<true, false>(ctx);
    if (e != cudaSuccess) return e;
    CUtensorMap tm_w, tm_x;
    if (!make_maps(tm_w, tm_x, w_base, x_sorted, m, n_out, n_in)) return cudaErrorInvalidValue;
    PrefillArgs a = {};
    fill_common(a, m, n_out, n_in, y, ctx);
    bool vec8 = (n_in / 8) % 8 == 0;
    for (int v = 0; v < vars.count; ++v) {
        a.vbits[v] = vars.bits[v];
        a.valpha[v] = vars.alpha[v];
        a.vmode[v] = vars.mode[v];
        vec8 = vec8 && (reinterpret_cast<uintptr_t>(vars.bits[v]) & 7) == 0;
    }
    a.bits_vec8 = vec8 ? 1 : 0;
    a.tiles = tab.tiles;
    a.n_tiles = tab.n_tiles;
    a.perm = tab.perm;
    a.max_slots = tab.max_slots;
    const int64_t grid = static_cast<int64_t>(a.row_tiles) * tab.max_slots;
    if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    if (tmem_a)
        prefill_kernel<true, true><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tm_w, tm_x, a);
    else
        prefill_kernel<true, false><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tm_w, tm_x, a);
    return cudaGetLastError();
}

}  // namespace bd
