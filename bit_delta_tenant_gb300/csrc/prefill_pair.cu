// prefill_pair.cu -- fused BitDelta linear for large token counts on CTA pairs:
// y = x . (W_base + alpha*S)^T with W_eff rebuilt tile by tile on chip and
// never written to HBM, one 256 (W rows) x 256 (tokens) output tile per pair
// of CTAs on the 5th-generation tensor cores (tcgen05, cta_group::2).
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": the effective weight is
// rebuilt on the fly by a fused kernel that reads the base weights and the
// delta bits together, in registers or shared memory, and the reconstruction
// is fused with the matrix multiply (conceptual fused_bitdelta_linear listing:
// unpack to {-1,+1}, W_eff = W_base + alpha*unpacked, linear).
//
// Why pairs: with one CTA per 128 x 256 tile, every 64-wide K step moves the
// whole 256-token activation tile into each SM's shared memory and the MMA
// reads all of it again; a pair's MMA (M = 256 over both CTAs' tensor memory)
// takes each CTA's half of the tokens from its own shared memory, so per SM
// the activation fill and the operand reads are halved for the same FLOPs.
//
// A cluster of two CTAs (rank r = 0, 1) computes W rows [256*i + 128*r, +128)
// of its tile in CTA r; per 64-wide K block:
//   warp 0      TMA producer of this CTA: the W_base tile [128 x 64] of its
//               own rows and its half of the token tile [N/2 x 64] (tokens
//               n0 + r*N/2 ...), both K-major with the 128-byte swizzle, into a
//               6-stage ring, completing on this CTA's full barrier.  No load
//               is multicast: each CTA reads its own halves.
//   warps 2..9  rebuild, in two groups of four taking alternate K blocks: one
//               thread per W row, W_eff = W_base + alpha_b*s as bf16 pairs (one
//               bf16x2 add per pair, alpha rounded to bf16), stored with
//               tcgen05.st into this CTA's tensor memory as the MMA's A operand;
//               then each warp arrives on the even CTA's "rebuilt" barrier.
//               After the K loop the same warps are the epilogue (TMEM lanes
//               32*(w%4)..+31, the groups splitting the token columns), writing
//               y in bf16.
//   warp 1      of the even CTA: one lane waits for both CTAs' rebuilt blocks
//               and issues tcgen05.mma.cta_group::2 kind::f16 (M = 256,
//               N = tokens <= 256, K = 16), committing each
//               stage to the empty barriers of both CTAs (multicast commit).
//               In both CTAs warp 1 allocates (and frees) the pair's tensor
//               memory: 256 accumulator columns plus 32 per ring stage of A.
// Every wait is bounded; a role that gives up records a timeout, its CTA
// drains its own copies (and, in the even CTA, its MMAs), and both CTAs meet
// at the closing cluster barrier before freeing tensor memory.
#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {
namespace {

constexpr int kPM = 128;                  // W rows per CTA (half of the pair MMA's M)
constexpr int kPN = 256;                  // tokens per pair tile (MMA N, at most)
constexpr int kPK = 64;                   // K per stage: one 128-byte swizzle row of bf16
constexpr int kPStages = 6;
constexpr uint32_t kPWBytes = kPM * kPK * 2;         // 16 KB
constexpr uint32_t kPXBytes = (kPN / 2) * kPK * 2;   // 16 KB: this CTA's half of the tokens
constexpr uint32_t kPStageTx = kPWBytes + kPXBytes;
constexpr uint32_t kPAccCols = kPN;                  // fp32 accumulator columns (one per token)
constexpr uint32_t kPTmemCols = 512;
constexpr int kPRebuildWarps = 8;
constexpr int kPThreads = (2 + kPRebuildWarps) * 32;
constexpr size_t kPSmem = 1024 + kPStages * (kPWBytes + kPXBytes) + 256;
static_assert(kPAccCols + kPStages * (kPK / 2) <= kPTmemCols, "accumulator + A stages fit in TMEM");

constexpr int kPMaxVariants = 64;
constexpr int kPMaxLinears = 8;  // independent linears per launch (a layer's q/k/v, gate/up)

// One linear of a launch: its pairs are [first_pair, first_pair + row_tiles * tok_tiles).
struct PairLinear {
    const uint8_t *bits;
    const float *alpha;
    uint16_t *y;
    int64_t m, n_out, n_in;
    int32_t mode;
    int32_t num_kb;
    int32_t row_tiles, tok_tiles, group;  // pair tiles: 256 W rows x 256 tokens
    int32_t bits_vec8;                    // rows of packed bits are 8-byte aligned
    int32_t first_pair;
};

struct PairMaps {
    CUtensorMap w[kPMaxLinears];  // W_base [n_out, n_in], boxes of 64 x 128 rows
    CUtensorMap x[kPMaxLinears];  // x [m, n_in], boxes of 64 x 128 token rows
};

struct PairArgs {
    PairLinear lin[kPMaxLinears];
    int32_t n_lin;
    unsigned *status;
    uint64_t wait_ns;
    // Multi-tenant mode only: token tiles come from a device-built table of
    // (variant, first row in the variant-sorted activations, row count <= 256);
    // consecutive pairs take every slot of one 256-row W tile, and output rows
    // are scattered back to the original token order through perm.
    const int32_t *tiles;
    const int32_t *n_tiles;
    const int32_t *perm;
    int32_t max_slots;
    const uint8_t *vbits[kPMaxVariants];
    const float *valpha[kPMaxVariants];
    int32_t vmode[kPMaxVariants];
};

template <int I>
__device__ __forceinline__ uint32_t rebuild_pair_b(uint32_t w, uint32_t byte, uint32_t neg_alpha2) {
    constexpr uint32_t mul = (1u << (15 - 2 * I)) + (1u << (30 - 2 * I));
    const uint32_t s = ((byte * mul) & 0x80008000u) ^ neg_alpha2;
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(s));
    return r;
}

__device__ __forceinline__ void give_up_p(volatile int *abort_flag, unsigned *status) {
    *abort_flag = 1;
    flag_status(status, kDevTimeout);
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

template <bool kGrouped>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_pair_kernel(const __grid_constant__ PairMaps maps, const __grid_constant__ PairArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sW = smem;
    uint8_t *sX = smem + kPStages * kPWBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sX + kPStages * kPXBytes);
    uint64_t *full = bars;                    // this CTA's TMA fills
    uint64_t *rebuilt = bars + kPStages;      // even CTA: both CTAs' rebuilt A blocks
    uint64_t *empty = bars + 2 * kPStages;    // the pair's MMAs of a stage are complete
    uint64_t *acc_full = bars + 3 * kPStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t rank = cluster_rank();
    int lp = 0;  // this pair's linear
    while (lp + 1 < a.n_lin && a.lin[lp + 1].first_pair <= static_cast<int>(blockIdx.x >> 1)) ++lp;
    const PairLinear &L = a.lin[lp];
    const CUtensorMap *tm_w = &maps.w[lp], *tm_x = &maps.x[lp];
    const int pair = static_cast<int>(blockIdx.x >> 1) - L.first_pair;
    int row_tile, n0, count;
    const uint8_t *bits;
    const float *alpha;
    int32_t mode;
    if constexpr (kGrouped) {
        // Consecutive pairs take every token tile of one W tile, so the W tile is
        // read from HBM once per wave and reused from L2.
        row_tile = pair / a.max_slots;
        const int slot = pair - row_tile * a.max_slots;
        if (slot >= *a.n_tiles) return;  // the same for both CTAs, before any barrier or TMEM use
        const int v = a.tiles[3 * slot];
        n0 = a.tiles[3 * slot + 1];
        count = a.tiles[3 * slot + 2];
        bits = a.vbits[v];
        alpha = a.valpha[v];
        mode = a.vmode[v];
    } else {
        // Grouped rasterisation: consecutive pairs cycle over `group` token tiles for
        // one W tile, so a wave touches a compact block of W and x in L2.
        const int per_group = L.group * L.row_tiles;
        const int grp = pair / per_group;
        const int rem = pair - grp * per_group;
        const int gsize = min(L.group, L.tok_tiles - grp * L.group);
        const int tok_tile = grp * L.group + rem % gsize;
        row_tile = rem / gsize;
        n0 = tok_tile * kPN;  // the pair's first token
        count = static_cast<int>(min(static_cast<int64_t>(kPN), L.m - n0));
        bits = L.bits;
        alpha = L.alpha;
        mode = L.mode;
    }
    const int m0 = row_tile * 2 * kPM + static_cast<int>(rank) * kPM;  // this CTA's W rows
    const int n_mma = (count + 15) & ~15;  // pair MMA N; each CTA holds n_mma / 2 token rows
    const int x_first = n0 + static_cast<int>(rank) * (n_mma / 2);
    const int nkb = L.num_kb;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&rebuilt[s], kPRebuildWarps);  // four warps of the block's group in each CTA
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(tm_w);
        tma_prefetch_desc(tm_x);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kPTmemCols);
        tmem_relinquish_pair();
    }
    // Barriers initialised and tensor memory allocated in both CTAs before any
    // remote arrive or multicast commit.
    tc_fence_before();
    cluster_arrive_release();
    cluster_wait_acquire();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kPStages;
                const uint32_t ph = (kb / kPStages) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, a.wait_ns, abort_flag)) {
                    give_up_p(abort_flag, a.status);
                    break;
                }
                mbar_arrive_expect_tx(&full[s], kPStageTx);
                tma_load_2d(sW + s * kPWBytes, tm_w, &full[s], kb * kPK, m0);
                tma_load_2d(sX + s * kPXBytes, tm_x, &full[s], kb * kPK, x_first);
                issued = kb + 1;
            }
            if (*abort_flag) {
                // the loads of the last stages issued land before the CTA may exit
                for (int kb = (issued > kPStages ? issued - kPStages : 0); kb < issued; ++kb)
                    mbar_wait(&full[kb % kPStages], (kb / kPStages) & 1, kDrainLimitNs, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = idesc_bf16_f32(2 * kPM, n_mma);
            // Every operand of every MMA (six ring stages x four 16-wide K slices) is computed
            // once here and the loop is unrolled by the ring depth, so that no address or
            // descriptor arithmetic sits between consecutive MMAs: measured on GB300, an MMA
            // whose descriptor is derived in the loop issues every ~250 clocks, one with a
            // precomputed descriptor every ~134 (M = 128, N = 256).
            uint64_t bdesc[kPStages][kPK / 16];
            uint32_t aaddr[kPStages][kPK / 16];
#pragma unroll
            for (int s = 0; s < kPStages; ++s)
#pragma unroll
                for (int kk = 0; kk < kPK / 16; ++kk) {
                    bdesc[s][kk] = sw128_kmajor_desc(smem_u32(sX + s * kPXBytes) + kk * 32);
                    aaddr[s][kk] = tmem + kPAccCols + s * (kPK / 2) + kk * 8;
                }
            bool ok = true;
            for (int ring = 0; ring < nkb && ok; ring += kPStages) {  // a ring's worth of K blocks at a time
#pragma unroll
                for (int s = 0; s < kPStages; ++s) {
                    const int kb = ring + s;
                    if (kb >= nkb) break;
                    const uint32_t ph = (ring / kPStages) & 1;
                    if (!mbar_wait(&rebuilt[s], ph, a.wait_ns, abort_flag)) {
                        give_up_p(abort_flag, a.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tc_mma_f16_ts_pair(tmem, aaddr[s][0], bdesc[s][0], idesc, kb != 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < kPK / 16; ++kk)
                        tc_mma_f16_ts_pair(tmem, aaddr[s][kk], bdesc[s][kk], idesc, 1u);
                    tc_commit_pair_mc(&empty[s], 0x3);
                }
            }
            // Always: both CTAs' epilogues wait for this, and this thread's MMAs are
            // complete before the pair may free tensor memory.
            tc_commit_pair_mc(acc_full, 0x3);
            mbar_wait(acc_full, 0, kDrainLimitNs, nullptr);
        }
    } else {
        // ---- rebuild (then epilogue) warps ------------------------------------------
        // Thread q of group h (warps 2..5: h = 0, warps 6..9: h = 1) owns tile row
        // r = 32*(warp%4) + lane: all eight 16-byte chunks of the row (its 8 packed
        // bytes) in the K blocks of parity h.  Warp w may access TMEM lanes
        // 32*(w%4)..+31 only, so the same row mapping serves the epilogue, where h
        // picks half of the token columns.
        const int sub = warp & 3;
        const int h = (warp - 2) >> 2;
        const int r = sub * 32 + lane;
        const int64_t row = static_cast<int64_t>(m0) + r;
        const bool row_ok = row < L.n_out;
        const float al = row_ok ? (mode ? alpha[row] : alpha[0]) : 0.0f;
        const uint32_t neg_al = pack_bf16x2(-al, -al);  // -alpha_b in both halves
        const int64_t bpr = L.n_in / 8;
        const uint8_t *brow = bits + (row_ok ? row : 0) * bpr;
        const uint32_t rebuilt0 = mapa_rank(smem_u32(rebuilt), 0);  // the even CTA's barriers
        const uint32_t a_lane = tmem + (static_cast<uint32_t>(sub * 32) << 16) + kPAccCols;

        auto load_bits = [&](int kb) -> uint2 {
            uint2 v = make_uint2(0u, 0u);
            const int64_t c0 = static_cast<int64_t>(kb) * 8;  // first packed byte of the block
            if (row_ok && kb < nkb) {
                if (L.bits_vec8 && c0 + 8 <= bpr) {
                    v = __ldg(reinterpret_cast<const uint2 *>(brow + c0));
                } else {
                    for (int c = 0; c < 8; ++c)
                        if (c0 + c < bpr) {
                            const uint32_t byte = __ldg(brow + c0 + c);
                            if (c < 4) v.x |= byte << (8 * c);
                            else v.y |= byte << (8 * (c - 4));
                        }
                }
            }
            return v;
        };

        // Packed bits arrive by plain loads three of this group's K blocks ahead.
        constexpr int kBitsAhead = 3;
        uint2 bq[kBitsAhead];
#pragma unroll
        for (int i = 0; i < kBitsAhead; ++i) bq[i] = load_bits(h + 2 * i);
        bool ok = true;
        for (int kb = h; kb < nkb; kb += 2) {
            const int s = kb % kPStages;
            const uint32_t ph = (kb / kPStages) & 1;
            const uint2 b_cur = bq[0];
#pragma unroll
            for (int i = 0; i + 1 < kBitsAhead; ++i) bq[i] = bq[i + 1];
            bq[kBitsAhead - 1] = load_bits(kb + 2 * kBitsAhead);
            const bool got = mbar_wait(&full[s], ph, a.wait_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up_p(abort_flag, a.status);
                ok = false;
                break;
            }
            const uint8_t *rowp = sW + s * kPWBytes + r * 128;
            uint32_t v[32];
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 w = *reinterpret_cast<const uint4 *>(rowp + ((cc ^ (r & 7)) << 4));
                const uint32_t byte = ((cc < 4 ? b_cur.x : b_cur.y) >> (8 * (cc & 3))) & 0xFFu;
                v[4 * cc + 0] = rebuild_pair_b<0>(w.x, byte, neg_al);
                v[4 * cc + 1] = rebuild_pair_b<1>(w.y, byte, neg_al);
                v[4 * cc + 2] = rebuild_pair_b<2>(w.z, byte, neg_al);
                v[4 * cc + 3] = rebuild_pair_b<3>(w.w, byte, neg_al);
            }
            tmem_st_32x32b_x32(a_lane + s * (kPK / 2), v);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(rebuilt0 + static_cast<uint32_t>(s) * 8u);
        }
        if (ok) {
            const bool got = mbar_wait(acc_full, 0, a.wait_ns, abort_flag);
            if (__all_sync(0xFFFFFFFFu, got)) {
                tc_fence_after();
                const uint32_t lane_addr = tmem + (static_cast<uint32_t>(sub * 32) << 16);
                uint16_t *ycol = L.y + row;
#pragma unroll 1
                for (int c0 = h * (kPN / 2); c0 < (h + 1) * (kPN / 2); c0 += 32) {
                    if (c0 >= count) break;  // warp-uniform
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(lane_addr + c0, v);
                    tmem_ld_wait();
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            if (c0 + i < count && in_bounds(n0 + c0 + i < L.m, a.status)) {
                                const int64_t t = kGrouped ? static_cast<int64_t>(a.perm[n0 + c0 + i])
                                                           : static_cast<int64_t>(n0) + c0 + i;
                                if (!in_bounds(t >= 0 && t < L.m, a.status)) continue;
                                __nv_bfloat16 hv = __float2bfloat16_rn(__uint_as_float(v[i]));
                                ycol[t * L.n_out] = *reinterpret_cast<uint16_t *>(&hv);
                            }
                        }
                    }
                }
            } else if (lane == 0) {
                give_up_p(abort_flag, a.status);
            }
        }
    }

    // Both CTAs are done with the pair's tensor memory (the even CTA's MMAs have
    // completed and every epilogue has read its accumulator) before it is freed.
    tc_fence_before();
    __syncthreads();
    cluster_arrive_release();
    cluster_wait_acquire();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kPTmemCols);
}

}  // namespace

bool prefill_pair_supported(int64_t m, int64_t n_out, int64_t n_in, const DevCtx &ctx) {
    if (m < 1 || n_out < 1 || n_in < 8 || ctx.num_sms < 2) return false;
    const int64_t pairs = ((n_out + 2 * kPM - 1) / (2 * kPM)) * ((m + kPN - 1) / kPN);
    return 2 * pairs <= 0x7FFFFFFFLL;
}

// Pair tiles of the shape: 256 W rows x 256 tokens.
int64_t prefill_pair_tiles(int64_t m, int64_t n_out) {
    return ((n_out + 2 * kPM - 1) / (2 * kPM)) * ((m + kPN - 1) / kPN);
}

namespace {

template <bool kGrouped>
cudaError_t launch_pair(const PairMaps &maps, const PairArgs &a, int64_t pairs, const DevCtx &ctx,
                        cudaStream_t stream) {
    static bool attr_set[128] = {false};
    if (ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel<kGrouped>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kPSmem));
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    if (pairs < 1) return cudaSuccess;
    if (2 * pairs > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<kGrouped>, maps, a);
}

// Shape, maps and tiling of linear i of a launch; returns false if a tensor map cannot be encoded.
bool fill_linear(PairMaps &maps, PairArgs &a, int i, const void *x, int64_t x_rows, const void *w_base,
                 const uint8_t *bits, const float *alpha, int32_t mode, int64_t m, int64_t n_out, int64_t n_in,
                 void *y, int32_t first_pair) {
    PairLinear &L = a.lin[i];
    L.bits = bits;
    L.alpha = alpha;
    L.y = static_cast<uint16_t *>(y);
    L.m = m;
    L.n_out = n_out;
    L.n_in = n_in;
    L.mode = mode;
    L.num_kb = static_cast<int32_t>((n_in + kPK - 1) / kPK);
    L.row_tiles = static_cast<int32_t>((n_out + 2 * kPM - 1) / (2 * kPM));
    L.tok_tiles = static_cast<int32_t>((m + kPN - 1) / kPN);
    L.group = L.tok_tiles < 8 ? L.tok_tiles : 8;
    L.bits_vec8 = ((n_in / 8) % 8 == 0 && (reinterpret_cast<uintptr_t>(bits) & 7) == 0) ? 1 : 0;
    L.first_pair = first_pair;
    return encode_tensor_map_2d(&maps.w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_base, n_in, n_out, n_in * 2, kPK,
                                kPM, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_tensor_map_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, n_in, x_rows, n_in * 2, kPK,
                                kPN / 2, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool prefill_pair_multi_supported(const BatchItem *items, int n, const DevCtx &ctx) {
    if (n < 1 || n > kPMaxLinears) return false;
    for (int i = 0; i < n; ++i)
        if (!prefill_pair_supported(items[i].m, items[i].n_out, items[i].n_in, ctx)) return false;
    return true;
}

cudaError_t launch_prefill_pair_multi(const BatchItem *items, int n, const DevCtx &ctx, cudaStream_t stream) {
    if (!prefill_pair_multi_supported(items, n, ctx)) return cudaErrorNotSupported;
    PairMaps maps;
    PairArgs a = {};
    a.n_lin = n;
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;
    int64_t pairs = 0;
    for (int i = 0; i < n; ++i) {
        const BatchItem &it = items[i];
        if (pairs > 0x3FFFFFFFLL) return cudaErrorInvalidValue;
        if (!fill_linear(maps, a, i, it.x, it.m, it.w_base, it.bits, it.alpha, it.alpha_mode, it.m, it.n_out, it.n_in,
                         it.y, static_cast<int32_t>(pairs)))
            return cudaErrorInvalidValue;
        pairs += prefill_pair_tiles(it.m, it.n_out);
    }
    return launch_pair<false>(maps, a, pairs, ctx, stream);
}

cudaError_t launch_prefill_pair(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                                int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                                cudaStream_t stream) {
    const BatchItem it{x, w_base, bits, alpha, y, m, n_out, n_in, alpha_mode};
    return launch_prefill_pair_multi(&it, 1, ctx, stream);
}

cudaError_t launch_prefill_pair_grouped(const void *x_sorted, int64_t m, const void *w_base,
                                        const GroupedVariants &vars, int64_t n_out, int64_t n_in, void *y,
                                        const GroupTable &tab, const DevCtx &ctx, cudaStream_t stream) {
    if (!prefill_pair_supported(m, n_out, n_in, ctx) || vars.count > kPMaxVariants) return cudaErrorNotSupported;
    PairMaps maps;
    PairArgs a = {};
    a.n_lin = 1;
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;
    if (!fill_linear(maps, a, 0, x_sorted, m, w_base, nullptr, nullptr, 0, m, n_out, n_in, y, 0))
        return cudaErrorInvalidValue;
    bool vec8 = (n_in / 8) % 8 == 0;
    for (int v = 0; v < vars.count; ++v) {
        a.vbits[v] = vars.bits[v];
        a.valpha[v] = vars.alpha[v];
        a.vmode[v] = vars.mode[v];
        vec8 = vec8 && (reinterpret_cast<uintptr_t>(vars.bits[v]) & 7) == 0;
    }
    a.lin[0].bits_vec8 = vec8 ? 1 : 0;
    a.tiles = tab.tiles;
    a.n_tiles = tab.n_tiles;
    a.perm = tab.perm;
    a.max_slots = tab.max_slots;
    return launch_pair<true>(maps, a, static_cast<int64_t>(a.lin[0].row_tiles) * tab.max_slots, ctx, stream);
}

}  // namespace bd
