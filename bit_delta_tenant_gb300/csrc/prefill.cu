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
//   warps 2..9  reconstruction, in two groups of four that take alternate K
//               blocks (so two blocks are rebuilt at once): one thread per tile
//               row, with the row's 8 packed bytes of the block (prefetched
//               three of its blocks ahead); it rebuilds the row's eight 16-byte
//               chunks of the swizzled W tile as bf16(W_base + alpha_r*s), one
//               bf16x2 add per pair with alpha_r rounded to bf16 -- one chunk is
//               exactly one packed byte.  After the K loop the
//               same warps are the epilogue (warp w reads TMEM lanes
//               32*(w%4)..+31, the two groups splitting the token columns).
//   warp 1      allocates TMEM (256 accumulator columns, plus 32 columns per
//               stage for the rebuilt A tile); lane 0 issues tcgen05.mma
//               kind::f16 (M=128, N=tokens<=256, K=16, bf16 in, fp32
//               accumulate in TMEM) and commits each stage back to the producer.
// The rebuilt tile goes from registers to tensor memory (tcgen05.st) and the
// MMA takes A from there, so shared memory carries only the TMA fills, the
// rebuild reads and the activation (B) operand; with BD_PREFILL_TMEM_A=0 the
// tile is instead written back in place and read by the MMA from shared memory.
// When the output tiles alone would leave SMs idle (small m or few W rows), a
// cluster of C CTAs shares one output tile, each rank covering K/C: after the
// last MMA every rank parks its fp32 tile in its (now idle) ring memory and the
// cluster adds the C tiles in rank order through distributed shared memory.
// Every wait is bounded; a role that gives up records a timeout in the status
// word, tells the other roles through a shared flag, drains its own copies
// and MMAs in flight, and the CTA frees its TMEM and returns.
#include <cooperative_groups.h>

#include <cstdlib>

#include "bd_device.cuh"
#include "bd_internal.h"

namespace cg = cooperative_groups;

namespace bd {
namespace {

constexpr int kBM = 128;  // W rows per tile (MMA M)
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr uint32_t kWBytes = kBM * kBK * 2;
constexpr int kRebuildWarps = 8;
constexpr int kThreads = (2 + kRebuildWarps) * 32;  // producer, MMA issuer, rebuild/epilogue

// Token tile BN (MMA N): 256 for prefill; 64 for m <= 64, whose smaller
// activation tile leaves room for a ring twice as deep (more W in flight).
template <int BN>
struct Tile {
    static constexpr int kStages = BN >= 256 ? 4 : 8;
    static constexpr uint32_t kXBytes = BN * kBK * 2;
    static constexpr uint32_t kStageTx = kWBytes + kXBytes;
    static constexpr uint32_t kAccCols = BN;  // fp32 accumulator columns (one per token)
    static constexpr size_t kSmemBytes = 1024 + kStages * (kWBytes + kXBytes) + 256;
};
constexpr int kMaxVariants = 64;

struct PrefillArgs {
    const uint8_t *bits;
    const float *alpha;
    uint16_t *y;
    float *y32;         // base-only mode (non-null): y32 = x . W_base^T in fp32, no rebuild, A read as loaded
    int64_t m, n_out, n_in;
    int32_t mode;
    int32_t num_kb;
    int32_t row_tiles, tok_tiles, group;
    int32_t ksplit;     // ranks of a cluster splitting K (1: no split)
    int32_t kb_per;     // K blocks per rank
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

// One bf16 pair of W_eff = W_base + alpha_b * s, rounded once to bf16
// (add.rn.bf16x2 adds exactly, then rounds to nearest even), with alpha_b =
// alpha rounded to bf16.  The pair of signed scales is built from -alpha_b in
// both halves: one multiply moves bit 2I of the packed byte to bit 15 and bit
// 2I+1 to bit 31 (the two shifted copies never overlap), and the xor clears the
// sign of -alpha_b where the bit is 1 (+alpha_b).  Three operations per pair
// instead of widening to fp32 and packing back.
template <int I>
__device__ __forceinline__ uint32_t rebuild_pair(uint32_t w, uint32_t byte, uint32_t neg_alpha2) {
    constexpr uint32_t mul = (1u << (15 - 2 * I)) + (1u << (30 - 2 * I));
    const uint32_t s = ((byte * mul) & 0x80008000u) ^ neg_alpha2;
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(s));
    return r;
}

__device__ __forceinline__ void give_up(volatile int *abort_flag, unsigned *status) {
    *abort_flag = 1;
    flag_status(status, kDevTimeout);
}

template <bool kGrouped, bool kTmemA, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ PrefillArgs a) {
    constexpr int kBN = BN;
    constexpr int kStages = Tile<BN>::kStages;
    constexpr uint32_t kXBytes = Tile<BN>::kXBytes;
    constexpr uint32_t kStageTx = Tile<BN>::kStageTx;
    constexpr uint32_t kAccCols = Tile<BN>::kAccCols;
    extern __shared__ uint8_t smem_raw[];
    // With kTmemA the rebuilt W tile goes to tensor memory (columns 256 + 32*stage)
    // and the MMA reads A from there; otherwise it is written back in place.
    constexpr uint32_t kTmemCols = kTmemA ? 512 : (BN < 32 ? 32 : BN);
    static_assert(!kTmemA || kAccCols + kStages * (kBK / 2) <= 512, "accumulator + A buffers fit in TMEM");
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
        const int tile = blockIdx.x / a.ksplit;  // the ranks of a cluster share one output tile
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
    // K blocks [kb0, kb0 + nkb) of this CTA (all of them unless a cluster splits K)
    const int kb0 = kGrouped ? 0 : static_cast<int>(blockIdx.x % a.ksplit) * a.kb_per;
    const int nkb = kGrouped ? a.num_kb : min(a.kb_per, a.num_kb - kb0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&rebuilt[s], kRebuildWarps / 2);  // the warp group of the block's parity
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
                tma_load_2d(sW + s * kWBytes, &tm_w, &full[s], (kb0 + kb) * kBK, m0);
                tma_load_2d(sX + s * kXBytes, &tm_x, &full[s], (kb0 + kb) * kBK, n0);
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
            // Every MMA operand of every ring stage is computed once and the loop is unrolled
            // by the ring depth: no descriptor arithmetic between consecutive MMAs (measured on
            // GB300: ~250 clocks per MMA with the descriptor derived in the loop, ~134 without).
            uint64_t adesc[kStages][kBK / 16], bdesc[kStages][kBK / 16];
            uint32_t aaddr[kStages][kBK / 16];
#pragma unroll
            for (int s = 0; s < kStages; ++s)
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    adesc[s][kk] = sw128_kmajor_desc(smem_u32(sW + s * kWBytes) + kk * 32);
                    bdesc[s][kk] = sw128_kmajor_desc(smem_u32(sX + s * kXBytes) + kk * 32);
                    aaddr[s][kk] = tmem + kAccCols + s * (kBK / 2) + kk * 8;
                }
            bool ok = true;
            for (int ring = 0; ring < nkb && ok; ring += kStages) {  // this CTA's K blocks, a ring's worth at a time
#pragma unroll
                for (int s = 0; s < kStages; ++s) {
                    const int kb = ring + s;
                    if (kb >= nkb) break;
                    const uint32_t ph = (ring / kStages) & 1;
                    if (!mbar_wait(&rebuilt[s], ph, a.wait_ns, abort_flag)) {
                        give_up(abort_flag, a.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t acc = (kk != 0 || kb != 0) ? 1u : 0u;
                        if constexpr (kTmemA)
                            tc_mma_f16_ts(tmem, aaddr[s][kk], bdesc[s][kk], idesc, acc);
                        else
                            tc_mma_f16_ss(tmem, adesc[s][kk], bdesc[s][kk], idesc, acc);
                    }
                    tc_commit(&empty[s]);
                }
            }
            // Always wait for this thread's MMAs before the CTA may free TMEM, even if
            // the epilogue gave up early (its wait can run out while MMAs still run).
            tc_commit(acc_full);
            (void)ok;
            mbar_wait(acc_full, 0, kDrainLimitNs, nullptr);
        }
    } else {
        // ---- rebuild (then epilogue) warps ------------------------------------------
        // Thread q of warp group h (warps 2..5: h = 0, warps 6..9: h = 1) owns tile
        // row r = 32*(warp%4) + lane: all eight 16-byte chunks of the row (its 8
        // packed bytes) in the K blocks of parity h, so the two groups rebuild
        // consecutive blocks at the same time.  Warp w may read TMEM lanes
        // 32*(w%4)..+31 only, so the same row mapping serves the epilogue, where h
        // picks half of the tokens.
        constexpr int kParts = 2;  // warp groups: K-block parity, then token half
        const int sub = warp & 3;
        const int h = (warp - 2) >> 2;
        const int r = sub * 32 + lane;
        const int64_t row = static_cast<int64_t>(m0) + r;
        const bool row_ok = row < a.n_out;
        const float al = (row_ok && alpha != nullptr) ? (mode ? alpha[row] : alpha[0]) : 0.0f;  // none: base only
        const uint32_t neg_al = pack_bf16x2(-al, -al);  // -alpha_b in both halves
        const int64_t bpr = a.n_in / 8;
        const uint8_t *brow = bits != nullptr ? bits + (row_ok ? row : 0) * bpr : nullptr;

        auto load_bits = [&](int kbl) -> uint2 {  // kbl: this CTA's K block index
            uint2 v = make_uint2(0u, 0u);
            const int64_t c0 = static_cast<int64_t>(kb0 + kbl) * 8;  // first packed byte
            if (row_ok && kbl < nkb && a.y32 == nullptr) {
                if (a.bits_vec8 && c0 + 8 <= bpr) {
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
            const int s = kb % kStages;
            const uint32_t ph = (kb / kStages) & 1;
            const uint2 b_cur = bq[0];
#pragma unroll
            for (int i = 0; i + 1 < kBitsAhead; ++i) bq[i] = bq[i + 1];
            bq[kBitsAhead - 1] = load_bits(kb + 2 * kBitsAhead);
            const bool got = mbar_wait(&full[s], ph, a.wait_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up(abort_flag, a.status);
                ok = false;
                break;
            }
            if (!kTmemA && a.y32 != nullptr) {  // base only: the MMA takes the W_base tile as loaded
                __syncwarp();
                if (lane == 0) mbar_arrive(&rebuilt[s]);
                continue;
            }
            uint8_t *rowp = sW + s * kWBytes + r * 128;
            uint4 w[8];
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) w[cc] = *reinterpret_cast<const uint4 *>(rowp + ((cc ^ (r & 7)) << 4));
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint32_t byte = ((cc < 4 ? b_cur.x : b_cur.y) >> (8 * (cc & 3))) & 0xFFu;
                w[cc].x = rebuild_pair<0>(w[cc].x, byte, neg_al);
                w[cc].y = rebuild_pair<1>(w[cc].y, byte, neg_al);
                w[cc].z = rebuild_pair<2>(w[cc].z, byte, neg_al);
                w[cc].w = rebuild_pair<3>(w[cc].w, byte, neg_al);
                if constexpr (!kTmemA) *reinterpret_cast<uint4 *>(rowp + ((cc ^ (r & 7)) << 4)) = w[cc];
            }
            if constexpr (kTmemA) {
                uint32_t v[32];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    v[4 * cc] = w[cc].x, v[4 * cc + 1] = w[cc].y;
                    v[4 * cc + 2] = w[cc].z, v[4 * cc + 3] = w[cc].w;
                }
                tmem_st_32x32b_x32(tmem + (static_cast<uint32_t>(sub * 32) << 16) + kAccCols + s * (kBK / 2), v);
                tmem_st_wait();
                tc_fence_before();
            } else {
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&rebuilt[s]);
        }
        if (ok && !kGrouped && a.ksplit > 1) {
            // Split K: park this rank's fp32 partial tile in the (now idle) ring
            // memory as red[token][row]; the cluster adds the ranks' tiles below.
            const bool got = mbar_wait(acc_full, 0, a.wait_ns, abort_flag);
            if (__all_sync(0xFFFFFFFFu, got)) {
                tc_fence_after();
                const uint32_t lane_addr = tmem + (static_cast<uint32_t>(sub * 32) << 16);
                float *red = reinterpret_cast<float *>(smem);
#pragma unroll 1
                for (int c0 = h * (kBN / kParts); c0 < (h + 1) * (kBN / kParts); c0 += 32) {
                    if (c0 >= count) break;  // warp-uniform
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(lane_addr + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) red[(c0 + i) * kBM + r] = __uint_as_float(v[i]);
                }
            } else if (lane == 0) {
                give_up(abort_flag, a.status);
            }
        } else if (ok) {
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
                            if (c0 + i < count && in_bounds(n0 + c0 + i < a.m, a.status)) {
                                const int64_t t = kGrouped ? static_cast<int64_t>(a.perm[n0 + c0 + i])
                                                           : static_cast<int64_t>(n0) + c0 + i;
                                if (!in_bounds(t >= 0 && t < a.m, a.status)) continue;
                                if (!kGrouped && a.y32 != nullptr) {
                                    a.y32[t * a.n_out + row] = __uint_as_float(v[i]);
                                } else {
                                    __nv_bfloat16 hv = __float2bfloat16_rn(__uint_as_float(v[i]));
                                    ycol[t * a.n_out] = *reinterpret_cast<uint16_t *>(&hv);
                                }
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

    if (!kGrouped && a.ksplit > 1) {
        // rank c adds elements [c*share, (c+1)*share) of the tile over the cluster's
        // ranks in rank order and writes them as bf16 (consecutive threads: consecutive rows)
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int rank = static_cast<int>(cluster.block_rank());
        const int total = count * kBM;
        const int share = (total + a.ksplit - 1) / a.ksplit;
        const int e1 = min(total, (rank + 1) * share);
        float *red = reinterpret_cast<float *>(smem);
        if (!*abort_flag) {
            for (int e = rank * share + threadIdx.x; e < e1; e += kThreads) {
                const int tok = e / kBM, rr = e - tok * kBM;
                const int64_t orow = static_cast<int64_t>(m0) + rr;
                if (orow < a.n_out && in_bounds(n0 + tok < a.m, a.status)) {
                    float sum = 0.0f;
                    for (int q = 0; q < a.ksplit; ++q) sum += cluster.map_shared_rank(red, q)[e];
                    if (a.y32 != nullptr) {
                        a.y32[(static_cast<int64_t>(n0) + tok) * a.n_out + orow] = sum;
                    } else {
                        __nv_bfloat16 hv = __float2bfloat16_rn(sum);
                        a.y[(static_cast<int64_t>(n0) + tok) * a.n_out + orow] = *reinterpret_cast<uint16_t *>(&hv);
                    }
                }
            }
        }
        cluster.sync();  // peers may still be reading this CTA's tile
    }
}

}  // namespace

namespace {

template <bool kGrouped, bool kTmemA, int BN>
cudaError_t set_smem_attr(const DevCtx &ctx) {
    static bool attr_set[128] = {false};
    if (ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<kGrouped, kTmemA, BN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(Tile<BN>::kSmemBytes));
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    return cudaSuccess;
}

// The rebuilt W tile feeds the MMA from tensor memory (measured ~19% faster
// on GB300 than writing it back to shared memory, which then carries only the
// TMA fills, the rebuild reads and the activation operand); the shared-memory
// form serves the base-only product, whose A tile is used as loaded.
constexpr bool use_tmem_a() { return true; }

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
               int64_t n_out, int64_t n_in, int bn) {
    return encode_tensor_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_base, n_in, n_out, n_in * 2, kBK, kBM,
                                CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, n_in, x_rows, n_in * 2, kBK,
                                static_cast<uint32_t>(bn), CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

namespace {

template <int BN>
cudaError_t launch_prefill_bn(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                              int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                              cudaStream_t stream, float *y32 = nullptr) {
    const bool tmem_a = y32 == nullptr && use_tmem_a();  // base-only reads A from shared memory
    cudaError_t e = tmem_a ? set_smem_attr<false, true, BN>(ctx) : set_smem_attr<false, false, BN>(ctx);
    if (e != cudaSuccess) return e;
    CUtensorMap tm_w, tm_x;
    if (!make_maps(tm_w, tm_x, w_base, x, m, n_out, n_in, BN)) return cudaErrorInvalidValue;
    PrefillArgs a = {};
    fill_common(a, m, n_out, n_in, y, ctx);
    a.bits = bits;
    a.alpha = alpha;
    a.mode = alpha_mode;
    a.y32 = y32;
    a.tok_tiles = static_cast<int32_t>((m + BN - 1) / BN);
    a.group = a.tok_tiles < 8 ? a.tok_tiles : 8;
    a.bits_vec8 = ((n_in / 8) % 8 == 0 && (reinterpret_cast<uintptr_t>(bits) & 7) == 0) ? 1 : 0;
    const int64_t tiles = static_cast<int64_t>(a.row_tiles) * a.tok_tiles;
    // Few output tiles (small m, or few W rows) leave SMs idle: split K over a
    // cluster of C CTAs (one CTA per SM; a cluster sits in one GPC, so at most
    // ~90% of the SMs are counted on), each rank keeping at least 8 K blocks.
    int c = 1;
    while (c < 8 && tiles * (2 * c) * 10 <= 9 * static_cast<int64_t>(ctx.num_sms) && a.num_kb / (2 * c) >= 8) c *= 2;
    a.kb_per = (a.num_kb + c - 1) / c;
    a.ksplit = (a.num_kb + a.kb_per - 1) / a.kb_per;  // no empty ranks
    const int64_t grid = tiles * a.ksplit;
    if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Tile<BN>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.ksplit);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return tmem_a ? cudaLaunchKernelEx(&cfg, prefill_kernel<false, true, BN>, tm_w, tm_x, a)
                  : cudaLaunchKernelEx(&cfg, prefill_kernel<false, false, BN>, tm_w, tm_x, a);
}

}  // namespace

cudaError_t launch_prefill(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                           int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                           cudaStream_t stream) {
    // CTA pairs (256 x 256 tiles, half the activation traffic per SM) when their tiles
    // fill at least 48 of the SMs' pairs (on 152 SMs: 5/8 of them), or at least 24 with
    // m >= 256 and K <= 8192; otherwise the single-CTA tiles, which split K over a
    // cluster to fill the SMs.  Measured on GB300 (single / pair, us): 14336 x 4096 at
    // m = 256 (56 tiles) 44.2 / 37.2; 32 tiles: 4096^2 x 512 37.6 / 31.4, 1024 x 4096 x
    // 2048 35.3 / 31.1, 8192^2 x 256 56.1 / 53.5, but 4096 x 14336 x 512 72.7 / 80.3 and
    // 8192^2 x 128 45.7 / 49.5; 16 tiles: 4096^2 x 256 24.8 / 31.3.
    const int64_t forced = option_value(BD_OPT_PREFILL_KERNEL);
    const int64_t tiles = prefill_pair_tiles(m, n_out);
    const int64_t pairs = ctx.num_sms / 2;
    const bool pair_auto = m > 64 && (8 * tiles >= 5 * pairs || (4 * tiles >= pairs && m >= 256 && n_in <= 8192));
    const bool pair = forced == 2 || (forced == 0 && pair_auto);
    if (pair && prefill_pair_supported(m, n_out, n_in, ctx))
        return launch_prefill_pair(x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y, ctx, stream);
    if (m <= 64)
        return launch_prefill_bn<64>(x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y, ctx, stream);
    return launch_prefill_bn<256>(x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y, ctx, stream);
}

cudaError_t launch_base_product(const void *x, int64_t m, const void *w_base, int64_t n_out, int64_t n_in,
                                float *y32, const DevCtx &ctx, cudaStream_t stream) {
    if (m <= 64)
        return launch_prefill_bn<64>(x, m, w_base, nullptr, nullptr, 0, n_out, n_in, nullptr, ctx, stream, y32);
    return launch_prefill_bn<256>(x, m, w_base, nullptr, nullptr, 0, n_out, n_in, nullptr, ctx, stream, y32);
}

cudaError_t launch_prefill_grouped(const void *x_sorted, int64_t m, const void *w_base, const GroupedVariants &vars,
                                   int64_t n_out, int64_t n_in, void *y, const GroupTable &tab, const DevCtx &ctx,
                                   cudaStream_t stream) {
    // CTA pairs when the tiles of the dense token count would fill the SMs (as for one variant)
    const int64_t forced = option_value(BD_OPT_PREFILL_KERNEL);
    const bool pair = forced == 2 || (forced == 0 && 2 * prefill_pair_tiles(m, n_out) >= static_cast<int64_t>(ctx.num_sms));
    if (pair) {
        const cudaError_t e = launch_prefill_pair_grouped(x_sorted, m, w_base, vars, n_out, n_in, y, tab, ctx, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    const bool tmem_a = use_tmem_a();
    cudaError_t e = tmem_a ? set_smem_attr<true, true, 256>(ctx) : set_smem_attr<true, false, 256>(ctx);
    if (e != cudaSuccess) return e;
    CUtensorMap tm_w, tm_x;
    if (!make_maps(tm_w, tm_x, w_base, x_sorted, m, n_out, n_in, 256)) return cudaErrorInvalidValue;
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
    a.ksplit = 1;
    a.kb_per = a.num_kb;
    const int64_t grid = static_cast<int64_t>(a.row_tiles) * tab.max_slots;
    if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    if (tmem_a)
        prefill_kernel<true, true, 256><<<static_cast<unsigned>(grid), kThreads, Tile<256>::kSmemBytes, stream>>>(
            tm_w, tm_x, a);
    else
        prefill_kernel<true, false, 256><<<static_cast<unsigned>(grid), kThreads, Tile<256>::kSmemBytes, stream>>>(
            tm_w, tm_x, a);
    return cudaGetLastError();
}

}  // namespace bd
