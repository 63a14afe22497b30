// prefill_pair.cu -- fused BitDelta linear for large token counts on CTA pairs:
// y = x . (W_base + alpha*S)^T with W_eff rebuilt tile by tile on chip and
// never written to HBM, 256 (W rows) x 256 (tokens) output tiles on pairs of
// CTAs on the 5th-generation tensor cores (tcgen05, cta_group::2).
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
// Why persistent: a pair stays resident and takes tiles p, p + G, p + 2G, ...
// (G pairs in the grid, at most one per two SMs), its ring of K blocks running
// on from one tile into the next.  Launching one pair per tile instead costs
// each tile a CTA start, a pipeline fill and an epilogue during which the
// tensor cores idle -- measured on GB300 as 5-8 us per tile, a quarter of a
// K = 4096 tile.  Here only the reading of the accumulator out of tensor
// memory holds the next tile's MMAs back.
//
// A cluster of two CTAs (rank r = 0, 1) computes W rows [256*i + 128*r, +128)
// of each of its tiles in CTA r; per 64-wide K block:
//   warp 0      TMA producer of this CTA: the W_base tile [128 x 64] of its
//               own rows and its half of the token tile [N/2 x 64] (tokens
//               n0 + r*N/2 ...), both K-major with the 128-byte swizzle, into a
//               kPStages-deep ring, completing on this CTA's full barrier.  No
//               load is multicast: each CTA reads its own halves.
//   warps 2..9  rebuild, in two groups of four taking alternate K blocks (by the
//               parity of the block's position in the pair's whole sequence):
//               one thread per W row, W_eff = W_base + alpha_b*s as bf16 pairs
//               (one bf16x2 add per pair, alpha rounded to bf16), stored with
//               tcgen05.st into this CTA's tensor memory as the MMA's A operand;
//               then each warp arrives on the even CTA's "rebuilt" barrier.
//   warp 1      of the even CTA: one lane waits for both CTAs' rebuilt blocks
//               and issues tcgen05.mma.cta_group::2 kind::f16 (M = 256,
//               N = tokens <= 256, K = 16), committing each stage to the empty
//               barriers of both CTAs and each finished tile to both CTAs'
//               acc_full (multicast commits); before a tile's first MMA it waits
//               until both epilogues have read the previous tile (acc_empty).
//               In both CTAs warp 1 allocates (and frees) the pair's tensor
//               memory: 256 accumulator columns plus 32 per ring stage of A.
//   warps 10..13 epilogue (TMEM lanes 32*(w%4)..+31): read the accumulator,
//               round to bf16 into a shared-memory staging tile, release the
//               accumulator, then write the staged rows of y with 16-byte stores
//               while the next tile's MMAs run.
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
constexpr uint32_t kPWBytes = kPM * kPK * 2;         // 16 KB
constexpr uint32_t kPXBytes = (kPN / 2) * kPK * 2;   // 16 KB: this CTA's half of the tokens
constexpr uint32_t kPAccCols = kPN;                  // fp32 accumulator columns (one per token)
constexpr uint32_t kPTmemCols = 512;
constexpr int kPRebuildWarps = 8;
constexpr int kPEpiWarps = 4;
constexpr int kPEpiFirstWarp = 2 + kPRebuildWarps;
constexpr int kPThreads = (2 + kPRebuildWarps + kPEpiWarps) * 32;
constexpr int kPEpiBar = 1;  // named barrier of the epilogue warps

// Two shapes of the same kernel share the 227 KB of shared memory differently
// between the K-block ring and the staged output tile ([token][128 rows] bf16):
//   kStages = 5, kParts = 1: the whole 64 KB tile is staged, so the accumulator
//     is released as soon as it has been read out of tensor memory;
//   kStages = 6, kParts = 2: 128 tokens (32 KB) at a time, the accumulator
//     released after the second half is read -- a deeper ring for long K, where
//     the L2 latency a ring must cover weighs more than the per-tile release.
template <int kStages, int kParts>
struct PairShape {
    static constexpr int kOutTokens = kPN / kParts;
    static constexpr uint32_t kOutBytes = kOutTokens * kPM * 2;
    static constexpr size_t kSmem = 1024 + kStages * (kPWBytes + kPXBytes) + kOutBytes + 256;
    static_assert(kPAccCols + kStages * (kPK / 2) <= kPTmemCols, "accumulator + A stages fit in TMEM");
    static_assert(kSmem <= 232448, "fits the 227 KB of shared memory a CTA may use");
};

constexpr int kPMaxVariants = 64;
constexpr int kPMaxLinears = 8;  // independent linears per launch (a layer's q/k/v, gate/up)

// One linear of a launch: its tiles are [first_pair, first_pair + row_tiles * tok_tiles).
struct PairLinear {
    const uint8_t *bits;
    const float *alpha;
    uint16_t *y;
    int64_t m, n_out, n_in;
    int32_t mode;
    int32_t num_kb;
    int32_t row_tiles, tok_tiles, group;  // pair tiles: 256 W rows x 256 tokens
    int32_t bits_vec8;                    // rows of packed bits are 8-byte aligned
    int32_t y_vec16;                      // y rows start 16-byte aligned (16-byte stores)
    int32_t first_pair;
};

// Token-operand boxes of 16, 32, 64 and 128 rows: a CTA loads the smallest box that holds
// its half of the tile's MMA N, so tiles of few tokens (multi-tenant segments, a ragged
// last token tile) do not pay for 128 rows.
constexpr int kPXBoxes = 4;
__host__ __device__ constexpr int x_box_rows(int i) { return 16 << i; }

struct PairMaps {
    CUtensorMap w[kPMaxLinears];             // W_base [n_out, n_in], boxes of 64 x 128 rows
    CUtensorMap x[kPMaxLinears][kPXBoxes];   // x [m, n_in], boxes of 64 x x_box_rows(i) token rows
};

struct PairArgs {
    PairLinear lin[kPMaxLinears];
    int32_t n_lin;
    int32_t n_units;  // tiles of the launch (multi-tenant mode: row tiles x max_slots, an upper bound)
    unsigned *status;
    uint64_t wait_ns;
    // Multi-tenant mode only: token tiles come from a device-built table of
    // (variant, first row in the variant-sorted activations, row count <= 256);
    // the launch's tiles are (W row tile, slot < *n_tiles), consecutive tiles
    // taking every slot of one W row tile, and output rows are scattered back to
    // the original token order through perm.
    const int32_t *tiles;
    const int32_t *n_tiles;
    const int32_t *perm;
    int32_t max_slots;
    const uint8_t *vbits[kPMaxVariants];
    const float *valpha[kPMaxVariants];
    int32_t vmode[kPMaxVariants];
};

// One tile of the launch, as every role of a pair needs it.
struct PairTile {
    int lp;        // linear
    int row0;      // first W row of the pair's 256
    int n0;        // first token (multi-tenant mode: first row of the sorted activations)
    int count;     // tokens, <= 256
    const uint8_t *bits;
    const float *alpha;
    int32_t mode;
};

template <bool kGrouped>
__device__ __forceinline__ PairTile pair_tile(const PairArgs &a, int unit, int n_slots) {
    PairTile t;
    if constexpr (kGrouped) {
        // Consecutive tiles take every token tile of one W tile, so the W tile is
        // read from HBM once per round of tiles and reused from L2.
        const int row_tile = unit / n_slots;
        const int slot = unit - row_tile * n_slots;
        const int v = a.tiles[3 * slot];
        t.lp = 0;
        t.row0 = row_tile * 2 * kPM;
        t.n0 = a.tiles[3 * slot + 1];
        t.count = a.tiles[3 * slot + 2];
        t.bits = a.vbits[v];
        t.alpha = a.valpha[v];
        t.mode = a.vmode[v];
    } else {
        int lp = 0;
        while (lp + 1 < a.n_lin && a.lin[lp + 1].first_pair <= unit) ++lp;
        const PairLinear &L = a.lin[lp];
        // Grouped rasterisation: consecutive tiles cycle over `group` token tiles for
        // one W tile, so a round of tiles touches a compact block of W and x in L2.
        const int pair = unit - L.first_pair;
        const int per_group = L.group * L.row_tiles;
        const int grp = pair / per_group;
        const int rem = pair - grp * per_group;
        const int gsize = min(L.group, L.tok_tiles - grp * L.group);
        const int tok_tile = grp * L.group + rem % gsize;
        t.lp = lp;
        t.row0 = (rem / gsize) * 2 * kPM;
        t.n0 = tok_tile * kPN;
        t.count = static_cast<int>(min(static_cast<int64_t>(kPN), L.m - t.n0));
        t.bits = L.bits;
        t.alpha = L.alpha;
        t.mode = L.mode;
    }
    return t;
}

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

__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kPEpiBar), "n"(kPEpiWarps * 32) : "memory");
}

template <bool kGrouped, int kPStages, int kParts>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_pair_kernel(const __grid_constant__ PairMaps maps, const __grid_constant__ PairArgs a) {
    using Shape = PairShape<kPStages, kParts>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sW = smem;
    uint8_t *sX = smem + kPStages * kPWBytes;
    uint16_t *sOut = reinterpret_cast<uint16_t *>(sX + kPStages * kPXBytes);  // [token][128 rows] bf16
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sOut) + Shape::kOutBytes);
    uint64_t *full = bars;                    // this CTA's TMA fills
    uint64_t *rebuilt = bars + kPStages;      // even CTA: both CTAs' rebuilt A blocks
    uint64_t *empty = bars + 2 * kPStages;    // the pair's MMAs of a stage are complete
    uint64_t *acc_full = bars + 3 * kPStages;       // a tile's MMAs are complete (both CTAs)
    uint64_t *acc_empty = acc_full + 1;             // even CTA: both epilogues have read a tile
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t rank = cluster_rank();
    const int p0 = static_cast<int>(blockIdx.x >> 1);  // this pair; it takes tiles p0, p0 + G, ...
    const int G = static_cast<int>(gridDim.x >> 1);
    int n_slots = 0, total = a.n_units;
    if constexpr (kGrouped) {
        n_slots = min(*a.n_tiles, a.max_slots);  // the same value in every thread of the launch
        if (n_slots < 0) n_slots = 0;
        total = a.lin[0].row_tiles * n_slots;
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&rebuilt[s], kPRebuildWarps);  // four warps of the block's group in each CTA
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * kPEpiWarps);  // the epilogue warps of both CTAs
        *abort_flag = 0;
        mbar_fence_init();
        for (int i = 0; i < a.n_lin; ++i) {
            tma_prefetch_desc(&maps.w[i]);
            for (int b = 0; b < kPXBoxes; ++b) tma_prefetch_desc(&maps.x[i][b]);
        }
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
            uint32_t g = 0;  // K blocks issued, over all of the pair's tiles
            bool ok = true;
            for (int u = p0; u < total && ok; u += G) {
                const PairTile t = pair_tile<kGrouped>(a, u, n_slots);
                const int nkb = a.lin[t.lp].num_kb;
                const int n_mma = (t.count + 15) & ~15;  // pair MMA N; each CTA holds n_mma / 2 token rows
                const int m0 = t.row0 + static_cast<int>(rank) * kPM;
                const int x_first = t.n0 + static_cast<int>(rank) * (n_mma / 2);
                const int bi = n_mma / 2 <= 16 ? 0 : n_mma / 2 <= 32 ? 1 : n_mma / 2 <= 64 ? 2 : 3;
                const uint32_t tx = kPWBytes + static_cast<uint32_t>(x_box_rows(bi)) * (kPK * 2);
                const CUtensorMap *tm_w = &maps.w[t.lp], *tm_x = &maps.x[t.lp][bi];
                for (int kb = 0; kb < nkb; ++kb) {
                    const uint32_t s = g % kPStages;
                    const uint32_t ph = (g / kPStages) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, a.wait_ns, abort_flag)) {
                        give_up_p(abort_flag, a.status);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], tx);
                    tma_load_2d(sW + s * kPWBytes, tm_w, &full[s], kb * kPK, m0);
                    tma_load_2d(sX + s * kPXBytes, tm_x, &full[s], kb * kPK, x_first);
                    ++g;
                }
            }
            if (*abort_flag) {
                // the loads of the last stages issued land before the CTA may exit
                for (uint32_t q = (g > kPStages ? g - kPStages : 0); q < g; ++q)
                    mbar_wait(&full[q % kPStages], (q / kPStages) & 1, kDrainLimitNs, nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0 && p0 < total) {
            // Every operand of every MMA (ring stages x four 16-wide K slices) is computed
            // once here and the loop is unrolled by the ring depth, so that no address or
            // descriptor arithmetic sits between consecutive MMAs: measured on GB300, an MMA
            // whose descriptor is derived in the loop issues every ~250 clocks, one with a
            // precomputed descriptor every ~134 (M = 128, N = 256).  A tile boundary may fall
            // anywhere in a ring; the next tile's shape is derived there, between two stages.
            uint64_t bdesc[kPStages][kPK / 16];
            uint32_t aaddr[kPStages][kPK / 16];
#pragma unroll
            for (int s = 0; s < kPStages; ++s)
#pragma unroll
                for (int kk = 0; kk < kPK / 16; ++kk) {
                    bdesc[s][kk] = sw128_kmajor_desc(smem_u32(sX + s * kPXBytes) + kk * 32);
                    aaddr[s][kk] = tmem + kPAccCols + s * (kPK / 2) + kk * 8;
                }
            int u = p0;
            PairTile t = pair_tile<kGrouped>(a, u, n_slots);
            int nkb = a.lin[t.lp].num_kb;
            uint32_t idesc = idesc_bf16_f32(2 * kPM, (t.count + 15) & ~15);
            uint32_t done = 0;  // tiles committed to acc_full
            int kb = 0;
            bool run = true, failed = false;
            for (uint32_t ring = 0; run; ring += kPStages) {  // a ring's worth of K blocks at a time
                const uint32_t ph = (ring / kPStages) & 1;
#pragma unroll
                for (int s = 0; s < kPStages; ++s) {
                    if (!run) break;
                    // A tile's first MMA overwrites the accumulator: both epilogues must have
                    // read the previous tile out of it.
                    if (kb == 0 && done > 0 && !mbar_wait(acc_empty, (done - 1) & 1, a.wait_ns, abort_flag)) {
                        give_up_p(abort_flag, a.status);
                        run = false;
                        failed = true;
                        break;
                    }
                    if (!mbar_wait(&rebuilt[s], ph, a.wait_ns, abort_flag)) {
                        give_up_p(abort_flag, a.status);
                        run = false;
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    tc_mma_f16_ts_pair(tmem, aaddr[s][0], bdesc[s][0], idesc, kb != 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < kPK / 16; ++kk)
                        tc_mma_f16_ts_pair(tmem, aaddr[s][kk], bdesc[s][kk], idesc, 1u);
                    tc_commit_pair_mc(&empty[s], 0x3);
                    if (++kb == nkb) {
                        tc_commit_pair_mc(acc_full, 0x3);
                        ++done;
                        kb = 0;
                        u += G;
                        if (u >= total) {
                            run = false;
                        } else {
                            t = pair_tile<kGrouped>(a, u, n_slots);
                            nkb = a.lin[t.lp].num_kb;
                            idesc = idesc_bf16_f32(2 * kPM, (t.count + 15) & ~15);
                        }
                    }
                }
            }
            // This thread's MMAs are complete before the pair may free tensor memory: after a
            // give-up one more commit covers the MMAs of the unfinished tile.
            if (failed) {
                tc_commit_pair_mc(acc_full, 0x3);
                mbar_wait(acc_full, done & 1, kDrainLimitNs, nullptr);
            } else if (done > 0) {
                mbar_wait(acc_full, (done - 1) & 1, kDrainLimitNs, nullptr);
            }
        }
    } else if (warp < kPEpiFirstWarp) {
        // ---- rebuild warps ----------------------------------------------------------
        // Thread q of group h (warps 2..5: h = 0, warps 6..9: h = 1) owns tile row
        // r = 32*(warp%4) + lane (warp w may access TMEM lanes 32*(w%4)..+31 only): all
        // eight 16-byte chunks of the row (its 8 packed bytes) in the K blocks whose
        // position in the pair's sequence of blocks, over all its tiles, has parity h.
        const int sub = warp & 3;
        const int h = (warp - 2) >> 2;
        const int r = sub * 32 + lane;
        const uint32_t rebuilt0 = mapa_rank(smem_u32(rebuilt), 0);  // the even CTA's barriers
        const uint32_t a_lane = tmem + (static_cast<uint32_t>(sub * 32) << 16) + kPAccCols;

        // A position in the group's sequence: K block kb of the pair's tile u, with what
        // the thread's row needs of that tile.
        struct Cursor {
            int u, kb, nkb;
            const uint8_t *brow;  // the row's packed bits
            int64_t bpr;          // packed bytes per row
            bool row_ok, vec8;
            float al;
        };
        auto cursor_tile = [&](Cursor &c, int u) {
            c.u = u;
            if (u >= total) return;
            const PairTile t = pair_tile<kGrouped>(a, u, n_slots);
            const PairLinear &L = a.lin[t.lp];
            const int64_t row = static_cast<int64_t>(t.row0) + static_cast<int>(rank) * kPM + r;
            c.row_ok = row < L.n_out;
            c.bpr = L.n_in / 8;
            c.brow = t.bits + (c.row_ok ? row : 0) * c.bpr;
            c.nkb = L.num_kb;
            c.vec8 = L.bits_vec8 != 0;
            c.al = c.row_ok ? (t.mode ? t.alpha[row] : t.alpha[0]) : 0.0f;
        };
        auto cursor_step = [&](Cursor &c, int by) {  // by blocks along the pair's sequence
            c.kb += by;
            while (c.u < total && c.kb >= c.nkb) {
                c.kb -= c.nkb;
                cursor_tile(c, c.u + G);
            }
        };
        auto cursor_bits = [&](const Cursor &c) -> uint2 {
            uint2 v = make_uint2(0u, 0u);
            if (c.u >= total || !c.row_ok) return v;
            const int64_t c0 = static_cast<int64_t>(c.kb) * 8;  // first packed byte of the block
            if (c.vec8 && c0 + 8 <= c.bpr) {
                v = __ldg(reinterpret_cast<const uint2 *>(c.brow + c0));
            } else {
                for (int q = 0; q < 8; ++q)
                    if (c0 + q < c.bpr) {
                        const uint32_t byte = __ldg(c.brow + c0 + q);
                        if (q < 4) v.x |= byte << (8 * q);
                        else v.y |= byte << (8 * (q - 4));
                    }
            }
            return v;
        };

        Cursor cur;  // the block being rebuilt
        cur.kb = 0;
        cursor_tile(cur, p0);
        cursor_step(cur, h);
        // Packed bits arrive by plain loads three of this group's K blocks ahead, across
        // tile boundaries.
        constexpr int kBitsAhead = 3;
        Cursor ahead = cur;
        uint2 bq[kBitsAhead];
#pragma unroll
        for (int i = 0; i < kBitsAhead; ++i) {
            bq[i] = cursor_bits(ahead);
            cursor_step(ahead, 2);
        }
        uint32_t g = static_cast<uint32_t>(h);  // the block's position in the pair's sequence
        int al_u = -1;
        uint32_t neg_al = 0;
        while (cur.u < total) {
            if (cur.u != al_u) {
                neg_al = pack_bf16x2(-cur.al, -cur.al);  // -alpha_b in both halves
                al_u = cur.u;
            }
            const uint32_t s = g % kPStages;
            const uint32_t ph = (g / kPStages) & 1;
            const uint2 b_cur = bq[0];
#pragma unroll
            for (int i = 0; i + 1 < kBitsAhead; ++i) bq[i] = bq[i + 1];
            bq[kBitsAhead - 1] = cursor_bits(ahead);
            cursor_step(ahead, 2);
            const bool got = mbar_wait(&full[s], ph, a.wait_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up_p(abort_flag, a.status);
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
            if (lane == 0) mbar_arrive_remote(rebuilt0 + s * 8u);
            g += 2;
            cursor_step(cur, 2);
        }
    } else {
        // ---- epilogue warps ---------------------------------------------------------
        // Thread e of warp w owns accumulator row r = 32*(w%4) + lane: it rounds the row's
        // tokens to bf16 into sOut[token][r], kParts slices of the token tile in turn; once
        // the four warps have staged a slice, each thread writes 16-byte pieces (8 rows of
        // one token) of it to y.  The accumulator is released after the last slice is read.
        const int sub = warp & 3;
        const int r = sub * 32 + lane;
        const int et = static_cast<int>(threadIdx.x) - kPEpiFirstWarp * 32;
        const uint32_t acc_empty0 = mapa_rank(smem_u32(acc_empty), 0);
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(sub * 32) << 16);
        constexpr int kOut = Shape::kOutTokens;
        bool ok = true;
        uint32_t done = 0;
        for (int u = p0; u < total; u += G, ++done) {
            const PairTile t = pair_tile<kGrouped>(a, u, n_slots);
            const PairLinear &L = a.lin[t.lp];
            const int m0 = t.row0 + static_cast<int>(rank) * kPM;
            if (ok) {
                const bool got = mbar_wait(acc_full, done & 1, a.wait_ns, abort_flag);
                if (__all_sync(0xFFFFFFFFu, got)) {
                    tc_fence_after();
                } else {
                    if (lane == 0) give_up_p(abort_flag, a.status);
                    ok = false;
                }
            }
#pragma unroll 1
            for (int part = 0; part < kParts; ++part) {
                const int t0 = part * kOut;  // first token of the slice
                if (ok) {
#pragma unroll 1
                    for (int c0 = t0; c0 < t0 + kOut; c0 += 32) {
                        if (c0 >= t.count) break;  // warp-uniform
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(lane_addr + c0, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            __nv_bfloat16 hv = __float2bfloat16_rn(__uint_as_float(v[i]));
                            sOut[(c0 - t0 + i) * kPM + r] = *reinterpret_cast<uint16_t *>(&hv);
                        }
                    }
                    if (part == kParts - 1) {
                        // This warp's reads of the accumulator are complete: release it to
                        // the next tile's MMAs.
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote(acc_empty0);
                    }
                }
                epi_bar_sync();  // every warp passes both barriers of every slice, given up or not
                if (ok) {
                    const int64_t n_out = L.n_out;
                    const bool vec = L.y_vec16 != 0;
                    const int ntok = min(t.count - t0, kOut);
#pragma unroll 1
                    for (int idx = et; idx < ntok * (kPM / 8); idx += kPEpiWarps * 32) {
                        const int tl = idx / (kPM / 8);  // token within the slice
                        const int c = idx - tl * (kPM / 8);
                        const int tok = t0 + tl;
                        const int64_t row = static_cast<int64_t>(m0) + c * 8;
                        if (row >= n_out || !in_bounds(t.n0 + tok < L.m, a.status)) continue;
                        const int64_t yt = kGrouped ? static_cast<int64_t>(a.perm[t.n0 + tok])
                                                    : static_cast<int64_t>(t.n0) + tok;
                        if (!in_bounds(yt >= 0 && yt < L.m, a.status)) continue;
                        const uint4 w = *reinterpret_cast<const uint4 *>(sOut + tl * kPM + c * 8);
                        uint16_t *dst = L.y + yt * n_out + row;
                        if (vec && row + 8 <= n_out) {
                            *reinterpret_cast<uint4 *>(dst) = w;
                        } else {
                            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                            for (int e = 0; e < 8 && row + e < n_out; ++e)
                                dst[e] = static_cast<uint16_t>(wv[e >> 1] >> (16 * (e & 1)));
                        }
                    }
                }
                epi_bar_sync();  // sOut is free for the next slice
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
    return pairs <= 0x3FFFFFFFLL;
}

// Pair tiles of the shape: 256 W rows x 256 tokens.
int64_t prefill_pair_tiles(int64_t m, int64_t n_out) {
    return ((n_out + 2 * kPM - 1) / (2 * kPM)) * ((m + kPN - 1) / kPN);
}

namespace {

// One launch over `units` tiles: a persistent grid of min(units, SMs / 2) pairs.
template <bool kGrouped, int kStages, int kParts>
cudaError_t launch_pair_shape(const PairMaps &maps, const PairArgs &a, int64_t units, const DevCtx &ctx,
                              cudaStream_t stream) {
    constexpr size_t smem = PairShape<kStages, kParts>::kSmem;
    static bool attr_set[128] = {false};
    if (ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel<kGrouped, kStages, kParts>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    if (units < 1) return cudaSuccess;
    if (units > 0x3FFFFFFFLL) return cudaErrorInvalidValue;
    const int64_t resident = ctx.num_sms / 2 > 0 ? ctx.num_sms / 2 : 1;
    const int64_t pairs = units < resident ? units : resident;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<kGrouped, kStages, kParts>, maps, a);
}

// The kernel's shape for a launch: the 6-deep ring when every linear has at least
// kDeepRingMinKb K blocks, else the 5-deep one with the whole tile staged; the
// BD_OPT_PAIR_RING option forces either (tests, measurements).
constexpr int kDeepRingMinKb = 128;

template <bool kGrouped>
cudaError_t launch_pair(const PairMaps &maps, const PairArgs &a, int64_t units, const DevCtx &ctx,
                        cudaStream_t stream) {
    int min_kb = 1 << 30;
    for (int i = 0; i < a.n_lin; ++i) min_kb = min(min_kb, a.lin[i].num_kb);
    const int64_t forced = option_value(BD_OPT_PAIR_RING);
    const bool deep = forced != 0 ? forced == 2 : min_kb >= kDeepRingMinKb;
    return deep ? launch_pair_shape<kGrouped, 6, 2>(maps, a, units, ctx, stream)
                : launch_pair_shape<kGrouped, 5, 1>(maps, a, units, ctx, stream);
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
    L.y_vec16 = (n_out % 8 == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) ? 1 : 0;
    L.first_pair = first_pair;
    if (!encode_tensor_map_2d(&maps.w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_base, n_in, n_out, n_in * 2, kPK,
                              kPM, CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    for (int b = 0; b < kPXBoxes; ++b)
        if (!encode_tensor_map_2d(&maps.x[i][b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, n_in, x_rows, n_in * 2, kPK,
                                  x_box_rows(b), CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
    return true;
}

}  // namespace

bool prefill_pair_multi_supported(const BatchItem *items, int n, const DevCtx &ctx) {
    if (n < 1 || n > kPMaxLinears) return false;
    int64_t tiles = 0;
    for (int i = 0; i < n; ++i) {
        if (!prefill_pair_supported(items[i].m, items[i].n_out, items[i].n_in, ctx)) return false;
        tiles += prefill_pair_tiles(items[i].m, items[i].n_out);
    }
    return tiles <= 0x3FFFFFFFLL;
}

cudaError_t launch_prefill_pair_multi(const BatchItem *items, int n, const DevCtx &ctx, cudaStream_t stream) {
    if (!prefill_pair_multi_supported(items, n, ctx)) return cudaErrorNotSupported;
    PairMaps maps;
    PairArgs a = {};
    a.n_lin = n;
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;
    int64_t tiles = 0;
    for (int i = 0; i < n; ++i) {
        const BatchItem &it = items[i];
        if (!fill_linear(maps, a, i, it.x, it.m, it.w_base, it.bits, it.alpha, it.alpha_mode, it.m, it.n_out, it.n_in,
                         it.y, static_cast<int32_t>(tiles)))
            return cudaErrorInvalidValue;
        tiles += prefill_pair_tiles(it.m, it.n_out);
    }
    a.n_units = static_cast<int32_t>(tiles);
    return launch_pair<false>(maps, a, tiles, ctx, stream);
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
    const int64_t units = static_cast<int64_t>(a.lin[0].row_tiles) * tab.max_slots;
    if (units > 0x3FFFFFFFLL) return cudaErrorInvalidValue;
    a.n_units = static_cast<int32_t>(units);
    return launch_pair<true>(maps, a, units, ctx, stream);
}

}  // namespace bd
