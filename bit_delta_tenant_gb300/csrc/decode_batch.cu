// decode_batch.cu -- the HBM-streaming fused BitDelta linear over a list of
// independent small-m linears in one launch, with the work split evenly over
// the resident CTAs.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": one fused pass reads the
// base weights and the packed delta bits together and never writes W_eff to
// HBM.  The arithmetic is the distributive form of decode_stage.cuh.
//
// Work split: a work item is one 128-column K step of one 64-row block of one
// linear.  Items are numbered linear by linear, row block by row block, K step
// fastest; CTA g of G takes items [T*g/G, T*(g+1)/G), so every CTA streams the
// same number of bytes (to within one item) through its TMA ring, across row
// block and linear boundaries without draining the ring.  A row block covered
// by one CTA is written directly.  Otherwise the block's first K range is the
// END of its owner CTA's item range and its other K ranges START the ranges
// of the CTAs after it: those CTAs write their fp32 partials (alpha folded
// in) to their own workspace slots and count them on the block's counter as
// soon as they have them, and the owner, once it has its own part, waits
// (bounded) for the count, adds the partials in K order -- a fixed order,
// so y is deterministic -- writes y and resets the counter to zero for the
// next launch.  A CTA only ever waits for CTAs with higher indices, which
// never wait for it, and all CTAs of a launch fit on the GPU at once.
//
// CTA: 4 row groups of 16 rows (64 W rows), 8 consumer warps (row group x K
// half) and one TMA producer warp, as in decode_tma.cu, plus an epilogue warp:
// at the end of its part of a row block the consumers add their K halves into
// one of two shared-memory buffers and go on with the next block's stages,
// while the epilogue warp writes y -- or publishes the partial and counts it,
// or, in the block's owner, adds the partials -- so the ring never waits on
// global memory round trips.  Launches allow programmatic dependent launch;
// with weight prefetch enabled the first stages' W_base and bits boxes are
// issued before griddepcontrol.wait, every other global access after it.
#include <cstdlib>

#include "bd_internal.h"
#include "decode_stage.cuh"

namespace bd {
namespace {

using dstage::kStepK;
using dstage::StageLayout;
using dstage::stage_layout;

constexpr int kRG = 4;                         // row groups of 16 rows per block
constexpr int kRows = 16 * kRG;                // W rows per block
constexpr int kConsumers = 2 * kRG;            // consumer warps: row group w % 4, K half w / 4
constexpr int kProducerWarp = kConsumers;      // issues the TMA copies (lane 0)
constexpr int kEpilogueWarp = kConsumers + 1;  // writes y or partials, completes shared blocks
constexpr int kThreads = 32 * (kConsumers + 2);
constexpr int kMaxSmem = 227 * 1024;

struct BatchProblem {
    const float *alpha;
    uint16_t *y;
    int64_t first_item;  // index of this linear's first work item
    int64_t m, n_out;
    int32_t mode;        // 0: scalar alpha, 1: per-row alpha
    int32_t steps;       // K steps of 128 columns
    int32_t blocks;      // 64-row blocks
    int32_t block0;      // its first block in the launch's block numbering (counters, slots)
};

struct BatchMaps {
    CUtensorMap w[kBatchMaxProblems];
    CUtensorMap b[kBatchMaxProblems];
    CUtensorMap x[kBatchMaxProblems];
};

struct BatchArgs {
    BatchProblem prob[kBatchMaxProblems];
    int32_t n_prob;
    int32_t stages;
    int32_t prefetch_weights;
    int32_t parts_max;      // partial slots per row block
    int64_t total_items;
    float *partials;        // [blocks][parts_max][MP x kRows] fp32
    unsigned *counters;     // [blocks], zero between launches
    unsigned *status;
    uint64_t wait_ns;
};

// Position of a work item: linear p, row block rb, K step s.
struct Cursor {
    int p, rb, s;
};
__device__ __forceinline__ Cursor locate(const BatchArgs &a, int64_t item) {
    int p = 0;
    while (p + 1 < a.n_prob && a.prob[p + 1].first_item <= item) ++p;
    const int64_t r = item - a.prob[p].first_item;
    Cursor c;
    c.p = p;
    c.rb = static_cast<int>(r / a.prob[p].steps);
    c.s = static_cast<int>(r - static_cast<int64_t>(c.rb) * a.prob[p].steps);
    return c;
}
__device__ __forceinline__ void advance(const BatchArgs &a, Cursor &c) {
    if (++c.s == a.prob[c.p].steps) {
        c.s = 0;
        if (++c.rb == a.prob[c.p].blocks) {
            c.rb = 0;
            ++c.p;
        }
    }
}
// The CTA whose item range holds `item`: the largest g with T*g/G <= item.
__device__ __forceinline__ int64_t owner_of(int64_t item, int64_t total, int64_t grid) {
    return ((item + 1) * grid + total - 1) / total - 1;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Barrier of the consumer warps (named barrier 1) that also ORs a predicate
// over them, so that every consumer warp takes the same branch after it.
__device__ __forceinline__ bool consumers_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "n"(32 * kConsumers)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory");
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_batch_kernel(const __grid_constant__ BatchMaps maps, const __grid_constant__ BatchArgs a) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int MP = 8 * NT;
    constexpr int kRed = MP * kRows;  // floats of one block's partial, [token][row]
    constexpr StageLayout L = stage_layout(kRG, NT);
    const int kStages = a.stages;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *red = reinterpret_cast<float *>(smem + kStages * L.stage);  // two buffers of kRed floats
    uint64_t *full = reinterpret_cast<uint64_t *>(red + 2 * kRed);
    uint64_t *empty = full + kStages;
    uint64_t *red_full = empty + kStages;  // [2]: a block's partial is in red[b]
    uint64_t *red_empty = red_full + 2;    // [2]: the epilogue warp is done with red[b]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(red_empty + 2);

    const int64_t grid = gridDim.x;
    const int64_t lo = a.total_items * blockIdx.x / grid;
    const int64_t hi = a.total_items * (blockIdx.x + 1) / grid;
    const int n_items = static_cast<int>(hi - lo);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&red_full[b], 32 * kConsumers);
            mbar_init(&red_empty[b], 1);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    pdl_trigger();

    auto issue_w = [&](const Cursor &c, uint8_t *st, uint64_t *bar) {
        const int kc = c.s * kStepK, row0 = c.rb * kRows;
        tma_load_2d(st, &maps.w[c.p], bar, kc, row0);
        tma_load_2d(st + L.w_box, &maps.w[c.p], bar, kc + 64, row0);
        tma_load_2d(st + L.bits_off, &maps.b[c.p], bar, kc / 8, row0);
    };
    auto issue_x = [&](const Cursor &c, uint8_t *st, uint64_t *bar) {
        const int kc = c.s * kStepK;
        tma_load_2d(st + L.x_off, &maps.x[c.p], bar, kc, 0);
        tma_load_2d(st + L.x_off + L.x_box, &maps.x[c.p], bar, kc + 64, 0);
    };
    auto give_up = [&]() {
        *abort_flag = 1;
        flag_status(a.status, kDevTimeout);
    };

    const int n_pre = a.prefetch_weights ? min(n_items, kStages) : 0;
    if (warp == kProducerWarp && lane == 0 && n_pre > 0) {
        // Weights are not written by the preceding kernel (the caller's
        // promise): start streaming them before that kernel completes.
        Cursor c = locate(a, lo);
        for (int i = 0; i < n_pre; ++i, advance(a, c)) {
            mbar_arrive_expect_tx(&full[i], L.tx);
            issue_w(c, smem + i * L.stage, &full[i]);
        }
    }
    pdl_wait();

    if (warp == kProducerWarp) {
        // ---- TMA producer (lane 0) ----
        if (lane == 0) {
            for (int p = 0; p < a.n_prob; ++p) {
                tma_prefetch_desc(&maps.w[p]);
                tma_prefetch_desc(&maps.b[p]);
                tma_prefetch_desc(&maps.x[p]);
            }
            Cursor c = locate(a, lo);
            for (int i = 0; i < n_pre; ++i, advance(a, c)) issue_x(c, smem + i * L.stage, &full[i]);
            int issued = n_pre;
            int s = n_pre % kStages;  // slot and phase advance incrementally
            uint32_t ph = (n_pre / kStages) & 1;
            for (int i = n_pre; i < n_items; ++i, advance(a, c), (++s == kStages ? (s = 0, ph ^= 1u) : 0u)) {
                if (!mbar_wait(&empty[s], ph ^ 1, a.wait_ns, abort_flag)) {
                    give_up();
                    break;
                }
                uint8_t *st = smem + s * L.stage;
                mbar_arrive_expect_tx(&full[s], L.tx);
                issue_w(c, st, &full[s]);
                issue_x(c, st, &full[s]);
                issued = i + 1;
            }
            if (*abort_flag) {  // wait (bounded) for this CTA's copies still in flight
                for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
                    mbar_wait(&full[i % kStages], (i / kStages) & 1, kDrainLimitNs, nullptr);
            }
        }
        return;
    }

    if (warp == kEpilogueWarp) {
        // ---- epilogue: y, or a partial and the fixed-order sum of a shared block ----
        Cursor c = locate(a, lo);
        int seg = 0;
        for (int i = 0; i < n_items; ++i, advance(a, c)) {
            const BatchProblem &P = a.prob[c.p];
            if (!(c.s == P.steps - 1 || i == n_items - 1)) continue;
            const int b = seg & 1;
            const bool got = mbar_wait(&red_full[b], (seg >> 1) & 1, a.wait_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up();
                break;
            }
            ++seg;
            const float *rb = red + b * kRed;
            const int64_t row0 = static_cast<int64_t>(c.rb) * kRows;
            const int m_here = static_cast<int>(P.m < MP ? P.m : MP);
            const int64_t blk_first = P.first_item + static_cast<int64_t>(c.rb) * P.steps;
            const int64_t g_first = owner_of(blk_first, a.total_items, grid);
            const int parts = static_cast<int>(owner_of(blk_first + P.steps - 1, a.total_items, grid) - g_first + 1);
            // lane handles float4 e = lane + 32u (u < kVec) of the valid token rows: 4 rows of one token
            constexpr int kVec = kRed / 4 / 32;
            const int n4 = m_here * (kRows / 4);
            auto store_y = [&](int e, const float4 &v) {
                const int tok = e / (kRows / 4), lr = 4 * (e - tok * (kRows / 4));
                const float sv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (row0 + lr + k < P.n_out && in_bounds(tok < P.m, a.status)) {
                        const __nv_bfloat16 h = __float2bfloat16_rn(sv[k]);
                        P.y[tok * P.n_out + row0 + lr + k] = *reinterpret_cast<const uint16_t *>(&h);
                    }
                }
            };
            if (parts == 1) {
#pragma unroll
                for (int u = 0; u < kVec; ++u)
                    if (lane + 32 * u < n4) store_y(lane + 32 * u, reinterpret_cast<const float4 *>(rb)[lane + 32 * u]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&red_empty[b]);
                continue;
            }
            const int part_i = static_cast<int>(blockIdx.x - g_first);
            const int64_t gblock = P.block0 + c.rb;
            float *slots = a.partials + gblock * a.parts_max * kRed;
            unsigned *counter = a.counters + gblock;
            if (part_i != 0) {
                // a later K range of the block: publish the partial and count it
#pragma unroll
                for (int u = 0; u < kVec; ++u) {
                    const int e = lane + 32 * u;
                    if (e < n4 && in_bounds(part_i < a.parts_max, a.status))
                        reinterpret_cast<float4 *>(slots + part_i * kRed)[e] = reinterpret_cast<const float4 *>(rb)[e];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&red_empty[b]);  // red[b] is free for the consumers again
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(counter, 1u);
                continue;
            }
            // The block's first K range is this CTA's last part of its item range (its
            // other parts start the ranges of the CTAs after it): wait for their count,
            // then add them after this CTA's own partial, in K order.
            bool ready = true;
            if (lane == 0) {
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_gpu(counter) != static_cast<unsigned>(parts - 1)) {
                    if (*abort_flag != 0 || globaltimer_ns() - t0 > a.wait_ns) {
                        ready = false;
                        break;
                    }
                }
            }
            ready = __shfl_sync(0xFFFFFFFFu, ready ? 1 : 0, 0) != 0;
            if (!ready) {
                if (lane == 0) give_up();
                break;
            }
            constexpr int kChunk = kVec < 4 ? kVec : 4;  // float4s per lane and pass (registers)
#pragma unroll
            for (int u0 = 0; u0 < kVec; u0 += kChunk) {
                float4 acc[kChunk];
#pragma unroll
                for (int u = 0; u < kChunk; ++u)
                    if (lane + 32 * (u0 + u) < n4) acc[u] = reinterpret_cast<const float4 *>(rb)[lane + 32 * (u0 + u)];
                for (int q = 1; q < parts; ++q) {
                    const float4 *src = reinterpret_cast<const float4 *>(slots + q * kRed);
                    float4 v[kChunk];
#pragma unroll
                    for (int u = 0; u < kChunk; ++u)  // a part's loads in flight together
                        if (lane + 32 * (u0 + u) < n4) v[u] = __ldcg(src + lane + 32 * (u0 + u));
#pragma unroll
                    for (int u = 0; u < kChunk; ++u)
                        if (lane + 32 * (u0 + u) < n4)
                            acc[u].x += v[u].x, acc[u].y += v[u].y, acc[u].z += v[u].z, acc[u].w += v[u].w;
                }
#pragma unroll
                for (int u = 0; u < kChunk; ++u)
                    if (lane + 32 * (u0 + u) < n4) store_y(lane + 32 * (u0 + u), acc[u]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&red_empty[b]);
            if (lane == 0) a.counters[gblock] = 0u;  // ready for the next launch
        }
        return;
    }

    // ---- consumers ----
    const int g = lane >> 2, t = lane & 3;
    const int rgi = warp % kRG;  // row group
    const int kh = warp / kRG;   // 64-column half of each stage
    const int r0 = rgi * 16 + g;
    const dstage::LaneSwizzle sw = dstage::lane_swizzle(t, r0);
    float accb[NT][4], accs[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) accb[i][j] = accs[i][j] = 0.0f;

    Cursor c = locate(a, lo);
    bool aborted = false;
    int seg = 0;
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < n_items; ++i, advance(a, c), (++s == kStages ? (s = 0, ph ^= 1u) : 0u)) {
        if (!aborted) {
            const bool got = mbar_wait(&full[s], ph, a.wait_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up();
                aborted = true;  // the slot is not released: its copy may still be in flight
            } else {
                dstage::consume_stage<NT>(smem + s * L.stage, L, kh, r0, g, t, sw, accb, accs);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
        }
        const BatchProblem &P = a.prob[c.p];
        if (!(c.s == P.steps - 1 || i == n_items - 1)) continue;
        // ---- the end of this CTA's part of row block (c.p, c.rb): hand it to the epilogue warp ----
        const int b = seg & 1;
        if (!aborted && !mbar_wait(&red_empty[b], ((seg >> 1) & 1) ^ 1, a.wait_ns, abort_flag)) {
            give_up();
            aborted = true;
        }
        if (consumers_any(aborted)) break;  // every consumer warp leaves together
        ++seg;
        const int64_t grow0 = static_cast<int64_t>(c.rb) * kRows + r0;
        const float al0 = grow0 < P.n_out ? (P.mode ? P.alpha[grow0] : P.alpha[0]) : 0.0f;
        const float al1 = grow0 + 8 < P.n_out ? (P.mode ? P.alpha[grow0 + 8] : P.alpha[0]) : 0.0f;
        float part[NT][4];
        dstage::fold_alpha<NT>(accb, accs, al0, al1, part);
        float *rb = red + b * kRed;
        if (kh == 1) dstage::halves_store<NT>(rb, kRows, r0, t, part);
        consumers_sync();
        if (kh == 0) dstage::halves_add<NT>(rb, kRows, r0, t, part);
        mbar_arrive(&red_full[b]);
#pragma unroll
        for (int q = 0; q < NT; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) accb[q][j] = accs[q][j] = 0.0f;
    }
}

// Ring depth: the deepest that keeps two CTAs per SM.
int stages_for(int nt) { return nt == 1 ? 5 : 4; }

size_t smem_for(int nt) {
    const StageLayout L = stage_layout(kRG, nt);
    return 1024 + static_cast<size_t>(stages_for(nt)) * L.stage + 2 * static_cast<size_t>(8 * nt) * kRows * 4 +
           (2 * stages_for(nt) + 4) * 8 + 16;
}

template <int NT>
int resident_per_sm() {
    static int cached = -1;
    if (cached >= 0) return cached;
    if (cudaFuncSetAttribute(decode_batch_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_batch_kernel<NT>, kThreads, smem_for(NT)) !=
        cudaSuccess)
        return 0;
    cached = n;
    return n;
}

}  // namespace

bool decode_batch_supported(int64_t m, int64_t n_out, int64_t n_in, const void *x, const void *w_base,
                            const uint8_t *bits, const void *y) {
    if (m < 1 || m > kBatchMaxM || n_out < 1 || n_in < kStepK || n_in % kStepK != 0) return false;
    if (n_out >= (int64_t(1) << 31) - kRows || n_in >= (int64_t(1) << 31) - kStepK) return false;
    for (const void *p : {x, static_cast<const void *>(w_base), static_cast<const void *>(bits), y})
        if (reinterpret_cast<uintptr_t>(p) & 15) return false;
    return true;
}

BatchPlan plan_decode_batch(const BatchItem *items, int n, const DevCtx &ctx) {
    BatchPlan pl{};
    if (n < 1 || n > kBatchMaxProblems) return pl;
    int64_t mmax = 0, total = 0, blocks = 0, steps_max = 0;
    for (int i = 0; i < n; ++i) {
        mmax = items[i].m > mmax ? items[i].m : mmax;
        const int64_t b = (items[i].n_out + kRows - 1) / kRows, st = items[i].n_in / kStepK;
        total += b * st;
        blocks += b;
        steps_max = st > steps_max ? st : steps_max;
    }
    pl.nt = mmax <= 8 ? 1 : 2;
    const int per_sm = pl.nt == 1 ? resident_per_sm<1>() : resident_per_sm<2>();
    if (per_sm < 1 || total < 1) return pl;
    int64_t grid = static_cast<int64_t>(per_sm) * ctx.num_sms;
    const int64_t forced = option_value(BD_OPT_BATCH_GRID);  // tests: CTAs per launch
    if (forced > 0) grid = forced;
    // every CTA resident at once: an owner may wait for the CTAs after it
    const int64_t resident = static_cast<int64_t>(per_sm) * ctx.num_sms;
    if (grid > resident) grid = resident;
    if (grid > total) grid = total;
    const int64_t q = total / grid;  // items per CTA: q or q + 1
    int64_t parts = (steps_max - 1 + q - 1) / q + 1;
    if (parts > steps_max) parts = steps_max;
    pl.grid = grid;
    pl.total_items = total;
    pl.blocks = blocks;
    pl.parts_max = static_cast<int32_t>(parts);
    pl.counter_bytes = (static_cast<size_t>(blocks) * sizeof(unsigned) + 255) / 256 * 256;
    pl.workspace_bytes =
        pl.counter_bytes + static_cast<size_t>(blocks) * parts * (8 * pl.nt) * kRows * sizeof(float);
    pl.ok = true;
    return pl;
}

cudaError_t launch_decode_batch(const BatchItem *items, int n, const BatchPlan &pl, void *workspace,
                                const DevCtx &ctx, cudaStream_t stream) {
    if (!pl.ok || n < 1 || n > kBatchMaxProblems) return cudaErrorInvalidValue;
    const int mp = 8 * pl.nt;
    BatchMaps maps;
    BatchArgs a{};
    int64_t first = 0;
    int64_t block0 = 0;
    for (int i = 0; i < n; ++i) {
        const BatchItem &it = items[i];
        if (!encode_tensor_map_2d(&maps.w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, it.w_base, it.n_in, it.n_out,
                                  it.n_in * 2, 64, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tensor_map_2d(&maps.b[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, it.bits, it.n_in / 8, it.n_out,
                                  it.n_in / 8, 16, kRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_tensor_map_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, it.x, it.n_in, it.m, it.n_in * 2, 64,
                                  static_cast<uint32_t>(mp), CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        const int64_t blocks = (it.n_out + kRows - 1) / kRows, steps = it.n_in / kStepK;
        BatchProblem &p = a.prob[i];
        p.alpha = it.alpha;
        p.y = static_cast<uint16_t *>(it.y);
        p.first_item = first;
        p.m = it.m;
        p.n_out = it.n_out;
        p.mode = it.alpha_mode;
        p.steps = static_cast<int32_t>(steps);
        p.blocks = static_cast<int32_t>(blocks);
        p.block0 = static_cast<int32_t>(block0);
        first += blocks * steps;
        block0 += blocks;
    }
    if (first != pl.total_items || block0 != pl.blocks || block0 >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    a.n_prob = n;
    a.stages = stages_for(pl.nt);
    a.prefetch_weights = ctx.weight_prefetch ? 1 : 0;
    a.parts_max = pl.parts_max;
    a.total_items = pl.total_items;
    a.counters = static_cast<unsigned *>(workspace);
    a.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + pl.counter_bytes);
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_for(pl.nt);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pl.nt == 1) return cudaLaunchKernelEx(&cfg, decode_batch_kernel<1>, maps, a);
    return cudaLaunchKernelEx(&cfg, decode_batch_kernel<2>, maps, a);
}

}  // namespace bd
