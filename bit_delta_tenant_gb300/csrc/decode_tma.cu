// decode_tma.cu -- the HBM-streaming fused BitDelta linear for small token
// counts, fed by TMA.  Same arithmetic as decode.cu (distributive form
// y = x.W_base^T + alpha * (x.S^T) on mma.m16n8k16, signs built in registers),
// but W_base, the packed bits and the activations arrive through a multi-stage
// ring of shared-memory tiles filled by one producer warp with cp.async.bulk.tensor,
// so each SM keeps well over 100 KB of HBM reads in flight for a handful of
// instructions.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": one fused kernel reads
// the base weights and the delta bits together and rebuilds the effective
// weight on chip, never writing W_eff to HBM (conceptual fused_bitdelta_linear
// listing).
//
// CTA (one per SM): R row groups of 16 W rows (R = 1..8, chosen per shape so
// that the busiest SM streams as little as possible), 2R consumer warps + 1
// producer warp.  A stage is a 128-column K step: two (16R x 64) bf16 W boxes
// (128-byte swizzle), one 16R x 16-byte box of packed bits and two (8*NT
// tokens x 64 columns) activation boxes (128-byte swizzle; rows beyond m
// arrive as zeros).  Consumer warp w owns row group w % R (16 rows, the M side
// of the MMA) and 64-column half w / R of every stage.  Lane (g, t) reads
// 16-byte chunks 2t and 2t+1 of rows g and g+8 -- with the swizzle the eight
// lanes of a shared-memory phase hit eight different bank groups -- so its 16
// columns are 16t..16t+15 of the half, and the k-slots of the four MMAs per
// half map to those columns in order, identically for the activations.  A
// cluster of C CTAs splits K; partials are added across the two halves in
// shared memory, and across the cluster by push: rank c owns a share of the
// block's rows, every other rank stores its partial of those rows straight
// into c's shared-memory inbox with st.async (the bytes counted on c's
// mbarrier), and c adds the ranks' partials in rank order (a fixed order) and
// writes y.  No rank reads another's shared memory, so none waits for its
// peers before it exits.
// Launches allow programmatic dependent launch: the next kernel on the stream
// may start its prologue while this one drains.  Every global read comes after
// griddepcontrol.wait, so data written by the previous kernel is seen -- except,
// when the caller enabled weight prefetch, the first stages' W_base and bits
// boxes, which are issued before the wait.
#include <cooperative_groups.h>

#include <cstdio>
#include <cstdlib>

#include "bd_internal.h"
#include "decode_stage.cuh"

namespace cg = cooperative_groups;

namespace bd {
namespace {

using dstage::kStepK;
using dstage::StageLayout;
using dstage::stage_layout;

constexpr int kMaxSmem = 227 * 1024;        // opt-in dynamic shared memory per CTA on sm_103
constexpr size_t kSmemPerSm = 228 * 1024;   // shared memory of one SM (1 KB of it reserved per CTA)

__host__ __device__ constexpr uint32_t red_bytes(int rg, int nt) { return 8u * nt * 16u * rg * 4u; }
// Inbox of the cluster reduction: [sender rank][token][owned row], at most (rows + 8) x MP floats.
__host__ __device__ constexpr uint32_t inbox_bytes(int rg, int nt) { return (16u * rg + 8u) * 8u * nt * 4u; }
inline size_t smem_bytes(int rg, int nt, int stages) {
    return 1024 + static_cast<size_t>(stages) * stage_layout(rg, nt).stage + red_bytes(rg, nt) + inbox_bytes(rg, nt) +
           (2 * stages + 1) * 8 + 16;
}

// One launch streams up to kTmaMaxLinears independent linears (bd_linear_batch);
// bd_linear is a list of one.  Linear p owns CTAs [first_cta, first_cta + blocks *
// cluster), so no cluster spans two linears.
constexpr int kTmaMaxLinears = 8;
struct TmaLinear {
    const float *alpha;
    uint16_t *y;
    int64_t m, n_out, n_in;
    int64_t ks;           // K columns per cluster rank
    int32_t mode;
    int32_t first_cta;
};
struct TmaMaps {
    CUtensorMap w[kTmaMaxLinears];
    CUtensorMap b[kTmaMaxLinears];
    CUtensorMap x[kTmaMaxLinears];
};
struct TmaDecodeArgs {
    TmaLinear lin[kTmaMaxLinears];
    int32_t n_lin;
    int32_t cluster;
    int32_t rg;                // row groups of 16 rows per CTA
    int32_t stages;            // ring depth
    int32_t prefetch_weights;  // issue the first stages' W and bits boxes before griddepcontrol.wait
    unsigned *status;
    uint64_t wait_ns;
};

__device__ __forceinline__ void give_up(volatile int *abort_flag, unsigned *status) {
    *abort_flag = 1;
    flag_status(status, kDevTimeout);
}

template <int NT, int RG>
__global__ void __launch_bounds__(32 * (2 * RG + 1), NT <= 2 && RG <= 4 ? 2 : 1)
    decode_tma_kernel(const __grid_constant__ TmaMaps maps, const __grid_constant__ TmaDecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int MP = 8 * NT;
    constexpr int rg_n = RG;
    constexpr int rows = 16 * RG;
    constexpr int n_cons = 2 * RG;  // consumer warps: row group w % R, K half w / R
    const int kStages = a.stages;
    constexpr StageLayout L = stage_layout(RG, NT);
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *red = reinterpret_cast<float *>(smem + kStages * L.stage);
    float *inbox = red + red_bytes(rg_n, NT) / 4;
    uint64_t *full = reinterpret_cast<uint64_t *>(inbox + inbox_bytes(rg_n, NT) / 4);
    uint64_t *empty = full + kStages;
    uint64_t *inbox_bar = empty + kStages;  // completes when every peer's rows of this rank have landed
    volatile int *abort_flag = reinterpret_cast<volatile int *>(inbox_bar + 1);

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    int lp = 0;  // this CTA's linear
    while (lp + 1 < a.n_lin && a.lin[lp + 1].first_cta <= static_cast<int>(blockIdx.x)) ++lp;
    const TmaLinear &P = a.lin[lp];
    const CUtensorMap *tm_w = &maps.w[lp], *tm_b = &maps.b[lp], *tm_x = &maps.x[lp];
    const int64_t row_block = (blockIdx.x - P.first_cta) / a.cluster;
    const int row0 = static_cast<int>(row_block * rows);
    const int64_t k_lo = static_cast<int64_t>(rank) * P.ks;
    const int64_t k_hi = min(k_lo + P.ks, P.n_in);
    const int n_steps = k_hi > k_lo ? static_cast<int>((k_hi - k_lo + kStepK - 1) / kStepK) : 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool is_producer = warp == n_cons;

    // Cluster reduction by push: rank c owns rows [c*share, c*share + owned(c)) of the block;
    // each peer stores its partial of those rows into c's inbox (st.async, counted in bytes
    // on c's inbox barrier), and c adds the ranks' partials in rank order.
    const int share = (rows + a.cluster - 1) / a.cluster;
    const int m_here = static_cast<int>(P.m < MP ? P.m : MP);
    auto owned = [&](int q) { return max(0, min(share, rows - q * share)); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], n_cons);
        }
        mbar_init(inbox_bar, 1);
        mbar_arrive_expect_tx(inbox_bar,
                              static_cast<uint32_t>((a.cluster - 1) * owned(rank) * m_here) * sizeof(float));
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    cluster_arrive_release();  // peers push into this CTA only after they have seen its barriers initialised
    pdl_trigger();
    const int n_pre = a.prefetch_weights ? min(n_steps, kStages) : 0;
    if (is_producer && lane == 0 && n_pre > 0) {
        // Weights are not written by the preceding kernel (the caller's
        // promise): start streaming them before that kernel completes.
        tma_prefetch_desc(tm_w);
        tma_prefetch_desc(tm_b);
        for (int i = 0; i < n_pre; ++i) {
            const int kc = static_cast<int>(k_lo) + i * kStepK;
            uint8_t *st = smem + i * L.stage;
            mbar_arrive_expect_tx(&full[i], L.tx);
            tma_load_2d(st, tm_w, &full[i], kc, row0);
            tma_load_2d(st + L.w_box, tm_w, &full[i], kc + 64, row0);
            tma_load_2d(st + L.bits_off, tm_b, &full[i], kc / 8, row0);
        }
    }
    pdl_wait();

    float accb[NT][4], accs[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) accb[i][j] = accs[i][j] = 0.0f;

    const int g = lane >> 2, t = lane & 3;
    const int rgi = warp % rg_n;   // row group
    const int kh = warp / rg_n;    // 64-column half of each stage
    const int r0 = rgi * 16 + g;   // tile rows r0, r0 + 8

    if (is_producer) {
        // ---- producer ----
        if (lane == 0) {
            tma_prefetch_desc(tm_w);
            tma_prefetch_desc(tm_b);
            tma_prefetch_desc(tm_x);
            for (int i = 0; i < n_pre; ++i) {  // the activations of the prefetched stages
                const int kc = static_cast<int>(k_lo) + i * kStepK;
                uint8_t *st = smem + i * L.stage;
                tma_load_2d(st + L.x_off, tm_x, &full[i], kc, 0);
                tma_load_2d(st + L.x_off + L.x_box, tm_x, &full[i], kc + 64, 0);
            }
            int issued = n_pre;
            int s = n_pre % kStages;  // slot and phase advance incrementally (the ring depth is a launch value)
            uint32_t ph = (n_pre / kStages) & 1;
            for (int i = n_pre; i < n_steps; ++i, (++s == kStages ? (s = 0, ph ^= 1u) : 0u)) {
                if (!mbar_wait(&empty[s], ph ^ 1, a.wait_ns, abort_flag)) {
                    give_up(abort_flag, a.status);
                    break;
                }
                const int kc = static_cast<int>(k_lo) + i * kStepK;
                uint8_t *st = smem + s * L.stage;
                mbar_arrive_expect_tx(&full[s], L.tx);
                tma_load_2d(st, tm_w, &full[s], kc, row0);
                tma_load_2d(st + L.w_box, tm_w, &full[s], kc + 64, row0);
                tma_load_2d(st + L.bits_off, tm_b, &full[s], kc / 8, row0);
                tma_load_2d(st + L.x_off, tm_x, &full[s], kc, 0);
                tma_load_2d(st + L.x_off + L.x_box, tm_x, &full[s], kc + 64, 0);
                issued = i + 1;
            }
            // Every copy issued has landed before the CTA can exit, also when the consumers gave up
            // after this loop ended (in a normal run these phases are complete and the waits return).
            for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
                mbar_wait(&full[i % kStages], (i / kStages) & 1, kDrainLimitNs, nullptr);
        }
    } else {
        // ---- consumers ----
        // Token rows of the x boxes use the same swizzle term as W rows: (8*tt + g) & 7 == r0 & 7 == g.
        const dstage::LaneSwizzle sw = dstage::lane_swizzle(t, r0);
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; i < n_steps; ++i, (++s == kStages ? (s = 0, ph ^= 1u) : 0u)) {
            const bool got = mbar_wait(&full[s], ph, a.wait_ns, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) give_up(abort_flag, a.status);
                break;
            }
            dstage::consume_stage<NT>(smem + s * L.stage, L, kh, r0, g, t, sw, accb, accs);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        // ---- fold alpha, add the two halves ----
        const int64_t grow0 = static_cast<int64_t>(row0) + r0;
        const bool v0 = grow0 < P.n_out, v1 = grow0 + 8 < P.n_out;
        const float al0 = v0 ? (P.mode ? P.alpha[grow0] : P.alpha[0]) : 0.0f;
        const float al1 = v1 ? (P.mode ? P.alpha[grow0 + 8] : P.alpha[0]) : 0.0f;
        float part[NT][4];
        dstage::fold_alpha<NT>(accb, accs, al0, al1, part);
        if (kh == 1) dstage::halves_store<NT>(red, rows, r0, t, part);
        asm volatile("bar.sync 1, %0;" ::"n"(32 * n_cons) : "memory");  // consumer warps only
        if (kh == 0) dstage::halves_add<NT>(red, rows, r0, t, part);
        asm volatile("bar.sync 1, %0;" ::"n"(32 * n_cons) : "memory");  // red complete
    }
    __syncwarp();
    cluster_wait_acquire();  // every peer's inbox barrier is initialised
    if (is_producer) return;

    // ---- push the rows other ranks own (this rank's partial; garbage after a timeout, but always sent) ----
    const int ctid = threadIdx.x;  // consumer threads: 0 .. 32 * n_cons - 1
    const uint32_t inbox_addr = smem_u32(inbox), bar_addr = smem_u32(inbox_bar);
    for (int e = ctid; e < m_here * rows; e += 32 * n_cons) {
        const int tok = e / rows, lr = e - tok * rows;
        const int q = lr / share;
        if (q == rank) continue;
        const uint32_t idx = static_cast<uint32_t>((rank * MP + tok) * share + (lr - q * share));
        st_async_remote_f32(mapa_rank(inbox_addr + idx * 4u, q), red[tok * rows + lr], mapa_rank(bar_addr, q));
    }
    // ---- add this rank's rows over the cluster in rank order and write y ----
    const int mine = owned(rank);
    if (mine == 0) return;
    // Peers push unconditionally (also after a timeout of their own), so this wait runs out only
    // if a peer has stalled for the wait limit plus a further second.  The kernel then flags a
    // timeout and this CTA exits without the closing cluster barrier that would otherwise order
    // late pushes before its exit: a push still in flight may then land in the shared memory the
    // SM hands to a later CTA.  The status word reports the launch as failed in that case, and
    // no closing barrier is paid in the normal case (measured: it costs every launch its tail).
    if (!mbar_wait(inbox_bar, 0, a.wait_ns + kDrainLimitNs, nullptr)) {
        if (ctid == 0) flag_status(a.status, kDevTimeout);
        return;
    }
    for (int e = ctid; e < m_here * mine; e += 32 * n_cons) {
        const int tok = e / mine, lrl = e - tok * mine;
        const int lr = rank * share + lrl;
        const int64_t row = static_cast<int64_t>(row0) + lr;
        float s = 0.0f;
        for (int q = 0; q < a.cluster; ++q)
            s += q == rank ? red[tok * rows + lr] : inbox[(q * MP + tok) * share + lrl];
        if (row < P.n_out && in_bounds(tok < P.m, a.status)) {
            __nv_bfloat16 h = __float2bfloat16_rn(s);
            P.y[static_cast<int64_t>(tok) * P.n_out + row] = *reinterpret_cast<uint16_t *>(&h);
        }
    }
}

struct TmaPlan {
    int nt, cluster, rg, stages;
    int64_t ks, row_blocks;
};

template <int NT, int RG>
cudaError_t ensure_smem_attr(int device) {
    static bool attr_set[128] = {false};
    if (device >= 0 && device < 128 && attr_set[device]) return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(decode_tma_kernel<NT, RG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e == cudaSuccess && device >= 0 && device < 128) attr_set[device] = true;
    return e;
}

// The (NT, R) pairs the plan can produce are instantiated: R = 4 everywhere,
// 5..8 for m <= 16 (the balanced split of row counts just above 64 x SMs),
// 7 for m <= 32.
bool plan_instantiated(int nt, int rg) { return rg == 4 || (nt <= 2 && rg >= 5 && rg <= 8) || (nt == 4 && rg == 7); }

// Deepest ring whose CTA fits in `budget` bytes of shared memory.
int stages_within(int rg, int nt, size_t budget) {
    int s = 8;
    while (s > 0 && smem_bytes(rg, nt, s) > budget) --s;
    return s;
}

// Launch plan: R (16-row groups per CTA), C (ranks splitting K in a
// cluster) and the ring depth, from sweeps of this kernel on GB300 (rows x
// K from 1024 x 4096 to 28672 x 8192, m = 1 .. 64):
//  * m <= 16: 64-row CTAs (R = 4), two per SM (rings of 5 / 4 stages of
//    19 / 21 KB), which lets the next launch's CTAs start prefetching on an
//    SM while this launch's second CTA drains.  K is split over a cluster
//    when the row blocks alone leave SMs idle: C = ceil(1.5 * SMs / blocks).
//    When the 64-row blocks exceed the SM count by at most a quarter (11008
//    rows -> 172 blocks), some SMs would stream two blocks while others
//    stream one; there R = ceil(groups / SMs) row groups per block, split in
//    two along K, puts two equal half-blocks on nearly every SM instead
//    (measured 17.4 us against 21.9 us for 11008 x 4096).
//  * 16 < m <= 32: the widest CTA the registers allow (R = 7, 14 consumer
//    warps), one per SM, when its blocks times a K split fill at least 90% of
//    the SMs in one wave -- the MMA work per byte has grown (8192 x 8192:
//    35.6 us against 44.5 us with R = 4); otherwise as below.
//  * 32 < m <= 64: R = 4, one CTA per SM.
bool make_tma_plan(int64_t m, int64_t n_out, int64_t n_in, const DevCtx &ctx, TmaPlan &p) {
    const int num_sms = ctx.num_sms;
    if (m < 1 || m > kDecodeMaxM || n_out < 1 || n_in < 1 || num_sms < 1) return false;
    p.nt = m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8;
    const int64_t groups = (n_out + 15) / 16;
    const int64_t steps = (n_in + kStepK - 1) / kStepK;
    int rg = 4;
    int c = 0;
    int stages = p.nt == 1 ? 5 : p.nt == 2 ? 4 : 8;
    const int64_t blocks7 = (groups + 6) / 7;
    if (p.nt == 4 && blocks7 <= num_sms) {
        const int64_t c7 = num_sms / blocks7 < 8 ? num_sms / blocks7 : 8;
        if (10 * blocks7 * c7 >= 9 * static_cast<int64_t>(num_sms)) rg = 7, c = static_cast<int>(c7);
    }
    const int64_t blocks4 = (groups + 3) / 4;
    if (p.nt <= 2 && blocks4 > num_sms && 4 * blocks4 <= 5 * static_cast<int64_t>(num_sms)) {
        const int64_t r = (groups + num_sms - 1) / num_sms;
        if (r <= 8) {
            rg = static_cast<int>(r);
            c = 2;
            stages = stages_within(rg, p.nt, kSmemPerSm / 2 - 1024);
        }
    }
    if (!plan_instantiated(p.nt, rg)) rg = 4;
    const int64_t blocks = (groups + rg - 1) / rg;
    if (c == 0) c = blocks >= num_sms ? 1 : static_cast<int>((3 * static_cast<int64_t>(num_sms) / 2 + blocks - 1) / blocks);
    if (c > 8) c = 8;
    if (c > steps) c = static_cast<int>(steps);
    const int deepest = stages_within(rg, p.nt, kMaxSmem);
    if (stages > deepest) stages = deepest;
    if (stages < 3) return false;
    const int64_t per = (steps + c - 1) / c;
    p.rg = rg;
    p.stages = stages;
    p.ks = per * kStepK;
    p.cluster = static_cast<int>((steps + per - 1) / per);  // no empty ranks
    p.row_blocks = blocks;
    if (p.row_blocks * p.cluster > 0x7FFFFFFFLL) return false;
    return true;
}

template <int NT, int RG>
cudaError_t launch_plan(const TmaMaps &maps, const TmaDecodeArgs &a, int64_t ctas, const TmaPlan &p,
                        const DevCtx &ctx, cudaStream_t stream) {
    cudaError_t e = ensure_smem_attr<NT, RG>(ctx.device);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * (2 * RG + 1)), 1, 1);
    cfg.dynamicSmemBytes = smem_bytes(RG, NT, p.stages);
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
    return cudaLaunchKernelEx(&cfg, decode_tma_kernel<NT, RG>, maps, a);
}

cudaError_t launch_any(const TmaMaps &maps, const TmaDecodeArgs &a, int64_t ctas, const TmaPlan &p,
                       const DevCtx &ctx, cudaStream_t stream) {
#define BD_DECODE_CASE(NT_, RG_) \
    if (p.nt == NT_ && p.rg == RG_) return launch_plan<NT_, RG_>(maps, a, ctas, p, ctx, stream);
    BD_DECODE_CASE(1, 4) BD_DECODE_CASE(1, 5) BD_DECODE_CASE(1, 6) BD_DECODE_CASE(1, 7) BD_DECODE_CASE(1, 8)
    BD_DECODE_CASE(2, 4) BD_DECODE_CASE(2, 5) BD_DECODE_CASE(2, 6) BD_DECODE_CASE(2, 7) BD_DECODE_CASE(2, 8)
    BD_DECODE_CASE(4, 4) BD_DECODE_CASE(4, 7) BD_DECODE_CASE(8, 4)
#undef BD_DECODE_CASE
    return cudaErrorNotSupported;
}

// Tensor maps and entry of linear i of a launch with `rows`-row blocks and token tiles of MP rows.
bool fill_linear(TmaMaps &maps, TmaDecodeArgs &a, int i, const void *x, int64_t m, const void *w_base,
                 const uint8_t *bits, const float *alpha, int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y,
                 uint32_t rows, int mp, int64_t ks, int64_t first_cta) {
    if (!encode_tensor_map_2d(&maps.w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_base, n_in, n_out, n_in * 2, 64, rows,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&maps.b[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, bits, n_in / 8, n_out, n_in / 8, 16, rows,
                              CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tensor_map_2d(&maps.x[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, n_in, m, n_in * 2, 64,
                              static_cast<uint32_t>(mp), CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    if (first_cta > 0x7FFFFFFFLL) return false;
    TmaLinear &l = a.lin[i];
    l.alpha = alpha;
    l.y = static_cast<uint16_t *>(y);
    l.m = m;
    l.n_out = n_out;
    l.n_in = n_in;
    l.ks = ks;
    l.mode = alpha_mode;
    l.first_cta = static_cast<int32_t>(first_cta);
    return true;
}

void fill_common(TmaDecodeArgs &a, const TmaPlan &p, int n_lin, const DevCtx &ctx) {
    a.n_lin = n_lin;
    a.cluster = p.cluster;
    a.rg = p.rg;
    a.stages = p.stages;
    a.prefetch_weights = ctx.weight_prefetch ? 1 : 0;
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;
}

}  // namespace

bool decode_tma_supported(int64_t m, int64_t n_out, int64_t n_in, const void *w_base, const uint8_t *bits,
                          const DevCtx &ctx) {
    if (n_in % kStepK != 0) return false;  // packed-bit rows must be 16-byte multiples for TMA
    if ((reinterpret_cast<uintptr_t>(w_base) & 15) || (reinterpret_cast<uintptr_t>(bits) & 15)) return false;
    if (n_in >= (int64_t(1) << 31) - kStepK) return false;
    TmaPlan p;
    return make_tma_plan(m, n_out, n_in, ctx, p);
}

cudaError_t launch_decode_tma(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                              int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                              cudaStream_t stream) {
    TmaPlan p;
    if (!make_tma_plan(m, n_out, n_in, ctx, p)) return cudaErrorNotSupported;
    TmaMaps maps;
    TmaDecodeArgs a{};
    if (!fill_linear(maps, a, 0, x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y,
                     static_cast<uint32_t>(16 * p.rg), 8 * p.nt, p.ks, 0))
        return cudaErrorInvalidValue;
    fill_common(a, p, 1, ctx);
    return launch_any(maps, a, p.row_blocks * p.cluster, p, ctx, stream);
}

bool decode_tma_multi_supported(const BatchItem *items, int n) {
    if (n < 1 || n > kTmaMaxLinears) return false;
    for (int i = 0; i < n; ++i)
        if (items[i].m < 1 || items[i].m > 16 || items[i].n_in % kStepK != 0 ||
            items[i].n_in >= (int64_t(1) << 31) - kStepK || (reinterpret_cast<uintptr_t>(items[i].w_base) & 15) ||
            (reinterpret_cast<uintptr_t>(items[i].bits) & 15))
            return false;
    return true;
}

// Several linears (m <= 16) in one launch of the cluster-split kernel: CTAs of R row groups (64
// rows unless the rule below applies), two per SM, one K split C for all of them from their blocks
// together, the same rule as for one linear (C = ceil(1.5 * SMs / blocks) while the blocks leave
// SMs idle; BD_DECODE_CLUSTER overrides).
struct MultiShape {
    int64_t mmax, blocks, min_steps;
    int cluster, rg;
};
// As for one linear, when the 64-row blocks exceed the SMs by less than a factor of two at m <= 8,
// taller CTAs split in two along K balance the SMs better: R = ceil(groups / SMs) up to 6 (a ring
// of three stages at two CTAs per SM), C = 2 (3 x 4096^2, m = 1: 18.2 against 19.7 us; at m = 16
// the shallower ring loses, 26.3 against 23.0, so R stays 4 there).  BD_MULTI_RG overrides R.
MultiShape multi_shape(const BatchItem *items, int n, const DevCtx &ctx) {
    MultiShape m{0, 0, -1, 1, 4};
    int64_t groups = 0, blocks4 = 0;
    for (int i = 0; i < n; ++i) {
        m.mmax = items[i].m > m.mmax ? items[i].m : m.mmax;
        groups += (items[i].n_out + 15) / 16;
        blocks4 += (items[i].n_out + 63) / 64;
        const int64_t st = items[i].n_in / kStepK;
        m.min_steps = m.min_steps < 0 || st < m.min_steps ? st : m.min_steps;
    }
    int c = 0;
    const int64_t sms = ctx.num_sms;
    if (m.mmax <= 8 && blocks4 > sms && blocks4 < 2 * sms) {
        const int64_t r = (groups + sms - 1) / sms;
        if (r <= 6) m.rg = static_cast<int>(r), c = 2;
    }
    if (m.rg < 4 || m.rg > 8) m.rg = 4;
    const int64_t rows = 16 * m.rg;
    for (int i = 0; i < n; ++i) m.blocks += (items[i].n_out + rows - 1) / rows;
    if (c == 0 || m.rg == 4)
        c = m.blocks >= sms ? 1 : static_cast<int>((3 * sms / 2 + m.blocks - 1) / m.blocks);
    if (c > 8) c = 8;
    if (c > m.min_steps) c = static_cast<int>(m.min_steps);
    m.cluster = c < 1 ? 1 : c;
    return m;
}

bool decode_tma_multi_one_wave(const BatchItem *items, int n, const DevCtx &ctx) {
    if (!decode_tma_multi_supported(items, n)) return false;
    const MultiShape m = multi_shape(items, n, ctx);
    return m.blocks * m.cluster <= 2 * static_cast<int64_t>(ctx.num_sms);  // two CTAs per SM
}

cudaError_t launch_decode_tma_multi(const BatchItem *items, int n, const DevCtx &ctx, cudaStream_t stream) {
    if (!decode_tma_multi_supported(items, n)) return cudaErrorNotSupported;
    const MultiShape ms = multi_shape(items, n, ctx);
    const int c = ms.cluster;
    TmaPlan p;
    p.nt = ms.mmax <= 8 ? 1 : 2;
    p.rg = plan_instantiated(p.nt, ms.rg) ? ms.rg : 4;
    p.cluster = c;
    p.stages = p.rg == 4 ? (p.nt == 1 ? 5 : 4) : stages_within(p.rg, p.nt, kSmemPerSm / 2 - 1024);  // two per SM
    if (p.stages < 3) return cudaErrorNotSupported;
    const int64_t rows = 16 * p.rg;
    TmaMaps maps;
    TmaDecodeArgs a{};
    int64_t first = 0;
    for (int i = 0; i < n; ++i) {
        const BatchItem &it = items[i];
        const int64_t steps = it.n_in / kStepK;
        const int64_t ks = (steps + c - 1) / c * kStepK;
        if (!fill_linear(maps, a, i, it.x, it.m, it.w_base, it.bits, it.alpha, it.alpha_mode, it.n_out, it.n_in, it.y,
                         static_cast<uint32_t>(rows), 8 * p.nt, ks, first))
            return cudaErrorInvalidValue;
        first += (it.n_out + rows - 1) / rows * c;
    }
    fill_common(a, p, n, ctx);
    return launch_any(maps, a, first, p, ctx, stream);
}

}  // namespace bd
