// grouped_decode_tc.cu -- the multi-tenant fused linear for small batches on
// the 5th-generation tensor cores: one HBM pass over the shared W_base and
// over every active variant's packed bits.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": the variants share one
// resident W_base and each request's delta is applied on the fly, never
// writing W_eff to HBM.
//
// Arithmetic (exact distributive form, fp32 alpha): for token t of variant v,
//     y[t, j] = sum_k x[t,k] W_base[j,k]  +  alpha_v(j) * sum_k x[t,k] s^v_jk.
// Tokens arrive sorted by variant (compact, at most 64).  Per 128-row tile and
// 64-column K block:
//   * base: tcgen05.mma with A = the W_base tile as TMA left it in shared
//     memory (no rebuild at all) and B = every token, into D_base (TMEM);
//   * signs: for each variant with tokens, the rebuild warps expand its
//     packed bits to bf16 +-1 (two integer ops per pair) straight into a
//     tensor-memory A buffer (double-buffered), and tcgen05.mma multiplies it
//     with that variant's token rows (B starts at the 8-row group holding the
//     variant's first token) into the variant's own D_sign columns.
// The epilogue adds D_base + alpha_v * D_sign per (row, token), sums the K
// slices of a cluster through distributed shared memory in a fixed order and
// writes each token's row of y in the original order.
//
// Warps: 0 TMA producer (W and x tiles, 128-byte swizzle); 1 TMEM allocator and
// single-thread MMA issuer; 2..9 sign expansion (two threads per W row, 32
// columns each) and then the epilogue.  All waits are bounded.
#include <cooperative_groups.h>

#include "bd_device.cuh"
#include "bd_internal.h"

namespace cg = cooperative_groups;

namespace bd {
namespace {

constexpr int kBM = 128;          // W rows per CTA (MMA M)
constexpr int kBK = 64;           // K per stage
constexpr int kStages = 6;
constexpr int kMaxTok = 64;       // tokens per batch
constexpr int kXRows = 80;        // x tile rows: a variant's B rows may run 16 past the last token
constexpr int kMaxVar = 16;
constexpr int kExpWarps = 8;
constexpr int kThreads = (2 + kExpWarps) * 32;
constexpr uint32_t kWBytes = kBM * kBK * 2;       // 16 KB
constexpr uint32_t kXBytes = kXRows * kBK * 2;    // 10 KB
constexpr uint32_t kStageBytes = kWBytes + kXBytes;
constexpr uint32_t kColBase = 0;                  // D_base: columns 0..63
constexpr uint32_t kColSign = 64;                 // D_sign: columns 64..64+S-1 (S fixed per launch)
constexpr uint32_t kMaxSignCols = 384;            // so that at least two A buffers fit
constexpr int kMaxABuf = 8;                       // A buffers of 32 columns in the remaining columns
constexpr size_t kRedBytes = kMaxTok * kBM * 4;
constexpr size_t kSmem = 1024 + kStages * kStageBytes + kRedBytes + kMaxVar * kBM * 4 + 1024 + 256;

struct GtcArgs {
    const uint8_t *bits[kMaxVar];
    const float *alpha[kMaxVar];
    int32_t mode[kMaxVar];
    int32_t nv;
    const int32_t *seg;      // [nv + 1] segment starts of the sorted tokens
    const int32_t *perm;     // sorted row -> original token
    uint16_t *y;
    int64_t m, n_out, n_in, ks;
    int32_t cluster;
    unsigned *status;
    uint64_t wait_ns;
    int32_t test_stall;      // the MMA issuer's first wait is on a barrier nothing completes (tests)
};

struct VarTab {              // active variants in order
    int32_t n;
    int32_t v[kMaxVar];
    int32_t start8[kMaxVar]; // first B row: the 8-row group of the variant's first token
    int32_t ncols[kMaxVar];  // MMA N (multiple of 16)
    int32_t off[kMaxVar];    // first D_sign column
    int32_t seg0[kMaxVar], seg1[kMaxVar];
    int32_t tok_var[kMaxTok];      // sorted token -> index into the active list
    int32_t n_tok;
    int32_t col_a, nbuf;           // first A-buffer column, number of A buffers
};

__device__ __forceinline__ void give_up(volatile int *abort_flag, unsigned *status) {
    *abort_flag = 1;
    flag_status(status, kDevTimeout);
}

__device__ __forceinline__ void tmem_ld_32x32b_x1(uint32_t taddr, uint32_t &r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
}

__global__ void __launch_bounds__(kThreads, 1) gdec_tc_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                              const __grid_constant__ CUtensorMap tm_x,
                                                              const __grid_constant__ GtcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *red = reinterpret_cast<float *>(smem + kStages * kStageBytes);        // [token][row]
    float *alpha_s = red + kMaxTok * kBM;                                         // [variant][row]
    VarTab *tab = reinterpret_cast<VarTab *>(alpha_s + kMaxVar * kBM);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(tab) + 1024);
    uint64_t *full = bars, *empty = bars + kStages;
    uint64_t *a_full = bars + 2 * kStages, *a_empty = a_full + kMaxABuf;
    uint64_t *acc_full = a_empty + kMaxABuf;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint64_t *never = reinterpret_cast<uint64_t *>(tmem_slot + 2);  // completed by no one

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t row_tile = blockIdx.x / a.cluster;
    const int m0 = static_cast<int>(row_tile * kBM);
    const int64_t k_lo = static_cast<int64_t>(rank) * a.ks;
    const int64_t k_hi = min(k_lo + a.ks, a.n_in);
    const int nkb = k_hi > k_lo ? static_cast<int>((k_hi - k_lo + kBK - 1) / kBK) : 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kMaxABuf; ++b) {
            mbar_init(&a_full[b], kExpWarps / 2);  // one warp group fills a buffer
            mbar_init(&a_empty[b], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(never, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger_and_wait();

    // Active-variant table (from the device-side sort) and per-row alphas.
    if (threadIdx.x == 0) {
        int n = 0, off = 0;
        for (int v = 0; v < a.nv; ++v) {
            const int s0 = a.seg[v], s1 = a.seg[v + 1];
            if (s1 <= s0) continue;
            const int st8 = s0 & ~7;
            const int nc = (s1 - st8 + 15) & ~15;
            tab->v[n] = v;
            tab->start8[n] = st8;
            tab->ncols[n] = nc;
            tab->off[n] = off;
            tab->seg0[n] = s0;
            tab->seg1[n] = s1;
            for (int c = s0; c < s1 && c < kMaxTok; ++c) tab->tok_var[c] = n;
            off += nc;
            ++n;
        }
        for (int q = n; q < kMaxVar; ++q) tab->v[q] = 0;  // unused slots name a valid variant
        tab->col_a = kColSign + ((off + 31) & ~31);
        tab->nbuf = min(kMaxABuf, (512 - tab->col_a) / 32);
        tab->n = n;
        tab->n_tok = min(a.seg[a.nv], kMaxTok);
    }
    for (int i = threadIdx.x; i < a.nv * kBM; i += kThreads) {
        const int v = i / kBM, r = i - v * kBM;
        const int64_t row = static_cast<int64_t>(m0) + r;
        alpha_s[i] = row < a.n_out ? (a.mode[v] ? a.alpha[v][row] : a.alpha[v][0]) : 0.0f;
    }
    __syncthreads();
    const int nq = tab->n;
    const int n_mma_base = (min(static_cast<int>(a.m), kMaxTok) + 15) & ~15;

    if (warp == 0) {
        // ---- TMA producer ----
        if (lane == 0) {
            tma_prefetch_desc(&tm_w);
            tma_prefetch_desc(&tm_x);
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % kStages;
                if (!mbar_wait(&empty[s], ((kb / kStages) & 1) ^ 1, a.wait_ns, abort_flag)) {
                    give_up(abort_flag, a.status);
                    break;
                }
                const int kc = static_cast<int>(k_lo) + kb * kBK;
                uint8_t *st = smem + s * kStageBytes;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                tma_load_2d(st, &tm_w, &full[s], kc, m0);
                tma_load_2d(st + kWBytes, &tm_x, &full[s], kc, 0);
                issued = kb + 1;
            }
            if (*abort_flag) {
                for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
                    mbar_wait(&full[kb % kStages], (kb / kStages) & 1, kDrainLimitNs, nullptr);
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ----
        if (lane == 0) {
            const uint32_t idesc_base = idesc_bf16_f32(kBM, n_mma_base);
            const int nbuf = tab->nbuf;
            const uint32_t col_a = static_cast<uint32_t>(tab->col_a);
            bool ok = true;
            int j = 0;  // running sign-tile counter (A buffer j % nbuf)
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % kStages;
                if (!mbar_wait(a.test_stall && kb == 0 ? never : &full[s], (kb / kStages) & 1, a.wait_ns,
                               abort_flag)) {
                    give_up(abort_flag, a.status);
                    break;
                }
                tc_fence_after();
                const uint32_t w_addr = smem_u32(smem + s * kStageBytes);
                const uint32_t x_addr = smem_u32(smem + s * kStageBytes + kWBytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    tc_mma_f16_ss(tmem + kColBase, sw128_kmajor_desc(w_addr + kk * 32),
                                  sw128_kmajor_desc(x_addr + kk * 32), idesc_base, (kb | kk) != 0 ? 1u : 0u);
                for (int q = 0; q < nq; ++q, ++j) {
                    const int b = j % nbuf;
                    if (!mbar_wait(&a_full[b], (j / nbuf) & 1, a.wait_ns, abort_flag)) {
                        give_up(abort_flag, a.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t idesc = idesc_bf16_f32(kBM, tab->ncols[q]);
                    const uint32_t xq = x_addr + static_cast<uint32_t>(tab->start8[q]) * 128;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma_f16_ts(tmem + kColSign + tab->off[q], tmem + col_a + b * 32 + kk * 8,
                                      sw128_kmajor_desc(xq + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
                    tc_commit(&a_empty[b]);
                }
                tc_commit(&empty[s]);
            }
            tc_commit(acc_full);
            mbar_wait(acc_full, 0, kDrainLimitNs, nullptr);  // own MMAs done before TMEM may be freed
        }
    } else {
        // ---- sign expansion, then the epilogue ----
        // Two warp groups take alternate sign tiles; thread r of a group writes
        // the 64 columns of row r (32 TMEM columns) of its tiles.
        const int sub = warp & 3;                 // TMEM lane quarter
        const int wg = (warp - 2) >> 2;           // warp group
        const int h = wg;                         // epilogue: token half
        const int r = sub * 32 + lane;
        const int64_t row = static_cast<int64_t>(m0) + r;
        const bool row_ok = row < a.n_out;
        const int64_t bpr = a.n_in / 8;
        const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
        const int nbuf = tab->nbuf;
        const uint32_t col_a = static_cast<uint32_t>(tab->col_a);
        // The row's 8 packed bytes of K block kb for every active variant (prefetched a block ahead).
        auto load_words = [&](int kb, uint2 (&w)[kMaxVar]) {
            const int64_t byte0 = (k_lo + static_cast<int64_t>(kb) * kBK) / 8;
            const bool in = row_ok && kb < nkb && byte0 + 8 <= bpr;
#pragma unroll
            for (int q = 0; q < kMaxVar; ++q)
                w[q] = (in && q < nq) ? __ldg(reinterpret_cast<const uint2 *>(a.bits[tab->v[q]] + row * bpr + byte0))
                                      : make_uint2(0u, 0u);
        };
        uint2 cur[kMaxVar], nxt[kMaxVar];
        load_words(0, cur);
        bool ok = true;
        int j = 0;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            load_words(kb + 1, nxt);
#pragma unroll
            for (int q = 0; q < kMaxVar; ++q) {
                if (q >= nq) break;
                const int jj = j++;
                if ((jj & 1) != wg) continue;  // the other group's tile (warp-uniform)
                const int b = jj % nbuf;
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t byte = ((c < 4 ? cur[q].x : cur[q].y) >> (8 * (c & 3))) & 0xFFu;
                    v[4 * c + 0] = sign_pair_bf16<0>(byte);
                    v[4 * c + 1] = sign_pair_bf16<1>(byte);
                    v[4 * c + 2] = sign_pair_bf16<2>(byte);
                    v[4 * c + 3] = sign_pair_bf16<3>(byte);
                }
                const bool free_ok = mbar_wait(&a_empty[b], ((jj / nbuf) & 1) ^ 1, a.wait_ns, abort_flag);
                if (!__all_sync(0xFFFFFFFFu, free_ok)) {
                    if (lane == 0) give_up(abort_flag, a.status);
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st_32x32b_x32(tmem + lane_off + col_a + b * 32, v);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[b]);
            }
#pragma unroll
            for (int q = 0; q < kMaxVar; ++q) cur[q] = nxt[q];
        }
        // epilogue: partial y[token][row] of this K slice into red (each entry one thread)
        if (ok) {
            const bool got = mbar_wait(acc_full, 0, a.wait_ns, abort_flag);
            if (__all_sync(0xFFFFFFFFu, got)) {
                tc_fence_after();
                const int n_tok = tab->n_tok;
                for (int c = h * 32; c < h * 32 + 32; ++c) {
                    if (c >= n_tok) break;  // warp-uniform
                    const int qi = tab->tok_var[c];
                    uint32_t vb, vs;
                    tmem_ld_32x32b_x1(tmem + lane_off + kColBase + c, vb);
                    tmem_ld_32x32b_x1(tmem + lane_off + kColSign + tab->off[qi] + (c - tab->start8[qi]), vs);
                    tmem_ld_wait();
                    red[c * kBM + r] = __uint_as_float(vb) + alpha_s[tab->v[qi] * kBM + r] * __uint_as_float(vs);
                }
            } else if (lane == 0) {
                give_up(abort_flag, a.status);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
    cluster.sync();

    // rank c sums rows [c*share, (c+1)*share) over the cluster and writes original token rows
    const int share = (kBM + a.cluster - 1) / a.cluster;
    const int n_tok = tab->n_tok;
    if (!*abort_flag) {
        for (int i = threadIdx.x; i < share * n_tok; i += kThreads) {
            const int tok = i / share;
            const int lr = rank * share + (i - tok * share);
            const int64_t grow = static_cast<int64_t>(m0) + lr;
            if (lr < kBM && grow < a.n_out) {
                float s = 0.0f;
                for (int q = 0; q < a.cluster; ++q) s += cluster.map_shared_rank(red, q)[tok * kBM + lr];
                __nv_bfloat16 hv = __float2bfloat16_rn(s);
                const int64_t t = in_bounds(tok < a.m, a.status) ? a.perm[tok] : -1;
                if (in_bounds(t >= 0 && t < a.m, a.status))
                    a.y[t * a.n_out + grow] = *reinterpret_cast<uint16_t *>(&hv);
            }
        }
    }
    cluster.sync();
}

}  // namespace

bool grouped_decode_tc_supported(int64_t m, int32_t n_variants, int64_t n_in, const void *x_sorted,
                                 const void *w_base, const GroupedVariants &vars) {
    if (m < 1 || m > kMaxTok || n_variants > kMaxVar || n_in % kBK != 0) return false;
    // D_sign columns: sum over variants of round16(tokens + 7) <= m + 22 * (variants present)
    const int64_t present = m < n_variants ? m : n_variants;
    if (m + 22 * present > kMaxSignCols) return false;
    if ((reinterpret_cast<uintptr_t>(w_base) & 15) || (reinterpret_cast<uintptr_t>(x_sorted) & 15)) return false;
    for (int v = 0; v < vars.count; ++v)
        if (reinterpret_cast<uintptr_t>(vars.bits[v]) & 3) return false;
    return true;
}

cudaError_t launch_grouped_decode_tc(const void *x_sorted, int64_t m, const void *w_base, const GroupedVariants &vars,
                                     int64_t n_out, int64_t n_in, void *y, const int32_t *seg, const int32_t *perm,
                                     const DevCtx &ctx, cudaStream_t stream) {
    static bool attr_set[128] = {false};
    if (ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e =
            cudaFuncSetAttribute(gdec_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem));
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    CUtensorMap tm_w, tm_x;
    if (!encode_tensor_map_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_base, n_in, n_out, n_in * 2, kBK, kBM,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x_sorted, n_in, m, n_in * 2, kBK, kXRows,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GtcArgs a = {};
    for (int v = 0; v < vars.count; ++v) {
        a.bits[v] = vars.bits[v];
        a.alpha[v] = vars.alpha[v];
        a.mode[v] = vars.mode[v];
    }
    a.nv = vars.count;
    a.seg = seg;
    a.perm = perm;
    a.y = static_cast<uint16_t *>(y);
    a.m = m;
    a.n_out = n_out;
    a.n_in = n_in;
    a.status = ctx.status;
    a.wait_ns = ctx.wait_ns;
    a.test_stall = ctx.test_stall ? 1 : 0;
    const int64_t row_tiles = (n_out + kBM - 1) / kBM;
    const int64_t kblocks = n_in / kBK;
    int64_t c = row_tiles >= ctx.num_sms ? 1 : ctx.num_sms / row_tiles;  // fill the SMs without a second wave
    if (c < 1) c = 1;
    if (c > 8) c = 8;
    if (c > kblocks) c = kblocks;
    const int64_t per = (kblocks + c - 1) / c;
    a.ks = per * kBK;
    a.cluster = static_cast<int32_t>((kblocks + per - 1) / per);
    if (row_tiles * a.cluster > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(row_tiles * a.cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
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
    return cudaLaunchKernelEx(&cfg, gdec_tc_kernel, tm_w, tm_x, a);
}

}  // namespace bd
