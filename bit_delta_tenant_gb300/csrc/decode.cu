// decode.cu -- fused BitDelta linear for small token counts (m <= 64): an
// HBM-streaming kernel that reads each W_base element and its packed sign bit
// exactly once, unpacks the bits in registers and never forms W_eff in memory.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Architecture de service": a fused kernel reads the
// base weights and the delta bits together and rebuilds the effective weight
// in registers, without materialising W_eff in HBM (conceptual
// fused_bitdelta_linear listing: y = linear(x, W_base + alpha * unpack)).
//
// The product is taken in its distributive form
//     y[t, j] = sum_k x[t,k] W_base[j,k]  +  alpha_(j) * sum_k x[t,k] s_jk,
// which is the listing's linear(x, W_base + alpha*s) up to fp32 rounding
// order: W_base feeds the tensor core as stored (bf16), the signs feed it as
// exact bf16 +-1 (two integer ops per pair of signs), and alpha is applied
// once per output in fp32.  This keeps the per-element ALU cost at ~1 op so
// the kernel stays on the HBM roofline.
//
// Tiling: a warp owns 16 W rows (the M side of mma.m16n8k16) and walks its
// CTA's K slice 128 columns at a time; each lane loads one 16-byte vector
// (8 consecutive k) per row and per 32-column step, and the 16-element K of
// each MMA is a permutation of actual columns (k-slot 2t,2t+1,2t+8,2t+9 of
// lane quad t <-> columns 8t..8t+3 of the step), applied identically to the
// activations, so every register is used as loaded.  Tokens are the N side
// (tiles of 8).  A CTA owns 128 rows; the clusterable K split over C CTAs
// keeps each CTA's activation slice in shared memory, and the C partial tiles
// are summed in a fixed order through distributed shared memory.
#include <cooperative_groups.h>

#include "bd_device.cuh"
#include "bd_internal.h"

namespace cg = cooperative_groups;

namespace bd {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = kWarps * 16;  // 128
constexpr int kStep = 128;                // K columns per warp iteration
constexpr int kSmemBudget = 200 * 1024;

struct DecodeArgs {
    const uint8_t *x;  // bf16 [m, n_in]
    const uint8_t *w;  // bf16 [n_out, n_in]
    const uint8_t *bits;
    const float *alpha;
    uint16_t *y;
    int64_t m, n_out, n_in;
    int64_t ks;        // K slice per cluster rank (multiple of kStep)
    int32_t mode;
    int32_t cluster;   // CTAs per cluster along K
    int32_t x_stride;  // bytes per token row of the staged slice
    int32_t bits16;    // packed rows are 16-byte aligned in kStep units
    unsigned *status;  // bounds-checked build: where a failed index check is recorded
};

__device__ __forceinline__ uint32_t byte_of(uint32_t word, int t) { return (word >> (8 * t)) & 0xFFu; }

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int MP = 8 * NT;  // padded token count
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t row_block = blockIdx.x / a.cluster;
    const int64_t k_lo = static_cast<int64_t>(rank) * a.ks;
    const int64_t k_hi = min(k_lo + a.ks, a.n_in);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;
    const int t = lane & 3;

    // 1. Stage x[:, k_lo:k_lo+ks] (zero-padded) in shared memory.
    const int vec_per_row = static_cast<int>(a.ks / 8);
    for (int i = tid; i < MP * vec_per_row; i += kThreads) {
        const int r = i / vec_per_row;
        const int c = i - r * vec_per_row;
        const int64_t k = k_lo + static_cast<int64_t>(c) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < a.m && k < k_hi) v = ldg_keep(a.x + (static_cast<int64_t>(r) * a.n_in + k) * 2);
        *reinterpret_cast<uint4 *>(smem + r * a.x_stride + c * 16) = v;
    }
    __syncthreads();

    // 2. Stream this warp's 16 rows over the slice.
    const int64_t r0 = row_block * kRowsPerCta + warp * 16 + g;
    const int64_t r1 = r0 + 8;
    const bool v0 = r0 < a.n_out;
    const bool v1 = r1 < a.n_out;
    const uint8_t *w0 = a.w + (v0 ? r0 : 0) * a.n_in * 2;
    const uint8_t *w1 = a.w + (v1 ? r1 : 0) * a.n_in * 2;
    const int64_t bpr = a.n_in / 8;
    const uint8_t *q0 = a.bits + (v0 ? r0 : 0) * bpr;
    const uint8_t *q1 = a.bits + (v1 ? r1 : 0) * bpr;

    float accb[NT][4], accs[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) accb[i][j] = accs[i][j] = 0.0f;

    auto load_step = [&](int64_t kc, uint4 (&wa)[4], uint4 (&wb)[4], uint32_t (&ba)[4], uint32_t (&bb)[4]) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t k0 = kc + 32 * u + 8 * t;
            const bool in = k0 < k_hi;
            wa[u] = (v0 && in) ? ldg_stream(w0 + k0 * 2) : make_uint4(0, 0, 0, 0);
            wb[u] = (v1 && in) ? ldg_stream(w1 + k0 * 2) : make_uint4(0, 0, 0, 0);
        }
        if (a.bits16 && kc + kStep <= k_hi) {
            // the quad shares one 16-byte load (same address -> one request)
            const uint4 p0 = v0 ? ldg_keep(q0 + kc / 8) : make_uint4(0, 0, 0, 0);
            const uint4 p1 = v1 ? ldg_keep(q1 + kc / 8) : make_uint4(0, 0, 0, 0);
            ba[0] = byte_of(p0.x, t), ba[1] = byte_of(p0.y, t), ba[2] = byte_of(p0.z, t), ba[3] = byte_of(p0.w, t);
            bb[0] = byte_of(p1.x, t), bb[1] = byte_of(p1.y, t), bb[2] = byte_of(p1.z, t), bb[3] = byte_of(p1.w, t);
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t k0 = kc + 32 * u + 8 * t;
                const bool in = k0 < k_hi;
                ba[u] = (v0 && in) ? static_cast<uint32_t>(__ldg(q0 + k0 / 8)) : 0u;
                bb[u] = (v1 && in) ? static_cast<uint32_t>(__ldg(q1 + k0 / 8)) : 0u;
            }
        }
    };

    uint4 wa[4], wb[4];
    uint32_t ba[4], bb[4];
    if (k_lo < k_hi) load_step(k_lo, wa, wb, ba, bb);
    for (int64_t kc = k_lo; kc < k_hi; kc += kStep) {
        uint4 nwa[4], nwb[4];
        uint32_t nba[4], nbb[4];
        const bool more = kc + kStep < k_hi;
        if (more) load_step(kc + kStep, nwa, nwb, nba, nbb);
        const uint8_t *xs = smem + (kc - k_lo) * 2 + (8 * t) * 2;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t sa0 = sign_pair_bf16<0>(ba[u]), sa1 = sign_pair_bf16<1>(ba[u]);
            const uint32_t sa2 = sign_pair_bf16<2>(ba[u]), sa3 = sign_pair_bf16<3>(ba[u]);
            const uint32_t sb0 = sign_pair_bf16<0>(bb[u]), sb1 = sign_pair_bf16<1>(bb[u]);
            const uint32_t sb2 = sign_pair_bf16<2>(bb[u]), sb3 = sign_pair_bf16<3>(bb[u]);
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xs + (8 * tt + g) * a.x_stride + 64 * u);
                mma_bf16_16816(accb[tt], wa[u].x, wb[u].x, wa[u].y, wb[u].y, xv.x, xv.y);
                mma_bf16_16816(accb[tt], wa[u].z, wb[u].z, wa[u].w, wb[u].w, xv.z, xv.w);
                mma_bf16_16816(accs[tt], sa0, sb0, sa1, sb1, xv.x, xv.y);
                mma_bf16_16816(accs[tt], sa2, sb2, sa3, sb3, xv.z, xv.w);
            }
        }
        if (more) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                wa[u] = nwa[u], wb[u] = nwb[u], ba[u] = nba[u], bb[u] = nbb[u];
            }
        }
    }

    // 3. y partial = base + alpha * signs, staged as red[token][row in CTA] (fp32).
    const float al0 = v0 ? (a.mode ? a.alpha[r0] : a.alpha[0]) : 0.0f;
    const float al1 = v1 ? (a.mode ? a.alpha[r1] : a.alpha[0]) : 0.0f;
    __syncthreads();  // every warp is done with the staged activations
    float *red = reinterpret_cast<float *>(smem);
    const int lr0 = warp * 16 + g;
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
        const int c = 8 * tt + 2 * t;
        red[c * kRowsPerCta + lr0] = accb[tt][0] + al0 * accs[tt][0];
        red[(c + 1) * kRowsPerCta + lr0] = accb[tt][1] + al0 * accs[tt][1];
        red[c * kRowsPerCta + lr0 + 8] = accb[tt][2] + al1 * accs[tt][2];
        red[(c + 1) * kRowsPerCta + lr0 + 8] = accb[tt][3] + al1 * accs[tt][3];
    }
    cluster.sync();

    // 4. Rank c sums rows [c*share, (c+1)*share) over the cluster, ranks in order.
    const int share = (kRowsPerCta + a.cluster - 1) / a.cluster;
    const int m_here = static_cast<int>(a.m < MP ? a.m : MP);
    for (int i = tid; i < share * m_here; i += kThreads) {
        const int tok = i / share;
        const int lr = rank * share + (i - tok * share);
        const int64_t row = row_block * kRowsPerCta + lr;
        if (lr < kRowsPerCta && row < a.n_out && in_bounds(tok < a.m, a.status)) {
            float s = 0.0f;
            for (int q = 0; q < a.cluster; ++q) {
                const float *rr = cluster.map_shared_rank(red, q);
                s += rr[tok * kRowsPerCta + lr];
            }
            __nv_bfloat16 h = __float2bfloat16_rn(s);
            a.y[static_cast<int64_t>(tok) * a.n_out + row] = *reinterpret_cast<uint16_t *>(&h);
        }
    }
    cluster.sync();  // keep this CTA's partials alive until every rank has read them
}

struct Plan {
    int nt;
    int cluster;
    int64_t ks;
    int x_stride;
    size_t smem;
    int64_t row_blocks;
};

bool make_plan(int64_t m, int64_t n_out, int64_t n_in, int num_sms, Plan &p) {
    if (m < 1 || m > kDecodeMaxM) return false;
    p.nt = m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8;
    const int mp = 8 * p.nt;
    p.row_blocks = (n_out + kRowsPerCta - 1) / kRowsPerCta;
    int c = static_cast<int>((2 * static_cast<int64_t>(num_sms) + p.row_blocks - 1) / p.row_blocks);
    if (c < 1) c = 1;
    if (c > 8) c = 8;
    for (;; ++c) {
        if (c > 8) return false;
        int64_t ks = (n_in + c - 1) / c;
        ks = (ks + kStep - 1) / kStep * kStep;
        const int x_stride = static_cast<int>(ks * 2 + 64);
        const size_t xs = static_cast<size_t>(mp) * x_stride;
        const size_t rs = static_cast<size_t>(kRowsPerCta) * mp * 4;
        const size_t smem = xs > rs ? xs : rs;
        if (smem <= static_cast<size_t>(kSmemBudget)) {
            p.cluster = static_cast<int>((n_in + ks - 1) / ks);  // drop empty ranks
            if (p.cluster < 1) p.cluster = 1;
            p.ks = ks;
            p.x_stride = x_stride;
            p.smem = smem;
            return true;
        }
    }
}

template <int NT>
cudaError_t launch_nt(const DecodeArgs &a, const Plan &p, const DevCtx &ctx, cudaStream_t stream) {
    static bool attr_set[128] = {false};
    if (ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBudget);
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.row_blocks * p.cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<NT>, a);
}

}  // namespace

bool decode_supported(int64_t m, int64_t n_out, int64_t n_in, int num_sms) {
    Plan p;
    return make_plan(m, n_out, n_in, num_sms, p);
}

cudaError_t launch_decode(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                          int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                          cudaStream_t stream) {
    Plan p;
    if (!make_plan(m, n_out, n_in, ctx.num_sms, p)) return cudaErrorNotSupported;
    if (p.row_blocks * p.cluster > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    DecodeArgs a;
    a.x = static_cast<const uint8_t *>(x);
    a.w = static_cast<const uint8_t *>(w_base);
    a.bits = bits;
    a.alpha = alpha;
    a.y = static_cast<uint16_t *>(y);
    a.m = m;
    a.n_out = n_out;
    a.n_in = n_in;
    a.ks = p.ks;
    a.mode = alpha_mode;
    a.cluster = p.cluster;
    a.x_stride = p.x_stride;
    a.bits16 = ((n_in % 128 == 0) && ((reinterpret_cast<uintptr_t>(bits) & 15) == 0)) ? 1 : 0;
    a.status = ctx.status;
    switch (p.nt) {
        case 1: return launch_nt<1>(a, p, ctx, stream);
        case 2: return launch_nt<2>(a, p, ctx, stream);
        case 4: return launch_nt<4>(a, p, ctx, stream);
        default: return launch_nt<8>(a, p, ctx, stream);
    }
}

}  // namespace bd
