// reconstruct.cu -- materialise the effective weight W_eff = W_base + alpha*s
// in bf16, once, for a standard matmul to consume.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog): section "Architecture de service" defines W_eff = W_base +
// alpha * unpacked signs (then a plain linear); section "Profil de latence"
// says decode runs as a standard matmul, which reads as rebuilding W_eff once
// per request and handing it to an ordinary GEMM.  The fused kernels never
// write W_eff; this pass exists to measure that reading against them.
//
// Rounding (the page prints no precision): the sum is formed in fp32 -- alpha
// times +-1 is exact, the add rounds once to nearest even -- and rounded once
// more, to nearest even, to bf16.
//
// Data path (HBM bound: read 2NK + NK/8, write 2NK bytes): thread t of a block
// owns 16-byte chunks (8 weights, one packed byte) base + t + 256u, four in
// flight at a time, so a warp's weight loads and stores are 512-byte
// contiguous and its bit loads 32-byte contiguous.  Each block walks one
// contiguous range of chunks; the row of a chunk (for per-row alpha) is found
// by one division when the block starts and then advanced incrementally.
#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ldg_nc(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_cs(uint4 *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Two bf16 weights (one 32-bit word) plus alpha with the signs of bits lo, hi.
__device__ __forceinline__ uint32_t rebuild_pair(uint32_t w, uint32_t byte, int i, float alpha) {
    const float w_lo = __uint_as_float(w << 16);
    const float w_hi = __uint_as_float(w & 0xFFFF0000u);
    // bit set -> +alpha, clear -> -alpha: flip alpha's sign bit when the bit is clear
    const float a_lo = __uint_as_float(__float_as_uint(alpha) ^ ((~byte >> (2 * i)) & 1u) << 31);
    const float a_hi = __uint_as_float(__float_as_uint(alpha) ^ ((~byte >> (2 * i + 1)) & 1u) << 31);
    const __nv_bfloat162 r = __floats2bfloat162_rn(__fadd_rn(w_lo, a_lo), __fadd_rn(w_hi, a_hi));
    return *reinterpret_cast<const uint32_t *>(&r);
}

__global__ void __launch_bounds__(kThreads) reconstruct_kernel(const uint4 *__restrict__ wb,
                                                              const uint8_t *__restrict__ bits,
                                                              const float *__restrict__ alpha, int32_t mode,
                                                              int64_t row_chunks, int64_t total, int64_t per_block,
                                                              uint4 *__restrict__ out) {
    pdl_trigger_and_wait();
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * per_block;
    const int64_t hi = min(lo + per_block, total);
    int64_t c = lo + threadIdx.x;
    if (c >= hi) return;
    int64_t row = c / row_chunks;
    int64_t row_end = (row + 1) * row_chunks;
    float a = mode ? alpha[row] : alpha[0];
    for (; c < hi; c += kThreads * kUnroll) {
        uint4 w[kUnroll];
        uint32_t b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t cu = c + u * kThreads;
            if (cu < hi) {
                w[u] = ldg_nc(wb + cu);
                b[u] = bits[cu];
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t cu = c + u * kThreads;
            if (cu < hi) {
                if (mode) {
                    while (cu >= row_end) {
                        ++row;
                        row_end += row_chunks;
                    }
                    a = alpha[row];
                }
                uint4 r;
                r.x = rebuild_pair(w[u].x, b[u], 0, a);
                r.y = rebuild_pair(w[u].y, b[u], 1, a);
                r.z = rebuild_pair(w[u].z, b[u], 2, a);
                r.w = rebuild_pair(w[u].w, b[u], 3, a);
                stg_cs(out + cu, r);
            }
        }
    }
}

}  // namespace

cudaError_t launch_reconstruct(const void *w_base, const uint8_t *bits, const float *alpha, int32_t alpha_mode,
                               int64_t n_out, int64_t n_in, void *w_eff, const DevCtx &ctx, cudaStream_t stream) {
    const int64_t row_chunks = n_in / 8;
    const int64_t total = n_out * row_chunks;
    if (total <= 0) return cudaSuccess;
    // about 8 blocks per SM; every block's range a whole number of unrolled passes
    const int64_t target = 8 * static_cast<int64_t>(ctx.num_sms);
    const int64_t pass = static_cast<int64_t>(kThreads) * kUnroll;
    int64_t per_block = (total + target - 1) / target;
    per_block = (per_block + pass - 1) / pass * pass;
    const int64_t blocks = (total + per_block - 1) / per_block;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reconstruct_kernel, static_cast<const uint4 *>(w_base), bits, alpha, alpha_mode,
                              row_chunks, total, per_block, static_cast<uint4 *>(w_eff));
}

}  // namespace bd
