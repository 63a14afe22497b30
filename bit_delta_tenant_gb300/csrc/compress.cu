// compress.cu -- BitDelta compression on the GPU: one HBM pass over W_base
// and W_ft that writes the packed sign bits and the |Delta| partial sums, then
// a small fixed-order pass that turns the partials into alpha.
//
// Method: "BitDelta : servir 14 modèles Zen depuis un seul cluster GPU"
// (Hanzo blog), section "Le fondement mathématique": Delta = W_ft - W_base,
// W_ft ~ W_base + alpha*sign(Delta), alpha = (1/n)*||Delta||_1; section
// "Détails d'infrastructure": signs stored 8 per byte, alpha stored in fp32,
// one per output dimension (per-row mode) -- the page's per-matrix form is the
// scalar mode.
//
// Layout and readings: byte c of row j holds elements 8c..8c+7 of that row,
// least significant bit first; bit = 1 iff Delta >= 0 (zero of either sign
// packs as 1).  Delta is formed in fp32 from the bf16 inputs.
//
// Data path: every thread owns 16-byte chunks (8 bf16) of both inputs, so one
// chunk yields exactly one output byte in registers, with no cross-lane
// exchange; lanes of a warp own consecutive chunks, so the loads are 512-byte
// coalesced and the byte stores 32-byte coalesced.  |Delta| of a chunk is
// summed pairwise in fp32 (8 terms), widened to fp64, reduced through the warp
// with xor-shuffles and across warps in shared memory in a fixed order; each
// block writes one fp64 partial.  A second kernel adds each row's partials in
// a fixed order and rounds alpha to fp32 once, so alpha is bitwise
// reproducible for a given shape on any device.
#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {
namespace {

struct CompressArgs {
    const uint4 *wb;   // W_base as 16-byte chunks, row-major
    const uint4 *wf;   // W_ft
    uint8_t *bits;     // one byte per chunk
    double *partials;  // [rows * segs]
    int64_t row_chunks;
    int64_t segs;
};

// Signs and |Delta| of one chunk: returns the packed byte, adds sum|Delta| to acc.
__device__ __forceinline__ uint32_t chunk_signs(const uint4 &b, const uint4 &f, double &acc) {
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
    const uint32_t fw[4] = {f.x, f.y, f.z, f.w};
    float ad[8];
    uint32_t byte = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float d_lo = bf16lo_to_f32(fw[i]) - bf16lo_to_f32(bw[i]);
        const float d_hi = bf16hi_to_f32(fw[i]) - bf16hi_to_f32(bw[i]);
        byte |= (d_lo >= 0.0f ? 1u : 0u) << (2 * i);
        byte |= (d_hi >= 0.0f ? 1u : 0u) << (2 * i + 1);
        ad[2 * i] = fabsf(d_lo);
        ad[2 * i + 1] = fabsf(d_hi);
    }
    const float s = ((ad[0] + ad[1]) + (ad[2] + ad[3])) + ((ad[4] + ad[5]) + (ad[6] + ad[7]));
    acc += static_cast<double>(s);
    return byte;
}

__global__ void __launch_bounds__(kCompressThreads) compress_pass1(CompressArgs a) {
    const int64_t seg_id = blockIdx.x;
    const int64_t row = seg_id / a.segs;
    const int64_t seg = seg_id - row * a.segs;
    const int64_t first = seg * kCompressChunksPerSeg;
    const int64_t base = row * a.row_chunks;
    const int tid = threadIdx.x;

    uint4 vb[kCompressChunksPerThread], vf[kCompressChunksPerThread];
#pragma unroll
    for (int u = 0; u < kCompressChunksPerThread; ++u) {
        const int64_t c = first + u * kCompressThreads + tid;
        if (c < a.row_chunks) {
            vb[u] = ldg_stream(a.wb + base + c);
            vf[u] = ldg_stream(a.wf + base + c);
        } else {
            vb[u] = make_uint4(0, 0, 0, 0);
            vf[u] = make_uint4(0, 0, 0, 0);
        }
    }
    double acc = 0.0;
#pragma unroll
    for (int u = 0; u < kCompressChunksPerThread; ++u) {
        const int64_t c = first + u * kCompressThreads + tid;
        if (c < a.row_chunks) {
            const uint32_t byte = chunk_signs(vb[u], vf[u], acc);
            a.bits[base + c] = static_cast<uint8_t>(byte);
        }
    }
    // Fixed-order fp64 reduction: xor-butterfly in the warp, then warps in order.
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    __shared__ double warp_sum[kCompressThreads / 32];
    if ((tid & 31) == 0) warp_sum[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
        double s = 0.0;
#pragma unroll
        for (int w = 0; w < kCompressThreads / 32; ++w) s += warp_sum[w];
        a.partials[seg_id] = s;
    }
}

// One thread per row (few segments per row): alpha_j = sum(partials)/count.
__global__ void compress_pass2_rows(const double *partials, int64_t rows, int64_t segs, double count,
                                    float *alpha) {
    const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    double s = 0.0;
    for (int64_t i = 0; i < segs; ++i) s += partials[r * segs + i];
    alpha[r] = static_cast<float>(s / count);
}

// One block per row (many segments): strided per-thread sums, then a fixed tree.
__global__ void __launch_bounds__(256) compress_pass2_block(const double *partials, int64_t segs, double count,
                                                            float *alpha) {
    const int64_t r = blockIdx.x;
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < segs; i += 256) s += partials[r * segs + i];
    __shared__ double red[256];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) alpha[r] = static_cast<float>(red[0] / count);
}

}  // namespace

CompressGeom compress_geometry(int64_t n_out, int64_t n_in, int32_t alpha_mode) {
    CompressGeom g;
    if (alpha_mode == 1) {
        g.rows = n_out;
        g.row_chunks = n_in / 8;
    } else {
        g.rows = 1;
        g.row_chunks = n_out * (n_in / 8);
    }
    g.segs = (g.row_chunks + kCompressChunksPerSeg - 1) / kCompressChunksPerSeg;
    if (g.segs < 1) g.segs = 1;
    return g;
}

cudaError_t launch_compress(const void *w_base, const void *w_ft, int64_t n_out, int64_t n_in, int32_t alpha_mode,
                            uint8_t *bits, float *alpha, double *partials, const DevCtx &ctx, cudaStream_t stream) {
    (void)ctx;
    const CompressGeom g = compress_geometry(n_out, n_in, alpha_mode);
    CompressArgs a;
    a.wb = static_cast<const uint4 *>(w_base);
    a.wf = static_cast<const uint4 *>(w_ft);
    a.bits = bits;
    a.partials = partials;
    a.row_chunks = g.row_chunks;
    a.segs = g.segs;
    const int64_t blocks = g.rows * g.segs;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    compress_pass1<<<static_cast<unsigned>(blocks), kCompressThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const double count = static_cast<double>(g.row_chunks) * 8.0;
    if (g.segs <= 32) {
        const int64_t nb = (g.rows + 127) / 128;
        compress_pass2_rows<<<static_cast<unsigned>(nb), 128, 0, stream>>>(partials, g.rows, g.segs, count, alpha);
    } else {
        compress_pass2_block<<<static_cast<unsigned>(g.rows), 256, 0, stream>>>(partials, g.segs, count, alpha);
    }
    return cudaGetLastError();
}

}  // namespace bd
