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
// Data path (default, "direct"): one block per 1024-chunk segment loads its
// chunks of W_base and W_ft straight into registers.  Alternative ("ring"): a
// persistent pass (two CTAs per SM) streams W_base and W_ft through a
// shared-memory ring with 1-D bulk copies; every consumer thread
// owns 16-byte chunks (8 bf16) of both inputs, so one chunk yields exactly one
// output byte in registers with no cross-lane exchange, and lanes own
// consecutive chunks, so the byte stores are 32-byte coalesced.  |Delta| is
// summed pairwise in fp32 per thread (32 terms), reduced through the warp with
// xor-shuffles in double-float and across warps in fp64, in a fixed order: one
// fp64 partial per 1024-chunk segment.  A second kernel adds each row's
// partials in a fixed order and rounds alpha to fp32 once, so alpha is bitwise
// reproducible for a given shape on any device; a row that is a single
// segment (per-row alpha, n_in <= 8192) gets its alpha from pass 1 directly.
#include <cstdlib>

#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {
namespace {

struct CompressArgs {
    const uint4 *wb;   // W_base as 16-byte chunks, row-major
    const uint4 *wf;   // W_ft
    uint8_t *bits;     // one byte per chunk
    double *partials;  // [rows * segs]
    float *alpha;      // written here directly when a row is one segment (segs == 1)
    double count;      // elements per row: alpha = sum / count
    int64_t row_chunks;
    int64_t segs;
    int64_t rows;        // alpha entries (1 or n_out); bits hold rows * row_chunks bytes
    unsigned *status;    // bounds-checked build: where a failed index check is recorded
    int32_t test_stall;  // ring form: the first consumer wait is on a barrier nothing completes (tests)
};

// Signs and |Delta| of one chunk: returns the packed byte and the pairwise
// fp32 sum of the chunk's eight |Delta|.
__device__ __forceinline__ uint32_t chunk_signs(const uint4 &b, const uint4 &f, float &sum) {
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
    sum = ((ad[0] + ad[1]) + (ad[2] + ad[3])) + ((ad[4] + ad[5]) + (ad[6] + ad[7]));
    return byte;
}

// (hi, lo) += (bhi, blo) in double-float arithmetic: TwoSum (Knuth) gives the
// exact rounding error of hi + bhi, the low parts join it, and a FastTwoSum
// renormalises.  Plain fp32 adds only (no multiplies, so nothing contracts).
__device__ __forceinline__ void df_add(float &hi, float &lo, float bhi, float blo) {
    const float s = __fadd_rn(hi, bhi);
    const float bb = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(bhi, bb));
    const float e = __fadd_rn(__fadd_rn(err, lo), blo);
    hi = __fadd_rn(s, e);
    lo = __fsub_rn(e, __fsub_rn(hi, s));
}

// Pass 1, persistent: CTA b walks segments b, b+G, b+2G, ... (2 CTAs per SM).
// A producer warp streams each segment's W_base and W_ft bytes (1024 chunks,
// 16 KB per tensor: one ring slot) into a 3-slot shared-memory ring with 1-D
// bulk copies; 256 consumer threads take chunk tid + 256u (u = 0..3) of the
// segment.  A thread's four chunk sums (fp32, pairwise over 8 elements) are
// added pairwise in fp32 and reduced with xor-shuffles in double-float (fp32
// pairs), then across warps in fp64, in a fixed order.  The assignment and order do not depend on
// the grid, so each segment's partial (and alpha) is the same on any device.
// Worst-case relative error of a thread's fp32 sum: 5 levels of pairwise
// rounding plus the fp32 subtraction, ~6 * 2^-24 < 5e-7.  Segments of 1024
// chunks spread a matrix evenly over the persistent CTAs (a 4096 x 4096 scalar
// compression has 2048 segments: at most 7 per CTA against 6.7 on average).
constexpr int kRingStages = 3;
constexpr int kHalfChunks = 1024;                                          // chunks per ring slot
constexpr int kSlotsPerSeg = static_cast<int>(kCompressChunksPerSeg / kHalfChunks);
constexpr int kChunksPerSlotThread = kCompressChunksPerThread / kSlotsPerSeg;
static_assert(kSlotsPerSeg * kHalfChunks == kCompressChunksPerSeg, "a segment is whole ring slots");
static_assert(kChunksPerSlotThread * kCompressThreads == kHalfChunks, "a slot is whole chunks per thread");
constexpr uint32_t kHalfBytes = static_cast<uint32_t>(kHalfChunks) * 16;  // per tensor
constexpr int kPass1Threads = kCompressThreads + 32;
constexpr size_t kPass1Smem = 128 + kRingStages * 2 * kHalfBytes + 256;

__global__ void __launch_bounds__(kPass1Threads, 2)
    compress_pass1(const __grid_constant__ CompressArgs a, int64_t n_segs_total, unsigned *status,
                   uint64_t wait_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kRingStages * 2 * kHalfBytes);
    uint64_t *empty = full + kRingStages;
    double *warp_sum = reinterpret_cast<double *>(empty + kRingStages);  // [2][8]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(warp_sum + 16);
    uint64_t *never = reinterpret_cast<uint64_t *>(warp_sum + 17);  // completed by no one
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kRingStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCompressThreads / 32);
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    pdl_trigger_and_wait();

    const int64_t first_seg = blockIdx.x;
    const int64_t stride = gridDim.x;
    if (warp == kCompressThreads / 32) {
        if (lane == 0) {
            int j = 0, issued = 0;
            bool stop = false;
            for (int64_t sg = first_seg; sg < n_segs_total && !stop; sg += stride) {
                const int64_t row = sg / a.segs;
                const int64_t first = (sg - row * a.segs) * kCompressChunksPerSeg;
                const int64_t n = min(static_cast<int64_t>(kCompressChunksPerSeg), a.row_chunks - first);
                for (int h = 0; h * kHalfChunks < n; ++h, ++j) {
                    const int st = j % kRingStages;
                    if (!mbar_wait(&empty[st], ((j / kRingStages) & 1) ^ 1, wait_ns, abort_flag)) {
                        *abort_flag = 1;
                        flag_status(status, kDevTimeout);
                        stop = true;
                        break;
                    }
                    const int64_t c0 = first + h * kHalfChunks;
                    const int64_t nh = min(static_cast<int64_t>(kHalfChunks), n - h * kHalfChunks);
                    const uint32_t bytes = static_cast<uint32_t>(nh) * 16;
                    uint8_t *dst = smem + st * 2 * kHalfBytes;
                    mbar_arrive_expect_tx(&full[st], 2 * bytes);
                    bulk_load(dst, a.wb + row * a.row_chunks + c0, bytes, &full[st]);
                    bulk_load(dst + kHalfBytes, a.wf + row * a.row_chunks + c0, bytes, &full[st]);
                    issued = j + 1;
                }
            }
            if (*abort_flag) {
                for (int q = (issued > kRingStages ? issued - kRingStages : 0); q < issued; ++q)
                    mbar_wait(&full[q % kRingStages], (q / kRingStages) & 1, kDrainLimitNs, nullptr);
            }
        }
        return;  // the producer takes no part in the consumers' barriers
    }

    int j = 0, seg_i = 0;
    bool ok = true;
    for (int64_t sg = first_seg; sg < n_segs_total && ok; sg += stride, ++seg_i) {
        const int64_t row = sg / a.segs;
        const int64_t first = (sg - row * a.segs) * kCompressChunksPerSeg;
        const int64_t n = min(static_cast<int64_t>(kCompressChunksPerSeg), a.row_chunks - first);
        uint8_t *bits = a.bits + row * a.row_chunks + first;
        float cs[kCompressChunksPerThread];
#pragma unroll
        for (int u = 0; u < kCompressChunksPerThread; ++u) cs[u] = 0.0f;
        for (int h = 0; h * kHalfChunks < n; ++h, ++j) {
            const int st = j % kRingStages;
            const bool got = mbar_wait(a.test_stall && j == 0 ? never : &full[st], (j / kRingStages) & 1, wait_ns,
                                       abort_flag);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    flag_status(status, kDevTimeout);
                }
                ok = false;
                break;
            }
            const uint4 *sb = reinterpret_cast<const uint4 *>(smem + st * 2 * kHalfBytes);
            const uint4 *sf = reinterpret_cast<const uint4 *>(smem + st * 2 * kHalfBytes + kHalfBytes);
#pragma unroll
            for (int uu = 0; uu < kChunksPerSlotThread; ++uu) {
                const int cl = uu * kCompressThreads + tid;        // chunk within this slot
                const int c = h * kHalfChunks + cl;                // chunk within the segment
                if (c < n) {
                    float sum;
                    const uint32_t byte = chunk_signs(sb[cl], sf[cl], sum);
                    if (in_bounds(row < a.rows && first + c < a.row_chunks, a.status))
                        bits[c] = static_cast<uint8_t>(byte);
#pragma unroll
                    for (int hh = 0; hh < kSlotsPerSeg; ++hh)
                        if (h == hh) cs[hh * kChunksPerSlotThread + uu] = sum;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        // all consumer warps leave together on a timeout: the barrier below counts them all
        ok = __all_sync(0xFFFFFFFFu, ok);
        float t32;
        if constexpr (kCompressChunksPerThread == 8)
            t32 = ((cs[0] + cs[1]) + (cs[2] + cs[3])) + ((cs[4] + cs[5]) + (cs[6] + cs[7]));
        else
            t32 = (cs[0] + cs[1]) + (cs[2] + cs[3]);
        // Warp tree in double-float (an fp32 pair, ~44 significant bits): GB300
        // runs fp64 at a small fraction of the fp32 rate, so only the per-warp
        // results are widened.  Lane 0's operand order is fixed, so its result is
        // the same on every run.
        float hi = t32, lo = 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, off);
            const float olo = __shfl_xor_sync(0xFFFFFFFFu, lo, off);
            df_add(hi, lo, ohi, olo);
        }
        double *ws = warp_sum + (seg_i & 1) * 8;
        if (lane == 0) ws[warp] = static_cast<double>(hi) + static_cast<double>(lo);
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (!*abort_flag && tid == 0) {
            double s = 0.0;
#pragma unroll
            for (int w = 0; w < kCompressThreads / 32; ++w) s += ws[w];
            if (a.segs == 1) {
                if (in_bounds(row < a.rows, a.status))
                    a.alpha[row] = static_cast<float>(s / a.count);  // the row's only partial: no second pass
            } else if (in_bounds(sg < a.rows * a.segs, a.status)) {
                a.partials[sg] = s;
            }
        }
        if (*abort_flag) break;
    }
}

// Pass 1, direct form: one 256-thread block per segment.  Thread tid loads
// chunks tid + 256u (u = 0..3) of the segment from both inputs straight into
// registers (read-only, not kept in L1; eight blocks per SM keep ~256 KB of
// reads in flight), writes their bytes and adds the four chunk sums, the warp
// tree and the warps in exactly the order of the ring form above, so the
// partials and alpha are the same bits.
__device__ __forceinline__ void compress_segment(const CompressArgs &a, int64_t sg, double *warp_sum) {
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int64_t row = sg / a.segs;
    const int64_t first = (sg - row * a.segs) * kCompressChunksPerSeg;
    const int64_t n = min(static_cast<int64_t>(kCompressChunksPerSeg), a.row_chunks - first);
    const uint4 *wb = a.wb + row * a.row_chunks + first;
    const uint4 *wf = a.wf + row * a.row_chunks + first;
    uint8_t *bits = a.bits + row * a.row_chunks + first;
    uint4 b[kCompressChunksPerThread], f[kCompressChunksPerThread];
#pragma unroll
    for (int u = 0; u < kCompressChunksPerThread; ++u) {
        const int c = u * kCompressThreads + tid;
        if (c < n) {
            b[u] = ldg_stream(wb + c);
            f[u] = ldg_stream(wf + c);
        }
    }
    float cs[kCompressChunksPerThread];
#pragma unroll
    for (int u = 0; u < kCompressChunksPerThread; ++u) {
        const int c = u * kCompressThreads + tid;
        cs[u] = 0.0f;
        if (c < n) {
            float sum;
            const uint32_t byte = chunk_signs(b[u], f[u], sum);
            if (in_bounds(row < a.rows && first + c < a.row_chunks, a.status)) bits[c] = static_cast<uint8_t>(byte);
            cs[u] = sum;
        }
    }
    float hi, lo = 0.0f;
    if constexpr (kCompressChunksPerThread == 8)
        hi = ((cs[0] + cs[1]) + (cs[2] + cs[3])) + ((cs[4] + cs[5]) + (cs[6] + cs[7]));
    else
        hi = (cs[0] + cs[1]) + (cs[2] + cs[3]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, off);
        const float olo = __shfl_xor_sync(0xFFFFFFFFu, lo, off);
        df_add(hi, lo, ohi, olo);
    }
    if (lane == 0) warp_sum[warp] = static_cast<double>(hi) + static_cast<double>(lo);
    __syncthreads();
    if (tid == 0) {
        double s = 0.0;
#pragma unroll
        for (int w = 0; w < kCompressThreads / 32; ++w) s += warp_sum[w];
        if (a.segs == 1) {
            if (in_bounds(row < a.rows, a.status)) a.alpha[row] = static_cast<float>(s / a.count);
        } else if (in_bounds(sg < a.rows * a.segs, a.status)) {
            a.partials[sg] = s;
        }
    }
}

__global__ void __launch_bounds__(kCompressThreads) compress_direct(const __grid_constant__ CompressArgs a) {
    pdl_trigger_and_wait();
    __shared__ double warp_sum[kCompressThreads / 32];
    compress_segment(a, blockIdx.x, warp_sum);
}

// Several matrices in one launch: block b takes segment b - first_block[p] of
// matrix p (the largest p with first_block[p] <= b); the same per-segment
// arithmetic, so bits and alpha equal those of one launch per matrix.
struct CompressBatchArgs {
    CompressArgs m[kCompressBatchPerLaunch];
    int64_t first_block[kCompressBatchPerLaunch];
    int32_t n;
};

__global__ void __launch_bounds__(kCompressThreads)
    compress_direct_batch(const __grid_constant__ CompressBatchArgs a) {
    pdl_trigger_and_wait();
    __shared__ double warp_sum[kCompressThreads / 32];
    const int64_t b = blockIdx.x;
    int p = 0;
    while (p + 1 < a.n && a.first_block[p + 1] <= b) ++p;
    compress_segment(a.m[p], b - a.first_block[p], warp_sum);
}

// Pass 2 is launched as a programmatic dependent of pass 1: its CTAs become
// resident while pass 1 streams and wait (griddepcontrol.wait) until pass 1
// has completed and its partials are visible.

// One thread per row (few segments per row): alpha_j = sum(partials)/count.
__device__ __forceinline__ void pass2_row(const double *partials, int64_t r, int64_t segs, double count,
                                          float *alpha) {
    double s = 0.0;
    for (int64_t i = 0; i < segs; ++i) s += partials[r * segs + i];
    alpha[r] = static_cast<float>(s / count);
}

// One 256-thread block per row (many segments): strided per-thread sums, then a fixed tree.
__device__ __forceinline__ void pass2_block_row(const double *partials, int64_t r, int64_t segs, double count,
                                                float *alpha, double *red) {
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < segs; i += 256) s += partials[r * segs + i];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) alpha[r] = static_cast<float>(red[0] / count);
}

__global__ void compress_pass2_rows(const double *partials, int64_t rows, int64_t segs, double count,
                                    float *alpha) {
    pdl_trigger_and_wait();
    const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r < rows) pass2_row(partials, r, segs, count, alpha);
}

__global__ void __launch_bounds__(256) compress_pass2_block(const double *partials, int64_t segs, double count,
                                                            float *alpha) {
    pdl_trigger_and_wait();
    __shared__ double red[256];
    pass2_block_row(partials, blockIdx.x, segs, count, alpha, red);
}

// Pass 2 of several matrices in one launch (256 threads): matrix p owns blocks
// [first_block[p], first_block[p+1]); with at most kPass2RowsMaxSegs segments per
// row each thread of its blocks sums one row, otherwise each block sums one row.
// The per-row orders are those of the two kernels above.
constexpr int64_t kPass2RowsMaxSegs = 32;
struct Pass2BatchArgs {
    const double *partials[kCompressBatchPerLaunch];
    float *alpha[kCompressBatchPerLaunch];
    int64_t rows[kCompressBatchPerLaunch];
    int64_t segs[kCompressBatchPerLaunch];
    double count[kCompressBatchPerLaunch];
    int64_t first_block[kCompressBatchPerLaunch];
    int32_t n;
};

__global__ void __launch_bounds__(256) compress_pass2_batch(const __grid_constant__ Pass2BatchArgs a) {
    pdl_trigger_and_wait();
    __shared__ double red[256];
    const int64_t b = blockIdx.x;
    int p = 0;
    while (p + 1 < a.n && a.first_block[p + 1] <= b) ++p;
    const int64_t lb = b - a.first_block[p];
    if (a.segs[p] <= kPass2RowsMaxSegs) {
        const int64_t r = lb * 256 + threadIdx.x;
        if (r < a.rows[p]) pass2_row(a.partials[p], r, a.segs[p], a.count[p], a.alpha[p]);
    } else {
        pass2_block_row(a.partials[p], lb, a.segs[p], a.count[p], a.alpha[p], red);
    }
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
    const CompressGeom g = compress_geometry(n_out, n_in, alpha_mode);
    CompressArgs a;
    a.wb = static_cast<const uint4 *>(w_base);
    a.wf = static_cast<const uint4 *>(w_ft);
    a.bits = bits;
    a.partials = partials;
    a.alpha = alpha;
    a.count = static_cast<double>(g.row_chunks) * 8.0;
    a.row_chunks = g.row_chunks;
    a.segs = g.segs;
    a.rows = g.rows;
    a.status = ctx.status;
    a.test_stall = ctx.test_stall ? 1 : 0;
    const int64_t n_segs = g.rows * g.segs;
    static bool attr_set[128] = {false};
    if (ctx.device >= 0 && ctx.device < 128 && !attr_set[ctx.device]) {
        cudaError_t e = cudaFuncSetAttribute(compress_pass1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kPass1Smem));
        if (e != cudaSuccess) return e;
        attr_set[ctx.device] = true;
    }
    // The direct form (one block per segment) unless the BD_OPT_COMPRESS_FORM
    // option selects the persistent ring form.  Measured on GB300 (graph-replayed): the direct
    // form is 4% faster on the Llama-7B layer step and up to 15% on per-row
    // compressions, the ring form 2-3% faster on scalar compressions of
    // 8192 x 8192 and 11008 x 4096; both give the same bits and alpha.
    const bool ring = option_value(BD_OPT_COMPRESS_FORM) == 1;
    const int64_t grid = ring ? (n_segs < 2 * ctx.num_sms ? n_segs : 2 * ctx.num_sms) : n_segs;
    if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid > 0 ? grid : 1), 1, 1);
    cfg.blockDim = dim3(ring ? kPass1Threads : kCompressThreads, 1, 1);
    cfg.dynamicSmemBytes = ring ? kPass1Smem : 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = ring ? cudaLaunchKernelEx(&cfg, compress_pass1, a, n_segs, ctx.status, ctx.wait_ns)
                         : cudaLaunchKernelEx(&cfg, compress_direct, a);
    if (e != cudaSuccess || g.segs == 1) return e;  // one segment per row: pass 1 wrote alpha
    const double count = a.count;
    cudaLaunchConfig_t c2 = {};
    c2.stream = stream;
    c2.attrs = attr;
    c2.numAttrs = 1;
    if (g.segs <= kPass2RowsMaxSegs) {
        c2.gridDim = dim3(static_cast<unsigned>((g.rows + 127) / 128), 1, 1);
        c2.blockDim = dim3(128, 1, 1);
        return cudaLaunchKernelEx(&c2, compress_pass2_rows, static_cast<const double *>(partials), g.rows, g.segs,
                                  count, alpha);
    }
    c2.gridDim = dim3(static_cast<unsigned>(g.rows), 1, 1);
    c2.blockDim = dim3(256, 1, 1);
    return cudaLaunchKernelEx(&c2, compress_pass2_block, static_cast<const double *>(partials), g.segs, count, alpha);
}

}  // namespace bd

namespace bd {

cudaError_t launch_compress_batch(const CompressItem *items, int n, const DevCtx &ctx, cudaStream_t stream) {
    if (n < 1 || n > kCompressBatchPerLaunch) return cudaErrorInvalidValue;
    CompressBatchArgs a1{};
    Pass2BatchArgs a2{};
    int64_t blocks1 = 0, blocks2 = 0;
    int n2 = 0;
    for (int i = 0; i < n; ++i) {
        const CompressItem &it = items[i];
        const CompressGeom g = compress_geometry(it.n_out, it.n_in, it.alpha_mode);
        CompressArgs &a = a1.m[i];
        a.wb = static_cast<const uint4 *>(it.w_base);
        a.wf = static_cast<const uint4 *>(it.w_ft);
        a.bits = it.bits;
        a.partials = it.partials;
        a.alpha = it.alpha;
        a.count = static_cast<double>(g.row_chunks) * 8.0;
        a.row_chunks = g.row_chunks;
        a.segs = g.segs;
        a.rows = g.rows;
        a.status = ctx.status;
        a.test_stall = 0;  // the direct form has no pipeline waits
        a1.first_block[i] = blocks1;
        blocks1 += g.rows * g.segs;
        if (g.segs > 1) {  // pass 2 only for rows split into several segments
            a2.partials[n2] = it.partials;
            a2.alpha[n2] = it.alpha;
            a2.rows[n2] = g.rows;
            a2.segs[n2] = g.segs;
            a2.count[n2] = a.count;
            a2.first_block[n2] = blocks2;
            blocks2 += g.segs <= kPass2RowsMaxSegs ? (g.rows + 255) / 256 : g.rows;
            ++n2;
        }
    }
    a1.n = n;
    a2.n = n2;
    if (blocks1 > 0x7FFFFFFFLL || blocks2 > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks1), 1, 1);
    cfg.blockDim = dim3(kCompressThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, compress_direct_batch, a1);
    if (e != cudaSuccess || n2 == 0) return e;
    cudaLaunchConfig_t c2 = cfg;
    c2.gridDim = dim3(static_cast<unsigned>(blocks2), 1, 1);
    c2.blockDim = dim3(256, 1, 1);
    return cudaLaunchKernelEx(&c2, compress_pass2_batch, a2);
}

}  // namespace bd
