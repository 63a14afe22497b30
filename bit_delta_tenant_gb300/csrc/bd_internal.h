// bd_internal.h -- host-side interfaces between the C-ABI layer (api.cu) and
// the kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "bitdelta.h"

namespace bd {

// Bits of the sticky device status word (set with atomicOr by kernels, read
// and cleared by the host).
constexpr unsigned kDevTimeout = 1u;
constexpr unsigned kDevBadVariant = 2u;
constexpr unsigned kDevBounds = 4u;  // bounds-checked build: an index failed its check (access skipped)

// Per-launch context every kernel receives: where to record device-side
// errors, and the wall-clock limit of bounded waits.
struct DevCtx {
    unsigned *status;     // device address of the sticky status word
    uint64_t wait_ns;     // limit of every bounded wait
    int num_sms;          // SM count of the current device
    int device;           // current device ordinal
    bool weight_prefetch; // weights may be read before the preceding kernel on the stream completes
    bool test_stall;      // BD_OPT_TEST_STALL: a first pipeline wait on a barrier nothing completes
};

// Current value of a bd_set_option knob (BD_OPT_*; 0 = automatic).
int64_t option_value(int32_t option);

// Device context of the current device (status word address, SM count, the
// process-wide wait limit); returns a bd_status code.
int32_t make_dev_ctx(DevCtx *ctx);

// ---- compression -------------------------------------------------------------------
constexpr int kCompressThreads = 256;
constexpr int kCompressChunksPerThread = 4;                                        // 16-byte chunks
constexpr int64_t kCompressChunksPerSeg = kCompressThreads * kCompressChunksPerThread;  // 1024 chunks

// Geometry of the deterministic two-level reduction: `rows` independent sums
// (1 for a scalar alpha, n_out per-row), each over `row_chunks` chunks of 8
// elements split into `segs` fixed segments.
struct CompressGeom {
    int64_t rows, row_chunks, segs;
};
CompressGeom compress_geometry(int64_t n_out, int64_t n_in, int32_t alpha_mode);

cudaError_t launch_compress(const void *w_base, const void *w_ft, int64_t n_out, int64_t n_in, int32_t alpha_mode,
                            uint8_t *bits, float *alpha, double *partials, const DevCtx &ctx, cudaStream_t stream);

// Several compressions in one launch of pass 1 (and one of pass 2): at most
// kCompressBatchPerLaunch matrices, each with its own partials region (the
// sizes bd_compress_workspace_size gives); same bits and alpha as one
// launch_compress per matrix.
constexpr int kCompressBatchPerLaunch = 8;
struct CompressItem {
    const void *w_base;
    const void *w_ft;
    int64_t n_out, n_in;
    int32_t alpha_mode;
    uint8_t *bits;
    float *alpha;
    double *partials;
};
cudaError_t launch_compress_batch(const CompressItem *items, int n, const DevCtx &ctx, cudaStream_t stream);

// ---- fused linear ---------------------------------------------------------------------
// HBM-streaming small-m kernel (m <= kDecodeMaxM).  Returns cudaErrorNotSupported
// if the activation slice does not fit in shared memory (caller falls back).
constexpr int kDecodeMaxM = 64;
// Automatic choice: the streaming kernels up to this many tokens, the tensor-core
// kernel (with a K split when its tiles are few) above.  Measured on GB300: at
// m = 32..64 the tensor-core kernel is 1.3-1.9x faster on 4096..14336-row
// matrices; at m = 16 the streaming kernel is 1.4x faster.
constexpr int kAutoStreamMaxM = 16;
bool decode_supported(int64_t m, int64_t n_out, int64_t n_in, int num_sms);
cudaError_t launch_decode(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                          int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                          cudaStream_t stream);

// y32 = x . W_base^T in fp32 ([m, n_out] row-major) on the tensor-core kernel, W_base taken as
// stored (the shared base product of the multi-tenant path).
cudaError_t launch_base_product(const void *x, int64_t m, const void *w_base, int64_t n_out, int64_t n_in,
                                float *y32, const DevCtx &ctx, cudaStream_t stream);

// W_eff = bf16(fp32(W_base) + alpha * s) materialised in HBM (for a standard matmul).
cudaError_t launch_reconstruct(const void *w_base, const uint8_t *bits, const float *alpha, int32_t alpha_mode,
                               int64_t n_out, int64_t n_in, void *w_eff, const DevCtx &ctx, cudaStream_t stream);

// TMA-fed variant of the streaming kernel (n_in % 128 == 0, 16-byte aligned
// W_base and bits); preferred whenever it applies.
bool decode_tma_supported(int64_t m, int64_t n_out, int64_t n_in, const void *w_base, const uint8_t *bits,
                          const DevCtx &ctx);
cudaError_t launch_decode_tma(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                              int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                              cudaStream_t stream);

// Several independent streaming linears (m <= kBatchMaxM each) in one launch
// with the K steps of all of them split evenly over the resident CTAs
// (decode_batch.cu).  The workspace holds one counter per 64-row block (zero
// between launches) and the fp32 partials of blocks split between CTAs.
constexpr int kBatchMaxProblems = 8;
constexpr int64_t kBatchMaxM = 16;
struct BatchItem {
    const void *x;
    const void *w_base;
    const uint8_t *bits;
    const float *alpha;
    void *y;
    int64_t m, n_out, n_in;
    int32_t alpha_mode;
};
struct BatchPlan {
    bool ok;
    int nt;                 // token tiles of 8 (from the largest m)
    int64_t grid;           // CTAs
    int64_t total_items;    // (64-row block, 128-column K step) pairs over all linears
    int64_t blocks;         // 64-row blocks over all linears
    int32_t parts_max;      // most CTAs sharing one block
    size_t counter_bytes;   // counters at the start of the workspace (256-byte multiple)
    size_t workspace_bytes;
};
bool decode_batch_supported(int64_t m, int64_t n_out, int64_t n_in, const void *x, const void *w_base,
                            const uint8_t *bits, const void *y);
BatchPlan plan_decode_batch(const BatchItem *items, int n, const DevCtx &ctx);
// The same list on the cluster-split kernel (decode_tma.cu): one launch, every linear's
// 64-row blocks split over one cluster size; no workspace.
bool decode_tma_multi_supported(const BatchItem *items, int n);
bool decode_tma_multi_one_wave(const BatchItem *items, int n, const DevCtx &ctx);  // its CTAs fit at once
cudaError_t launch_decode_tma_multi(const BatchItem *items, int n, const DevCtx &ctx, cudaStream_t stream);
cudaError_t launch_decode_batch(const BatchItem *items, int n, const BatchPlan &plan, void *workspace,
                                const DevCtx &ctx, cudaStream_t stream);

// Tensor-core kernel on CTA pairs (prefill_pair.cu): 256 W rows x 256 tokens per pair
// of CTAs (tcgen05 cta_group::2), no K split.
bool prefill_pair_supported(int64_t m, int64_t n_out, int64_t n_in, const DevCtx &ctx);
int64_t prefill_pair_tiles(int64_t m, int64_t n_out);
// Up to 8 independent linears (m > 64 each) in one launch of the pair kernel, their pair
// tiles numbered linear by linear (a layer's q/k/v or gate/up share one wave sequence).
constexpr int kPairMaxLinears = 8;
bool prefill_pair_multi_supported(const BatchItem *items, int n, const DevCtx &ctx);
cudaError_t launch_prefill_pair_multi(const BatchItem *items, int n, const DevCtx &ctx, cudaStream_t stream);
cudaError_t launch_prefill_pair(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                                int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                                cudaStream_t stream);

// Tensor-core (tcgen05 + TMA) kernel for any m: CTA pairs when their tiles fill the
// GPU, else one CTA per 128 x 256 tile (K split over a cluster when tiles are few).
cudaError_t launch_prefill(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                           int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const DevCtx &ctx,
                           cudaStream_t stream);

// ---- multi-tenant ----------------------------------------------------------------------
constexpr int kMaxVariantsDev = 64;  // = BD_MAX_VARIANTS
struct GroupedVariants {
    const uint8_t *bits[kMaxVariantsDev];
    const float *alpha[kMaxVariantsDev];
    int32_t mode[kMaxVariantsDev];
    int32_t count;
};
// Device-built schedule of the multi-tenant tensor-core path: `tiles` holds
// (variant, first row in the variant-sorted activations, rows <= 256) per
// token tile, `*n_tiles` how many are valid, `perm` maps sorted rows back to
// original tokens; the grid is sized for `max_slots` tiles per W row tile.
struct GroupTable {
    const int32_t *tiles;
    const int32_t *n_tiles;
    const int32_t *perm;
    int32_t max_slots;
};
cudaError_t launch_prefill_grouped(const void *x_sorted, int64_t m, const void *w_base, const GroupedVariants &vars,
                                   int64_t n_out, int64_t n_in, void *y, const GroupTable &tab, const DevCtx &ctx,
                                   cudaStream_t stream);
// The same on CTA pairs: 256 W rows per pair and a token tile of one variant.
cudaError_t launch_prefill_pair_grouped(const void *x_sorted, int64_t m, const void *w_base,
                                        const GroupedVariants &vars, int64_t n_out, int64_t n_in, void *y,
                                        const GroupTable &tab, const DevCtx &ctx, cudaStream_t stream);

// Tensor-core streaming multi-tenant kernel for small batches (grouped_decode_tc.cu).
bool grouped_decode_tc_supported(int64_t m, int32_t n_variants, int64_t n_in, const void *x_sorted,
                                 const void *w_base, const GroupedVariants &vars);
cudaError_t launch_grouped_decode_tc(const void *x_sorted, int64_t m, const void *w_base, const GroupedVariants &vars,
                                     int64_t n_out, int64_t n_in, void *y, const int32_t *seg, const int32_t *perm,
                                     const DevCtx &ctx, cudaStream_t stream);

// mma.sync streaming multi-tenant kernel for small batches (grouped_decode.cu).
bool grouped_decode_supported(int64_t m, int32_t n_variants, int64_t n_in, const void *w_base,
                              const GroupedVariants &vars);
cudaError_t launch_grouped_decode(const void *x_sorted, int64_t m, const void *w_base, const GroupedVariants &vars,
                                  int64_t n_out, int64_t n_in, void *y, const int32_t *s_tiles,
                                  const int32_t *n_s_tiles, const int32_t *perm, const int32_t *n_valid,
                                  const float *ybase, const DevCtx &ctx, cudaStream_t stream);

size_t grouped_workspace_size(int64_t m, int32_t n_variants, int64_t n_out, int64_t n_in);
cudaError_t launch_grouped(const void *x, const int32_t *ids, int64_t m, const void *w_base,
                           const GroupedVariants &vars, int64_t n_out, int64_t n_in, void *y, void *ws,
                           size_t ws_bytes, const DevCtx &ctx, cudaStream_t stream);

// ---- driver entry point for tensor maps (resolved through the runtime) ---------------
bool encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                          uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle);

}  // namespace bd
