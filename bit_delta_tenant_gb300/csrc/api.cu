// api.cu -- the extern "C" boundary of libbitdelta.so (declared in
// include/bitdelta.h): argument validation before any launch, the sticky
// device status word, the wait-limit knob, path dispatch for the fused
// linear, and tensor-map encoding through the runtime's driver entry point
// (so the library needs no link-time dependency on the driver library).
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "bd_internal.h"
#include "bitdelta.h"

#define BD_API extern "C" __attribute__((visibility("default")))

// Sticky device status word (bits bd::kDevTimeout, bd::kDevBadVariant).  Kernels
// receive its device address; the host reads and clears it in bd_get_device_status.
__device__ unsigned int g_bd_status_word;

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_mu;
unsigned *g_status_ptr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};
std::atomic<int64_t> g_wait_ns{-1};
std::atomic<int32_t> g_linear_path{0};
std::atomic<int32_t> g_weight_prefetch{0};
constexpr int kNumOptions = BD_OPT_PAIR_RING + 1;
std::atomic<int64_t> g_options[kNumOptions] = {};

int64_t wait_limit_ns() {
    int64_t v = g_wait_ns.load();
    if (v < 0) {
        int64_t expected = -1;
        g_wait_ns.compare_exchange_strong(expected, 2000000000LL);  // 2 s
        v = g_wait_ns.load();
    }
    return v;
}

// Largest value each bd_set_option knob accepts (index = BD_OPT_*).
int64_t option_max(int32_t option) {
    switch (option) {
        case BD_OPT_COMPRESS_FORM: return 1;
        case BD_OPT_GROUPED_PATH: return 4;
        case BD_OPT_BATCH_KERNEL: return 2;
        case BD_OPT_BATCH_SINGLE: return 1;
        case BD_OPT_BATCH_GRID: return 0x7FFFFFFFLL;
        case BD_OPT_TEST_STALL: return 1;
        case BD_OPT_PREFILL_KERNEL: return 2;
        case BD_OPT_PAIR_RING: return 2;
        default: return -1;
    }
}

int32_t make_ctx(bd::DevCtx *ctx) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BD_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_status_ptr[dev] == nullptr) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_bd_status_word) != cudaSuccess) return BD_ERR_CUDA;
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BD_ERR_CUDA;
            g_status_ptr[dev] = static_cast<unsigned *>(p);
            g_num_sms[dev] = sms;
        }
        ctx->status = g_status_ptr[dev];
        ctx->num_sms = g_num_sms[dev];
    }
    ctx->device = dev;
    ctx->weight_prefetch = g_weight_prefetch.load() != 0;
    ctx->wait_ns = static_cast<uint64_t>(wait_limit_ns());
    ctx->test_stall = g_options[BD_OPT_TEST_STALL].load() != 0;
    return BD_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int32_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return BD_OK;
    return BD_ERR_CUDA;
}

int32_t check_matrix_shape(int64_t n_out, int64_t n_in) {
    if (n_out < 1 || n_in < 1) return BD_ERR_INVALID_ARG;
    if (n_in % 8 != 0) return BD_ERR_UNSUPPORTED_SHAPE;
    if (n_out >= BD_MAX_DIM || n_in >= BD_MAX_DIM) return BD_ERR_UNSUPPORTED_SHAPE;
    return BD_OK;
}

}  // namespace

namespace bd {

int32_t make_dev_ctx(DevCtx *ctx) { return make_ctx(ctx); }

int64_t option_value(int32_t option) {
    return option > 0 && option < kNumOptions ? g_options[option].load() : 0;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                          uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace bd

BD_API int32_t bd_version(void) { return 100; }

BD_API int32_t bd_build_flags(void) {
#ifdef BD_DEBUG
    return 1;
#else
    return 0;
#endif
}

BD_API const char *bd_status_string(int32_t status) {
    switch (status) {
        case BD_OK: return "ok";
        case BD_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive size or unknown mode)";
        case BD_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (n_in must be a multiple of 8; sizes below 2^31)";
        case BD_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case BD_ERR_WORKSPACE: return "workspace missing or too small";
        case BD_ERR_CUDA: return "CUDA runtime error";
        case BD_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
        case BD_ERR_BAD_VARIANT_ID: return "variant id outside [0, n_variants)";
        case BD_ERR_NO_SPACE: return "delta cache: no evictable delta leaves room for the request";
        case BD_ERR_DEVICE_BOUNDS: return "bounds-checked build: a device index failed its check (access skipped)";
        default: return "unknown status";
    }
}

BD_API int64_t bd_set_wait_limit_ns(int64_t limit_ns) {
    const int64_t prev = wait_limit_ns();
    if (limit_ns >= 0) g_wait_ns.store(limit_ns);
    return prev;
}

BD_API int32_t bd_set_linear_path(int32_t path) {
    const int32_t prev = g_linear_path.load();
    if (path >= 0 && path <= 3) g_linear_path.store(path);
    return prev;
}

BD_API int64_t bd_set_option(int32_t option, int64_t value) {
    const int64_t mx = option_max(option);
    if (mx < 0 || value < 0 || value > mx) return -1;
    return g_options[option].exchange(value);
}

BD_API int32_t bd_set_weight_prefetch(int32_t enable) {
    return g_weight_prefetch.exchange(enable != 0 ? 1 : 0);
}

BD_API int32_t bd_get_device_status(void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return BD_ERR_CUDA;
    bd::DevCtx ctx;
    const int32_t rc = make_ctx(&ctx);
    if (rc != BD_OK) return rc;
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, g_bd_status_word, sizeof(word)) != cudaSuccess) return BD_ERR_CUDA;
    const unsigned zero = 0;
    if (word != 0 && cudaMemcpyToSymbol(g_bd_status_word, &zero, sizeof(zero)) != cudaSuccess) return BD_ERR_CUDA;
    if (word & bd::kDevBounds) return BD_ERR_DEVICE_BOUNDS;
    if (word & bd::kDevTimeout) return BD_ERR_DEVICE_TIMEOUT;
    if (word & bd::kDevBadVariant) return BD_ERR_BAD_VARIANT_ID;
    return BD_OK;
}

// ---------------------------------------------------------------- compression

BD_API size_t bd_compress_workspace_size(int64_t n_out, int64_t n_in, int32_t alpha_mode) {
    if (check_matrix_shape(n_out, n_in) != BD_OK) return 0;
    if (alpha_mode != BD_ALPHA_SCALAR && alpha_mode != BD_ALPHA_PER_ROW) return 0;
    const bd::CompressGeom g = bd::compress_geometry(n_out, n_in, alpha_mode);
    return static_cast<size_t>(g.rows * g.segs) * sizeof(double);
}

BD_API int32_t bd_compress(const void *w_base, const void *w_ft, int64_t n_out, int64_t n_in, int32_t alpha_mode,
                           uint8_t *bits_out, float *alpha_out, void *workspace, size_t workspace_bytes,
                           void *stream) {
    if (!w_base || !w_ft || !bits_out || !alpha_out) return BD_ERR_INVALID_ARG;
    if (alpha_mode != BD_ALPHA_SCALAR && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    const int32_t shape = check_matrix_shape(n_out, n_in);
    if (shape != BD_OK) return shape;
    if (!aligned16(w_base) || !aligned16(w_ft) || !aligned16(bits_out) || !aligned16(alpha_out))
        return BD_ERR_MISALIGNED;
    const size_t need = bd_compress_workspace_size(n_out, n_in, alpha_mode);
    if (workspace == nullptr || workspace_bytes < need) return BD_ERR_WORKSPACE;
    if (!aligned16(workspace)) return BD_ERR_MISALIGNED;
    bd::DevCtx ctx;
    const int32_t rc = make_ctx(&ctx);
    if (rc != BD_OK) return rc;
    return cuda_status(bd::launch_compress(w_base, w_ft, n_out, n_in, alpha_mode, bits_out, alpha_out,
                                           static_cast<double *>(workspace), ctx,
                                           static_cast<cudaStream_t>(stream)));
}

namespace {

// Workspace offset of each matrix's partial sums in a batched compression (256-byte aligned regions).
size_t compress_region(const bd_compress_desc &d) {
    return (bd_compress_workspace_size(d.n_out, d.n_in, d.alpha_mode) + 255) / 256 * 256;
}

int32_t validate_compress_batch(const bd_compress_desc *d, int32_t n) {
    if (n < 0 || n > BD_COMPRESS_BATCH_MAX) return BD_ERR_INVALID_ARG;
    if (n > 0 && d == nullptr) return BD_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        const bd_compress_desc &q = d[i];
        if (q.reserved != 0) return BD_ERR_INVALID_ARG;
        if (!q.w_base || !q.w_ft || !q.bits_out || !q.alpha_out) return BD_ERR_INVALID_ARG;
        if (q.alpha_mode != BD_ALPHA_SCALAR && q.alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
        const int32_t shape = check_matrix_shape(q.n_out, q.n_in);
        if (shape != BD_OK) return shape;
        if (!aligned16(q.w_base) || !aligned16(q.w_ft) || !aligned16(q.bits_out) || !aligned16(q.alpha_out))
            return BD_ERR_MISALIGNED;
    }
    return BD_OK;
}

}  // namespace

BD_API size_t bd_compress_batch_workspace_size(const bd_compress_desc *descs, int32_t n) {
    if (validate_compress_batch(descs, n) != BD_OK) return 0;
    size_t need = 0;
    for (int32_t i = 0; i < n; ++i) need += compress_region(descs[i]);
    return need;
}

BD_API int32_t bd_compress_batch(const bd_compress_desc *descs, int32_t n, void *workspace, size_t workspace_bytes,
                                 void *stream) {
    const int32_t v = validate_compress_batch(descs, n);
    if (v != BD_OK) return v;
    if (n == 0) return BD_OK;
    const size_t need = bd_compress_batch_workspace_size(descs, n);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return BD_ERR_WORKSPACE;
    bd::DevCtx ctx;
    const int32_t rc = make_ctx(&ctx);
    if (rc != BD_OK) return rc;
    std::vector<bd::CompressItem> items;
    size_t off = 0;
    for (int32_t i = 0; i < n; ++i) {
        const bd_compress_desc &q = descs[i];
        items.push_back({q.w_base, q.w_ft, q.n_out, q.n_in, q.alpha_mode, q.bits_out, q.alpha_out,
                         reinterpret_cast<double *>(static_cast<uint8_t *>(workspace) + off)});
        off += compress_region(q);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (size_t first = 0; first < items.size(); first += bd::kCompressBatchPerLaunch) {
        const int count = static_cast<int>(std::min(items.size() - first, static_cast<size_t>(bd::kCompressBatchPerLaunch)));
        const int32_t r = cuda_status(bd::launch_compress_batch(items.data() + first, count, ctx, s));
        if (r != BD_OK) return r;
    }
    return BD_OK;
}

// ---------------------------------------------------------------- fused linear

namespace {

int32_t validate_linear(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                        int32_t alpha_mode, int64_t n_out, int64_t n_in, const void *y) {
    if (m < 0) return BD_ERR_INVALID_ARG;
    if (!w_base || !bits || !alpha) return BD_ERR_INVALID_ARG;
    if (m > 0 && (!x || !y)) return BD_ERR_INVALID_ARG;
    if (alpha_mode != BD_ALPHA_SCALAR && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    const int32_t shape = check_matrix_shape(n_out, n_in);
    if (shape != BD_OK) return shape;
    if (m >= BD_MAX_DIM) return BD_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(w_base) || !aligned16(bits) || !aligned16(alpha)) return BD_ERR_MISALIGNED;
    if (m > 0 && (!aligned16(x) || !aligned16(y))) return BD_ERR_MISALIGNED;
    return BD_OK;
}

// One validated linear with m >= 1 on the path the knob selects.
int32_t run_linear(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                   int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, const bd::DevCtx &ctx, cudaStream_t s) {
    const int32_t path = g_linear_path.load();
    const bool tma_ok = bd::decode_tma_supported(m, n_out, n_in, w_base, bits, ctx);
    const bool decode_ok = tma_ok || bd::decode_supported(m, n_out, n_in, ctx.num_sms);
    bool use_decode = decode_ok && m <= bd::kAutoStreamMaxM;
    if (path == 1) {
        if (!decode_ok) return BD_ERR_UNSUPPORTED_SHAPE;
        use_decode = true;
    } else if (path == 2) {
        use_decode = false;
    } else if (path == 3) {
        if (!bd::decode_supported(m, n_out, n_in, ctx.num_sms)) return BD_ERR_UNSUPPORTED_SHAPE;
        use_decode = true;
    }
    if (use_decode && tma_ok && path != 3)
        return cuda_status(bd::launch_decode_tma(x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y, ctx, s));
    if (use_decode)
        return cuda_status(bd::launch_decode(x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y, ctx, s));
    return cuda_status(bd::launch_prefill(x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y, ctx, s));
}

// Splits a validated batch into launches of the batched streaming kernel
// (problems grouped by m <= 8 / m <= 16, at most kBatchMaxProblems each) and
// problems that run alone.
struct BatchSchedule {
    std::vector<std::vector<bd::BatchItem>> launches;       // batched streaming kernels (m <= 16)
    std::vector<std::vector<bd::BatchItem>> pair_launches;  // tensor-core pair kernel over several linears
    std::vector<int32_t> alone;
};
int32_t schedule_batch(const bd_linear_desc *d, int32_t n, BatchSchedule &out) {
    if (n < 0 || n > BD_LINEAR_BATCH_MAX) return BD_ERR_INVALID_ARG;
    if (n > 0 && d == nullptr) return BD_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        if (d[i].reserved != 0) return BD_ERR_INVALID_ARG;
        const int32_t rc = validate_linear(d[i].x, d[i].m, d[i].w_base, d[i].bits, d[i].alpha, d[i].alpha_mode,
                                           d[i].n_out, d[i].n_in, d[i].y);
        if (rc != BD_OK) return rc;
    }
    const int32_t path = g_linear_path.load();
    // A launch of one linear gains nothing from the shared split: it runs as bd_linear
    // (the cluster-split kernel) unless the BD_OPT_BATCH_SINGLE option keeps it (tests).
    const size_t min_size = bd::option_value(BD_OPT_BATCH_SINGLE) == 1 ? 1 : 2;
    std::vector<int32_t> group[2];  // problems of the batched kernel, by token tiles
    std::vector<int32_t> tensor;    // problems for the pair kernel (m > 64)
    const bool pairs_ok = bd::option_value(BD_OPT_PREFILL_KERNEL) != 1;
    for (int32_t i = 0; i < n; ++i) {
        const bd_linear_desc &q = d[i];
        if (q.m == 0) continue;
        if ((path == 0 || path == 1) && bd::decode_batch_supported(q.m, q.n_out, q.n_in, q.x, q.w_base, q.bits, q.y))
            group[q.m <= 8 ? 0 : 1].push_back(i);
        else if ((path == 0 || path == 2) && pairs_ok && q.m > 64)
            tensor.push_back(i);
        else
            out.alone.push_back(i);
    }
    // Pair-kernel launches of up to kPairMaxLinears problems when their pair tiles together fill
    // the SMs (fewer tiles: each runs as bd_linear, which may split K on single-CTA tiles).
    bd::DevCtx ctx;
    const bool have_ctx = !tensor.empty() && make_ctx(&ctx) == BD_OK;
    for (size_t first = 0; first < tensor.size(); first += bd::kPairMaxLinears) {
        const size_t count = std::min(tensor.size() - first, static_cast<size_t>(bd::kPairMaxLinears));
        std::vector<bd::BatchItem> items;
        int64_t tiles = 0;
        for (size_t k = first; k < first + count; ++k) {
            const bd_linear_desc &q = d[tensor[k]];
            items.push_back({q.x, q.w_base, q.bits, q.alpha, q.y, q.m, q.n_out, q.n_in, q.alpha_mode});
            tiles += bd::prefill_pair_tiles(q.m, q.n_out);
        }
        if (count >= 2 && have_ctx && 2 * tiles >= ctx.num_sms &&
            bd::prefill_pair_multi_supported(items.data(), static_cast<int>(count), ctx))
            out.pair_launches.push_back(items);
        else
            out.alone.insert(out.alone.end(), tensor.begin() + first, tensor.begin() + first + count);
    }
    for (const auto &g : group) {
        for (size_t first = 0; first < g.size(); first += bd::kBatchMaxProblems) {
            const size_t count = std::min(g.size() - first, static_cast<size_t>(bd::kBatchMaxProblems));
            if (count < min_size) {
                out.alone.insert(out.alone.end(), g.begin() + first, g.begin() + first + count);
                continue;
            }
            std::vector<bd::BatchItem> items;
            for (size_t k = first; k < first + count; ++k) {
                const bd_linear_desc &q = d[g[k]];
                items.push_back({q.x, q.w_base, q.bits, q.alpha, q.y, q.m, q.n_out, q.n_in, q.alpha_mode});
            }
            out.launches.push_back(items);
        }
    }
    return BD_OK;
}

}  // namespace

BD_API int32_t bd_linear(const void *x, int64_t m, const void *w_base, const uint8_t *bits, const float *alpha,
                         int32_t alpha_mode, int64_t n_out, int64_t n_in, void *y, void *stream) {
    const int32_t v = validate_linear(x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y);
    if (v != BD_OK) return v;
    if (m == 0) return BD_OK;
    bd::DevCtx ctx;
    const int32_t rc = make_ctx(&ctx);
    if (rc != BD_OK) return rc;
    return run_linear(x, m, w_base, bits, alpha, alpha_mode, n_out, n_in, y, ctx, static_cast<cudaStream_t>(stream));
}

BD_API size_t bd_linear_batch_workspace_size(const bd_linear_desc *descs, int32_t n) {
    BatchSchedule sch;
    if (schedule_batch(descs, n, sch) != BD_OK || sch.launches.empty()) return 0;
    bd::DevCtx ctx;
    if (make_ctx(&ctx) != BD_OK) return 0;
    size_t need = 0;
    for (const auto &g : sch.launches) {
        const bd::BatchPlan pl = bd::plan_decode_batch(g.data(), static_cast<int>(g.size()), ctx);
        if (pl.ok && pl.workspace_bytes > need) need = pl.workspace_bytes;
    }
    return need;
}

BD_API int32_t bd_linear_batch(const bd_linear_desc *descs, int32_t n, void *workspace, size_t workspace_bytes,
                               void *stream) {
    BatchSchedule sch;
    const int32_t v = schedule_batch(descs, n, sch);
    if (v != BD_OK) return v;
    if (sch.launches.empty() && sch.pair_launches.empty() && sch.alone.empty()) return BD_OK;
    bd::DevCtx ctx;
    const int32_t rc = make_ctx(&ctx);
    if (rc != BD_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::vector<bd::BatchPlan> plans;
    for (const auto &g : sch.launches) {
        plans.push_back(bd::plan_decode_batch(g.data(), static_cast<int>(g.size()), ctx));
        if (!plans.back().ok) return BD_ERR_CUDA;
        if (plans.back().workspace_bytes > 0 &&
            (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
             workspace_bytes < plans.back().workspace_bytes))
            return BD_ERR_WORKSPACE;
    }
    // Launches share the workspace: each one's accesses follow the previous one's completion on the stream.
    // Kernel per launch: the cluster-split kernel when its CTAs fit in one wave (measured faster
    // there, e.g. 3 x 4096^2 at m = 1: 19.7 against 22.8 us), else the evenly split one (2 x
    // 11008x4096: 33.8 against 41.4 us); the BD_OPT_BATCH_KERNEL option forces one (tests).
    const int64_t kern = bd::option_value(BD_OPT_BATCH_KERNEL);
    for (size_t i = 0; i < sch.launches.size(); ++i) {
        const bd::BatchItem *items = sch.launches[i].data();
        const int cnt = static_cast<int>(sch.launches[i].size());
        const bool cluster = kern != 0 ? kern == 1 : bd::decode_tma_multi_one_wave(items, cnt, ctx);
        const int32_t r = cluster && bd::decode_tma_multi_supported(items, cnt)
                              ? cuda_status(bd::launch_decode_tma_multi(items, cnt, ctx, s))
                              : cuda_status(bd::launch_decode_batch(items, cnt, plans[i], workspace, ctx, s));
        if (r != BD_OK) return r;
    }
    for (const auto &g : sch.pair_launches) {
        const int32_t r = cuda_status(bd::launch_prefill_pair_multi(g.data(), static_cast<int>(g.size()), ctx, s));
        if (r != BD_OK) return r;
    }
    for (int32_t i : sch.alone) {
        const bd_linear_desc &q = descs[i];
        const int32_t r = run_linear(q.x, q.m, q.w_base, q.bits, q.alpha, q.alpha_mode, q.n_out, q.n_in, q.y, ctx, s);
        if (r != BD_OK) return r;
    }
    return BD_OK;
}

BD_API int32_t bd_reconstruct(const void *w_base, const uint8_t *bits, const float *alpha, int32_t alpha_mode,
                              int64_t n_out, int64_t n_in, void *w_eff, void *stream) {
    if (!w_base || !bits || !alpha || !w_eff) return BD_ERR_INVALID_ARG;
    if (alpha_mode != BD_ALPHA_SCALAR && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    const int32_t shape = check_matrix_shape(n_out, n_in);
    if (shape != BD_OK) return shape;
    if (!aligned16(w_base) || !aligned16(bits) || !aligned16(alpha) || !aligned16(w_eff)) return BD_ERR_MISALIGNED;
    bd::DevCtx ctx;
    const int32_t rc = make_ctx(&ctx);
    if (rc != BD_OK) return rc;
    return cuda_status(bd::launch_reconstruct(w_base, bits, alpha, alpha_mode, n_out, n_in, w_eff, ctx,
                                              static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- multi-tenant

BD_API size_t bd_linear_grouped_workspace_size(int64_t m, int32_t n_variants, int64_t n_out, int64_t n_in) {
    if (m < 0 || n_variants < 1 || n_variants > BD_MAX_VARIANTS) return 0;
    if (check_matrix_shape(n_out, n_in) != BD_OK) return 0;
    return bd::grouped_workspace_size(m, n_variants, n_out, n_in);
}

BD_API int32_t bd_linear_grouped(const void *x, const int32_t *variant_ids, int64_t m, const void *w_base,
                                 const uint8_t *const *bits_v, const float *const *alpha_v,
                                 const int32_t *alpha_modes_v, int32_t n_variants, int64_t n_out, int64_t n_in,
                                 void *y, void *workspace, size_t workspace_bytes, void *stream) {
    if (m < 0 || !w_base || !bits_v || !alpha_v || !alpha_modes_v) return BD_ERR_INVALID_ARG;
    if (n_variants < 1 || n_variants > BD_MAX_VARIANTS) return BD_ERR_INVALID_ARG;
    if (m > 0 && (!x || !y || !variant_ids)) return BD_ERR_INVALID_ARG;
    const int32_t shape = check_matrix_shape(n_out, n_in);
    if (shape != BD_OK) return shape;
    if (m >= BD_MAX_DIM) return BD_ERR_UNSUPPORTED_SHAPE;
    bd::GroupedVariants vars;
    vars.count = n_variants;
    for (int v = 0; v < n_variants; ++v) {
        if (!bits_v[v] || !alpha_v[v]) return BD_ERR_INVALID_ARG;
        if (alpha_modes_v[v] != BD_ALPHA_SCALAR && alpha_modes_v[v] != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
        if (!aligned16(bits_v[v]) || !aligned16(alpha_v[v])) return BD_ERR_MISALIGNED;
        vars.bits[v] = bits_v[v];
        vars.alpha[v] = alpha_v[v];
        vars.mode[v] = alpha_modes_v[v];
    }
    if (!aligned16(w_base)) return BD_ERR_MISALIGNED;
    if (m > 0 && (!aligned16(x) || !aligned16(y) || !aligned16(variant_ids))) return BD_ERR_MISALIGNED;
    if (m == 0) return BD_OK;
    const size_t need = bd::grouped_workspace_size(m, n_variants, n_out, n_in);
    if (workspace == nullptr || workspace_bytes < need) return BD_ERR_WORKSPACE;
    if (!aligned16(workspace)) return BD_ERR_MISALIGNED;
    bd::DevCtx ctx;
    const int32_t rc = make_ctx(&ctx);
    if (rc != BD_OK) return rc;
    return cuda_status(bd::launch_grouped(x, variant_ids, m, w_base, vars, n_out, n_in, y, workspace,
                                          workspace_bytes, ctx, static_cast<cudaStream_t>(stream)));
}
