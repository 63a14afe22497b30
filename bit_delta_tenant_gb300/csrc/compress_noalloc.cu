// compress_noalloc.cu -- bd_compress_noalloc: compression for callers that
// cannot give the library any device memory beyond the inputs and outputs.
//
// Who needs it: code that runs inside a host framework which owns every
// byte of device memory through its own arena or budget (a serving runtime
// that plans memory up front and forbids stray cudaMalloc), and
// latency-critical paths where cudaMalloc's implicit device synchronisation
// is not acceptable.  Such callers can pass W_base, W_ft and the two outputs,
// but not a workspace.
//
// How: the per-block fp64 partial sums that bd_compress keeps in the caller's
// workspace live here in a fixed file-scope device array instead.  The same
// kernels as bd_compress run, so the results are identical.  The array is
// part of the library image: every GPU that loads the library holds it
// (BD_NOALLOC_MAX_PARTIALS doubles = 1 MiB) until the process exits.
#include <mutex>

#include "bd_internal.h"
#include "bitdelta.h"

#define BD_API extern "C" __attribute__((visibility("default")))

namespace {

// Shared scratch of every bd_compress_noalloc call in this process (per device).
static __device__ __align__(256) double g_noalloc_partials[BD_NOALLOC_MAX_PARTIALS];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mu;
double *g_partials_addr[kMaxDevices] = {nullptr};

// Set-up, once per device with that device current: the host-side name of a
// __device__ array is only a stand-in, so the kernels receive the device
// address returned by cudaGetSymbolAddress.
int32_t setup_device(int dev, double **partials) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_partials_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr) return BD_ERR_CUDA;
        g_partials_addr[dev] = static_cast<double *>(p);
    }
    *partials = g_partials_addr[dev];
    return BD_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

BD_API int32_t bd_compress_noalloc(const void *w_base, const void *w_ft, int64_t n_out, int64_t n_in,
                                   int32_t alpha_mode, uint8_t *bits_out, float *alpha_out, void *stream) {
    if (!w_base || !w_ft || !bits_out || !alpha_out) return BD_ERR_INVALID_ARG;
    if (alpha_mode != BD_ALPHA_SCALAR && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    if (n_out < 1 || n_in < 1) return BD_ERR_INVALID_ARG;
    if (n_in % 8 != 0 || n_out >= BD_MAX_DIM || n_in >= BD_MAX_DIM) return BD_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(w_base) || !aligned16(w_ft) || !aligned16(bits_out) || !aligned16(alpha_out))
        return BD_ERR_MISALIGNED;
    // The built-in scratch holds BD_NOALLOC_MAX_PARTIALS partial sums; shapes
    // needing more must use bd_compress with a caller-provided workspace.  A
    // shape whose rows are one segment each needs none: pass 1 writes alpha.
    const bd::CompressGeom g = bd::compress_geometry(n_out, n_in, alpha_mode);
    if (g.segs > 1 && g.rows * g.segs > static_cast<int64_t>(BD_NOALLOC_MAX_PARTIALS)) return BD_ERR_WORKSPACE;

    bd::DevCtx ctx;
    int32_t rc = bd::make_dev_ctx(&ctx);  // status word and wait limit, as for bd_compress
    if (rc != BD_OK) return rc;
    if (ctx.device >= kMaxDevices) return BD_ERR_CUDA;
    double *partials = nullptr;
    rc = setup_device(ctx.device, &partials);
    if (rc != BD_OK) return rc;
    // Every partial slot the kernels read is written earlier in the same call
    // (one slot per block of the first pass), so nothing needs clearing.  The
    // compression kernels are programmatic dependents of the kernel before
    // them and wait for it before touching the partials, so calls queued on
    // one stream never overlap on the array.
    const cudaError_t e = bd::launch_compress(w_base, w_ft, n_out, n_in, alpha_mode, bits_out, alpha_out, partials,
                                              ctx, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}
