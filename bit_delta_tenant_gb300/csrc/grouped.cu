// grouped.cu -- multi-tenant fused linear (placeholder until the grouped kernels land).
#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {

size_t grouped_workspace_size(int64_t m, int32_t n_variants, int64_t n_out, int64_t n_in) {
    (void)n_out;
    return static_cast<size_t>((m + 8 * n_variants) * n_in * 2 + (m + 4 * n_variants + 1024) * 16);
}

cudaError_t launch_grouped(const void *, const int32_t *, int64_t, const void *, const GroupedVariants &, int64_t,
                           int64_t, void *, void *, size_t, const DevCtx &, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace bd
