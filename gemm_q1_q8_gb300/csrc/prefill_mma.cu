// tcgen05 MMA prefill path (placeholder until the kernel lands).
#include "gq_internal.cuh"

namespace gq {
GQ_ERROR_ACCESSOR(prefill_mma)
cudaError_t launch_prefill_mma(const uint32_t*, const float*, const uint16_t*, const uint16_t*, float*, int, int, int,
                               cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace gq
