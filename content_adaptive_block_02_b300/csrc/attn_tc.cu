// Placeholder for the tcgen05 attention kernels (filled in next).
#include "prism_internal.cuh"

namespace prism {
cudaError_t launch_attn_fwd_tc(const Plan&, const uint16_t*, const uint16_t*, const uint16_t*,
                               const int32_t*, const int32_t*, const int32_t*, float, uint16_t*,
                               float*, uint8_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_attn_bwd_tc(const Plan&, const uint16_t*, const uint16_t*, const uint16_t*,
                               const uint16_t*, const float*, const float*, const int32_t*,
                               const int32_t*, const int32_t*, float, float*, uint16_t*,
                               uint16_t*, uint8_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace prism
