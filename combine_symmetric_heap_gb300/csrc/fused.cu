// fused.cu -- persistent single-launch pipeline (placeholder until built).
#include "symmoe_dev.cuh"

namespace symmoe {
cudaError_t launch_fused(const sym_heap &, const float *, const uint16_t *, const uint16_t *,
                         const uint16_t *, const uint16_t *, int32_t *, float *, uint16_t *, int,
                         cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace symmoe
