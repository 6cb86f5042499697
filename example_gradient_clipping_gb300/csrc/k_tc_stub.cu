// Placeholder until the tensor-core kernels land: every shape takes the SIMT path.
#include "tc.cuh"

namespace dph {
bool tc_sum_supported(const Geom&) { return false; }
size_t tc_sum_ws_bytes(const Geom&) { return 0; }
cudaError_t launch_tc_sum(const Geom&, const void*, const void*, const float*, float*, float*, int,
                          float*, cudaStream_t) { return cudaErrorNotSupported; }
bool tc_ghost_supported(const Geom&) { return false; }
size_t tc_ghost_ws_bytes(const Geom&) { return 0; }
cudaError_t launch_tc_ghost(const Geom&, const void*, const void*, float*, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace dph
