// Tensor-core (tcgen05) residual transition -- placeholder until the kernel lands.
#include "nt_common.cuh"
namespace nt {
bool transition_tc_supported(nt_dtype, int, int) { return false; }
cudaError_t launch_transition_tc(const void*, void*, int64_t, int, int, const float*, const float*,
                                 float, const void*, const float*, const void*, const float*,
                                 unsigned int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace nt
