// Tensor-core (tcgen05) varlen attention -- placeholder until the kernel lands.
#include "nt_common.cuh"
namespace nt {
bool attn_tc_supported(nt_dtype, int) { return false; }
cudaError_t launch_attn_tc(const void*, const void*, const void*, const int32_t*, int32_t, int64_t,
                           int32_t, int, int, float, void*, float*, unsigned int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace nt
