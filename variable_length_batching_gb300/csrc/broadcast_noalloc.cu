// nt_pair_broadcast_noalloc: the pair broadcast for callers that cannot
// allocate device memory.
//
// nt_pair_broadcast needs a caller-supplied workspace for the two projected
// single representations u and v (2 * T * C_z fp32).  Some callers have no
// way to provide one: a plug-in whose host framework owns every device
// allocation and exposes none to it, or a real-time loop that must not pay
// for an allocation (or risk an out-of-memory failure) on its hot path.
// This entry point keeps u and v in a fixed array of device memory that the
// library itself declares, so the call needs no workspace and allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library routine.
//
// Cost of the choice: every GPU that loads the library holds the array
// (kNoAllocScratchFloats * 4 bytes = 8 MiB) until the process exits, the
// problem size is capped at (T + T_cols) * C_z <= kNoAllocScratchFloats
// (2 * T * C_z for square pairs), and all
// calls share the one array, so calls that overlap on the GPU (different
// streams, or different host threads on the same device) race on it.  The
// kernels overwrite every element of u and v they read, so nothing needs to
// start at zero and the previous call's contents never leak into a result.
#include "nt_common.cuh"

namespace nt {
namespace {

constexpr size_t kNoAllocScratchFloats = size_t(1) << 21;   // 8 MiB of fp32

static __device__ __align__(256) float g_noalloc_uv[kNoAllocScratchFloats];

// Device address of g_noalloc_uv on the current device.  In host code the
// array's name is only a stand-in; the real address is looked up with the
// device current, on every call (a cheap query): after a cudaDeviceReset the
// module is loaded again and the array may sit elsewhere, so no address is
// kept from one call to the next.  With CUDA's default lazy module loading
// the first lookup on a device is what loads the module holding the array,
// which commits its 8 MiB of device memory there and can fail then.
cudaError_t noalloc_scratch(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_uv);
  if (e != cudaSuccess) return e;
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

}  // namespace
}  // namespace nt

using namespace nt;

extern "C" {

nt_status nt_pair_broadcast_noalloc(const nt_partition* part, nt_dtype dtype, const void* s_left,
                                    const void* s_right, int32_t C_s, const void* W_a, const void* W_b,
                                    int32_t C_z, void* z, void* stream) {
  if (!part) return record_error(NT_ERR_INVALID, "partition is NULL");
  if (part->T < 0 || C_z <= 0) return record_error(NT_ERR_INVALID, "T must be >= 0 and C_z > 0");
  const int64_t T_cols = t_cols_of(part);
  if (T_cols < 0) return record_error(NT_ERR_INVALID, "T_cols must be >= 0");
  const size_t need = (size_t)(part->T + T_cols) * (size_t)C_z;   // u and v
  if (need > kNoAllocScratchFloats)
    return record_error(NT_ERR_UNSUPPORTED,
                        "(T + T_cols) * C_z exceeds the 2,097,152 fp32 elements of the built-in scratch; "
                        "use nt_pair_broadcast with a caller workspace");
  float* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess)
    return record_error(NT_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch failed (the first call on a "
                                     "device loads the 8 MiB array there)");
  // The regular entry point validates every argument and launches the same
  // kernels; the library's own array stands in for the caller's workspace.
  return nt_pair_broadcast(part, dtype, s_left, s_right, C_s, W_a, W_b, C_z, z, scratch,
                           kNoAllocScratchFloats * sizeof(float), stream);
}

}  // extern "C"
