// Self-test of the device-side failure reporting.  The tensor-core kernels
// bound every mbarrier wait (mbar_wait in tc_ptx.cuh): a wait that runs out
// raises its CTA's abort flag and sets the timeout bit of the device status
// word, and the CTA's other roles, seeing the flag, give up their own waits
// without flagging again.  This kernel drives that same wait through each of
// its three outcomes on a barrier of its own, so the reporting path can be
// checked on a GPU without a protocol fault in a real kernel.
#include "nt_common.cuh"
#include "tc_ptx.cuh"

namespace nt {
namespace {

using namespace tc;

// One CTA of 64 threads.  Warp 0 waits, as one warp, on a barrier with an
// arrival count of 1 that thread 32 either completes after delay_ns (mode 0),
// never completes (mode 1: the wait runs out after limit_ns), or leaves
// incomplete while raising the abort flag after delay_ns (mode 2).  result[0]
// = 1 if the wait succeeded, else 0; result[1] = its duration in ns.  Every
// loop here ends: the wait by limit_ns, thread 32's delay by delay_ns, both
// checked on the host to be at most 2 s.
__global__ void selftest_wait_kernel(int mode, uint64_t delay_ns, uint64_t limit_ns, int64_t* result,
                                     unsigned int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const uint64_t t0 = global_timer_ns();
    const bool ok = mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
    const bool all = __all_sync(0xffffffffu, ok);
    const uint64_t t1 = global_timer_ns();
    if (threadIdx.x == 0) {
      result[0] = all ? 1 : 0;
      result[1] = (int64_t)(t1 - t0);
    }
  } else if (threadIdx.x == 32 && mode != 1) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < delay_ns) __nanosleep(1000);
    if (mode == 0) {
      mbar_arrive(&bar);
    } else {
      *static_cast<volatile int*>(&abort_flag) = 1;
    }
  }
}

}  // namespace

cudaError_t launch_selftest_wait(int mode, uint64_t delay_ns, uint64_t limit_ns, int64_t* result,
                                 unsigned int* status, cudaStream_t s) {
  selftest_wait_kernel<<<1, 64, 0, s>>>(mode, delay_ns, limit_ns, result, status);
  return cudaGetLastError();
}

}  // namespace nt
