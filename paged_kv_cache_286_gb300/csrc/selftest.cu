// Self-test of the bounded device-side wait that every kernel of the library uses.
//
// One thread initialises an mbarrier that nothing ever arrives on and waits for its first phase
// with the library's own bounded wait (mbar_wait).  The wait must give up after the limit and
// record PA_DEVERR_TIMEOUT in the workspace's error word, the same signal a kernel raises when
// a copy it waits for never lands; the kernel then returns normally, so the context stays
// usable.  Nothing is copied and no memory outside the error word is touched.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(uint32_t* err,
                                                                   uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!mbar_wait(&bar, 0, limit_ns)) set_error(err, PA_DEVERR_TIMEOUT);
}

cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace pa
