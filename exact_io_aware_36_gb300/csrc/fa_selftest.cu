// fa_selftest.cu -- on-device check of the failure path of the pipelines.
//
// Every pipeline wait in the kernels is bounded: when a barrier phase never
// completes, the waiting warp records FA_ERR_DEVICE_TIMEOUT, raises the
// CTA's abort flag and returns.  This kernel runs that same wait (wait_warp)
// on a barrier nothing ever arrives on, so a caller can confirm on its own
// device that a stall comes back as an error status, within the limit, and
// that the context stays usable afterwards.
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace {

__global__ void __launch_bounds__(32) selftest_wait_kernel(unsigned int* status,
                                                           unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    fa::mbar_init(&bar, 1);          // expects one arrival that never comes
    abort_flag = 0;
    fa::fence_mbarrier_init();
  }
  __syncwarp();
  const fa::WaitCtx wc{&abort_flag, status, limit_ns};
  fa::wait_warp(&bar, 0, wc);        // returns false after limit_ns
}

}  // namespace

namespace fa {
int launch_selftest_wait(unsigned int* status, unsigned long long limit_ns, void* stream) {
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  return (int)cudaGetLastError();
}
}  // namespace fa
