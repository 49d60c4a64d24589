// Self-test of the device-side failure path: one CTA waits on an mbarrier that
// nothing ever arrives on.  The bounded wait gives up after its deadline, records
// FA_ERR_TIMEOUT in the device status word and the kernel returns normally, so
// the context stays usable.  Used by the tests to check failure detection
// without faulting or hanging the GPU.
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__global__ void wait_timeout_kernel(unsigned int* status) {
  __shared__ __align__(8) uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&never, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, status};
  if (threadIdx.x == 0) (void)mbar_wait(&never, 0, wc);  // nobody arrives: times out
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned int* status, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace fa
