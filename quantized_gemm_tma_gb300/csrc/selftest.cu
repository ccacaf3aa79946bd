// selftest.cu — a kernel whose one wait cannot complete, for tests of the
// failure path every library kernel shares: a bounded mbarrier wait runs out
// (about 2 s), the CTA records HQ_ERR_DEVICE_TIMEOUT in the status word and
// exits normally, and the context stays usable.  No trap, no bad address.
#include <cuda_runtime.h>

#include "hq_launch.h"
#include "hq_ptx.cuh"

namespace hq {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  if (threadIdx.x == 0) {
    dev::mbar_init(&bar, 1);  // one arrival expected; nothing arrives
    *abort_flag = 0;
    dev::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !dev::mbar_wait(&bar, 0, abort_flag))
    dev::raise_error(status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout(int* status, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace hq
