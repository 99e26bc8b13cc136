// selftest.cu -- the failure path of the bounded pipeline waits, on demand.
//
// Every mbarrier wait in the library gives up after a time limit, records
// FP8MOE_STATUS_WAIT_TIMEOUT (plus where) in the device status word and lets its
// kernel finish, so a broken pipeline ends with a status the host can read
// instead of hanging the GPU. This kernel exercises exactly that path: one
// thread waits on an mbarrier that nothing ever arrives on, with a short limit,
// and returns. The context stays usable afterwards.
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "kernels.h"

namespace fp8moe {

__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  // phase 0 never completes: no thread arrives and no copy counts bytes on it
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(&bar, 0)) return;
    if ((it & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) {
      status_set(kStatusWaitTimeout | kWhereSelftest);
      return;
    }
  }
}

}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_selftest)

cudaError_t fp8moe_launch_selftest_wait(uint64_t limit_ns, cudaStream_t s) {
  fp8moe::selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}
