// selftest.cu -- checks of the library's own building blocks, on demand.
//
// * selftest_wait_kernel: the failure path of the bounded pipeline waits.
//
// Every mbarrier wait in the library gives up after a time limit, records
// FP8MOE_STATUS_WAIT_TIMEOUT (plus where) in the device status word and lets its
// kernel finish, so a broken pipeline ends with a status the host can read
// instead of hanging the GPU. This kernel exercises exactly that path: one
// thread waits on an mbarrier that nothing ever arrives on, with a short limit,
// and returns. The context stays usable afterwards.
//
// * selftest_cast_kernel: the f32 -> fp8 cast that every quantizer ends in
//   (cvt.rn.satfinite on a pair of values, e4m3 or e5m2, through the same
//   helpers), on arbitrary f32 inputs, so that whole binades of bit patterns
//   can be compared with the oracle's encoder.
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

// Two values per conversion, as in the quantizers: x[2p] is the low code of the
// pair and x[2p + 1] the high one; an odd last value is converted beside a zero.
__global__ void selftest_cast_kernel(const float* __restrict__ x, int64_t n, int fmt,
                                     uint8_t* __restrict__ out) {
  const int64_t pairs = (n + 1) / 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < pairs; p += stride) {
    const int64_t i = 2 * p;
    const bool two = i + 1 < n;
    const float lo = x[i], hi = two ? x[i + 1] : 0.0f;
    const uint16_t c = fmt == 1 ? f32x2_to_e5m2x2(lo, hi) : f32x2_to_e4m3x2(lo, hi);
    out[i] = (uint8_t)(c & 0xFFu);
    if (two) out[i + 1] = (uint8_t)(c >> 8);
  }
}

}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_selftest)

cudaError_t fp8moe_launch_selftest_wait(uint64_t limit_ns, cudaStream_t s) {
  fp8moe::selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t fp8moe_launch_selftest_cast(const float* x, int64_t n, int fmt, uint8_t* out,
                                        int num_sms, cudaStream_t s) {
  const int64_t pairs = (n + 1) / 2;
  const int64_t cap = (int64_t)num_sms * 8;
  int64_t grid = (pairs + 255) / 256;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  fp8moe::selftest_cast_kernel<<<(unsigned)grid, 256, 0, s>>>(x, n, fmt, out);
  return cudaGetLastError();
}
