// fp8moe_status.cuh -- the device status word.
//
// Data-dependent problems that the host cannot see without synchronizing (a
// negative group size, group sizes that add up past the static buffer, a
// pipeline wait that ran out of time) set bits in a per-translation-unit device
// word; fp8moe_read_status() collects and clears them. Kernels never trap.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fp8moe {

constexpr uint32_t kStatusNegativeGroup = 1u << 0;
constexpr uint32_t kStatusGroupsExceedM = 1u << 1;
constexpr uint32_t kStatusWaitTimeout = 1u << 2;
constexpr uint32_t kStatusTooManySegments = 1u << 3;
// bits [8, 16) name the wait that timed out
constexpr uint32_t kWhereProducer = 1u << 8;
constexpr uint32_t kWhereMma = 2u << 8;
constexpr uint32_t kWhereEpilogue = 3u << 8;
constexpr uint32_t kWhereDequant = 4u << 8;
constexpr uint32_t kWhereDrain = 5u << 8;
constexpr uint32_t kWhereSelftest = 6u << 8;

static __device__ uint32_t g_status_word;

__device__ __forceinline__ void status_set(uint32_t bits) { atomicOr(&g_status_word, bits); }

}  // namespace fp8moe

// Defines `uint32_t <fn>(cudaStream_t)`: waits for the stream, returns this
// translation unit's status word and clears it.
#define FP8MOE_DEFINE_STATUS_TAKE(fn)                                              \
  uint32_t fn(cudaStream_t s) {                                                    \
    uint32_t v = 0, z = 0;                                                         \
    if (cudaMemcpyFromSymbolAsync(&v, fp8moe::g_status_word, 4, 0,                 \
                                  cudaMemcpyDeviceToHost, s) != cudaSuccess)       \
      return 0xFFFFFFFFu;                                                          \
    if (cudaStreamSynchronize(s) != cudaSuccess) return 0xFFFFFFFFu;               \
    if (cudaMemcpyToSymbolAsync(fp8moe::g_status_word, &z, 4, 0,                   \
                                cudaMemcpyHostToDevice, s) != cudaSuccess)         \
      return 0xFFFFFFFFu;                                                          \
    if (cudaStreamSynchronize(s) != cudaSuccess) return 0xFFFFFFFFu;               \
    return v;                                                                      \
  }
