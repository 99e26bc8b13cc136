// groups.cuh -- ragged group layout, computed on the device by every CTA.
//
// Rows of expert e are [begin[e], end[e]) of the static buffer of M rows:
// begin = exclusive prefix sum of the group sizes, negative sizes count as 0 and
// both ends are clipped at M (the status word records either fix). T = rows
// covered by some group. Nothing here ever reads a row of the buffer.
#pragma once
#include <cstdint>
#include "fp8moe_status.cuh"

namespace fp8moe {

constexpr int kMaxExperts = 1024;

// Warp 0 of the block fills s_begin/s_end[E] and *s_T; the caller synchronizes
// afterwards. report != 0: also record clamping in the status word.
__device__ __forceinline__ void load_groups_warp0(const int32_t* __restrict__ gs, int E,
                                                  int64_t M, int32_t* s_begin, int32_t* s_end,
                                                  int32_t* s_T, int report) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int64_t carry = 0;
  bool neg = false;
  for (int base = 0; base < E; base += 32) {
    int e = base + lane;
    int64_t g = 0;
    if (e < E) {
      int32_t v = __ldg(gs + e);
      if (v < 0) neg = true;
      g = v < 0 ? 0 : v;
    }
    // inclusive scan over the warp
    int64_t incl = g;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int64_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int64_t excl = carry + incl - g;
    if (e < E) {
      s_begin[e] = (int32_t)(excl < M ? excl : M);
      int64_t en = excl + g;
      s_end[e] = (int32_t)(en < M ? en : M);
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  neg = __any_sync(0xffffffffu, neg);
  if (lane == 0) {
    *s_T = (int32_t)(carry < M ? carry : M);
    if (report) {
      if (neg) status_set(kStatusNegativeGroup);
      if (carry > M) status_set(kStatusGroupsExceedM);
    }
  }
}

// Given prefix[0..E] (ascending), the e with prefix[e] <= u < prefix[e+1].
__device__ __forceinline__ int find_bucket(const int32_t* prefix, int E, int32_t u) {
  int lo = 0, hi = E;   // invariant: prefix[lo] <= u < prefix[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace fp8moe
