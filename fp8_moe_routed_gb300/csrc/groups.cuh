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

// Warp 0 of the block writes the row range [*s_lo, *s_hi) of experts [e0, e1)
// (clipped at M like load_groups_warp0) without per-expert arrays; the caller
// synchronizes afterwards. report != 0: also record clamping in the status word.
__device__ __forceinline__ void group_row_range_warp0(const int32_t* __restrict__ gs, int E,
                                                      int64_t M, int e0, int e1, int32_t* s_lo,
                                                      int32_t* s_hi, int report) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int64_t before = 0, upto = 0, total = 0;   // sums over e < e0, e < e1, all e
  bool neg = false;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    int64_t g = 0;
    if (e < E) {
      const int32_t v = __ldg(gs + e);
      if (v < 0) neg = true;
      g = v < 0 ? 0 : v;
    }
    int64_t a = e < e0 ? g : 0, b = e < e1 ? g : 0, c = g;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, d);
      b += __shfl_xor_sync(0xffffffffu, b, d);
      c += __shfl_xor_sync(0xffffffffu, c, d);
    }
    before += a;
    upto += b;
    total += c;
  }
  neg = __any_sync(0xffffffffu, neg);
  if (lane == 0) {
    *s_lo = (int32_t)(before < M ? before : M);
    *s_hi = (int32_t)(upto < M ? upto : M);
    if (report) {
      if (neg) status_set(kStatusNegativeGroup);
      if (total > M) status_set(kStatusGroupsExceedM);
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
