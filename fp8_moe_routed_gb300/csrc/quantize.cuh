// quantize.cuh -- the activation quantization arithmetic of the quantizer
// kernels (quant.cu): scale = max(amax, 1e-12) / fmt_max by IEEE division, codes
// of the correctly rounded f32 quotient x / scale ("MoE: native FP8 QAT for
// routed-expert GMMs", Implementation: per-row full-K f32 scale).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fp8moe {

constexpr float kEps = 1e-12f;
constexpr float kE4m3Max = 448.0f;
constexpr float kE5m2Max = 57344.0f;

__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t acc, uint32_t v) {
  uint32_t a = v & 0x7FFF7FFFu, r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(a));
  return r;
}

__device__ __forceinline__ float bf16x2_hmax_to_f32(uint32_t v) {
  return fmaxf(bf16lo_to_f32(v), bf16hi_to_f32(v));
}

// Codes of the correctly rounded f32 quotients RN(x0 / s), RN(x1 / s), two per
// conversion, from rl = RN(r * (1 - 2^-20)) and rh = RN(r * (1 + 2^-20)),
// r = RN(1 / s).
//   r is within 2^-24 of 1 / s (relative), rl and rh add 2^-24 each, and the
//   products another 2^-24: x * rl and x * rh (as computed) lie more than 2^-21
//   below and above x / s, and RN(x / s) within 2^-24 of it, so RN(x / s) is
//   always between the two ends. Rounding to the fp8 grid (nearest, saturating)
//   is monotonic: when both ends give the same code, every value between them
//   does, RN(x / s) included. Otherwise a rounding boundary lies within ~2^-20
//   of x / s (rare) and the exact IEEE quotients are converted instead. Below
//   the f32 normal range the relative bounds fail, but such quotients and both
//   ends then round to the zero code anyway. NaN and infinite x give the codes
//   the quotient would (NaN; saturation).
template <bool E5M2>
__device__ __forceinline__ uint16_t cvt_x2(float a, float b) {
  return E5M2 ? f32x2_to_e5m2x2(a, b) : f32x2_to_e4m3x2(a, b);
}

template <bool E5M2>
__device__ __forceinline__ uint16_t quotient_x2(float x0, float x1, float s0, float s1, float rl0,
                                                float rl1, float rh0, float rh1) {
  // both bracket products as packed f32x2 multiplies (two RN multiplies each:
  // the same bits as four scalar ones, in half the instructions)
  float pl0, pl1, ph0, ph1;
  mul_f32x2(x0, x1, rl0, rl1, pl0, pl1);
  mul_f32x2(x0, x1, rh0, rh1, ph0, ph1);
  const uint16_t lo = cvt_x2<E5M2>(pl0, pl1);
  const uint16_t hi = cvt_x2<E5M2>(ph0, ph1);
  if (lo == hi) return lo;
  return cvt_x2<E5M2>(__fdiv_rn(x0, s0), __fdiv_rn(x1, s1));
}

__device__ __forceinline__ void bracket(float s, float& rl, float& rh) {
  const float r = __frcp_rn(s);
  rl = __fmul_rn(r, 1.0f - 0x1p-20f);
  rh = __fmul_rn(r, 1.0f + 0x1p-20f);
}

// 8 bf16 (one uint4) / s -> 8 e4m3 codes (one uint2). The bracket products of
// all four pairs are converted first; only when some pair's two codes differ
// (about once in 2^16 values) are the exact IEEE quotients of the eight values
// converted instead, so the common case takes one test and one branch per eight
// values (row quantizer: K = 7168 122.0 -> 120.5 us, K = 2048 39.1 -> 37.3 us at
// 32768 rows; the per-column tile quantizer measured slower this way and keeps
// quotient_x2).
__device__ __forceinline__ uint2 quant8(uint4 v, float s, float rl, float rh) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t lo[2], hi[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint16_t cl[2], ch[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float x0 = bf16lo_to_f32(w[2 * i + j]), x1 = bf16hi_to_f32(w[2 * i + j]);
      float pl0, pl1, ph0, ph1;
      mul_f32x2(x0, x1, rl, rl, pl0, pl1);
      mul_f32x2(x0, x1, rh, rh, ph0, ph1);
      cl[j] = f32x2_to_e4m3x2(pl0, pl1);
      ch[j] = f32x2_to_e4m3x2(ph0, ph1);
    }
    lo[i] = (uint32_t)cl[0] | ((uint32_t)cl[1] << 16);
    hi[i] = (uint32_t)ch[0] | ((uint32_t)ch[1] << 16);
  }
  if ((lo[0] ^ hi[0]) | (lo[1] ^ hi[1])) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint16_t c[2];
#pragma unroll
      for (int j = 0; j < 2; ++j)
        c[j] = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_to_f32(w[2 * i + j]), s),
                               __fdiv_rn(bf16hi_to_f32(w[2 * i + j]), s));
      lo[i] = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
    }
  }
  return make_uint2(lo[0], lo[1]);
}

}  // namespace fp8moe
