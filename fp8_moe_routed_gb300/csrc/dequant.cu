// dequant.cu -- dequantize_fp8_codes: w[e, k, n] = bf16(f32(code[e, k, n]) * scale[e, n]),
// one f32 multiply then round-to-nearest-even to bf16 ("MoE: native FP8 QAT for
// routed-expert GMMs", Implementation: dequantize_fp8_codes, bit-identical to
// the weight dequantization of the fake-QAT path).
//
// HBM-bound: 1 byte read + 2 bytes written per element. A CTA takes four whole
// rows of [E*K, N] per step (grid-stride over row blocks); each thread converts
// the same 16-code vector of the four rows (four loads in flight) and writes each vector's
// 32 output bytes with one 32-byte store (two 16-byte stores when the output is
// only 16-byte aligned), so a warp writes whole lines.
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "kernels.h"

namespace fp8moe {

constexpr int kDqThreads = 256;
constexpr int kRows = 4;

__device__ __forceinline__ void load_scales16(const float* __restrict__ srow, int64_t n0,
                                              float (&sc)[16]) {
  const float4* sp = reinterpret_cast<const float4*>(srow + n0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = __ldg(sp + i);
    sc[4 * i] = f.x; sc[4 * i + 1] = f.y; sc[4 * i + 2] = f.z; sc[4 * i + 3] = f.w;
  }
}

__device__ __forceinline__ void dequant16(uint4 c, const float (&sc)[16], uint32_t (&o)[8]) {
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float f0, f1, f2, f3;
    half2_to_f32(e4m3x2_to_f16x2((uint16_t)(cw[i] & 0xFFFFu)), f0, f1);
    half2_to_f32(e4m3x2_to_f16x2((uint16_t)(cw[i] >> 16)), f2, f3);
    o[2 * i] = f32x2_to_bf16x2(__fmul_rn(f0, sc[4 * i]), __fmul_rn(f1, sc[4 * i + 1]));
    o[2 * i + 1] = f32x2_to_bf16x2(__fmul_rn(f2, sc[4 * i + 2]), __fmul_rn(f3, sc[4 * i + 3]));
  }
}

__device__ __forceinline__ void store32(uint4* dst, const uint32_t (&o)[8], bool v32) {
  if (v32) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(o[0]),
                 "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                 : "memory");
  } else {
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

template <bool ONE_V>
__global__ void __launch_bounds__(kDqThreads, 3) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                                   const float* __restrict__ scale,
                                                                   int64_t rows, int64_t K, int64_t N,
                                                                   uint4* __restrict__ out) {
  const int64_t vpr = N >> 4;   // 16-code vectors per row (N % 16 == 0)
  const bool v32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  // The kRows rows of a step share one expert (K % 16 == 0 and the first row is
  // a multiple of kRows), so their scales are loaded once per step; when every
  // thread owns a single vector of columns (ONE_V: N <= 16 * kDqThreads) they
  // stay in registers until the expert changes. The load/store pipe, not DRAM,
  // was the limit while every row reloaded them.
  float sc[16];
  int64_t e_keep = -1;
  // kRows rows per CTA step: every thread has kRows loads in flight
  for (int64_t r0 = (int64_t)blockIdx.x * kRows; r0 < rows; r0 += (int64_t)gridDim.x * kRows) {
    const int64_t e = r0 / K;
    for (int64_t v = threadIdx.x; v < vpr; v += kDqThreads) {
      uint4 c[kRows];
#pragma unroll
      for (int i = 0; i < kRows; ++i)
        c[i] = r0 + i < rows ? __ldg(reinterpret_cast<const uint4*>(codes + (r0 + i) * N) + v)
                             : make_uint4(0u, 0u, 0u, 0u);
      if (!ONE_V || e != e_keep) {
        load_scales16(scale + e * N, v << 4, sc);
        e_keep = e;
      }
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        if (r0 + i < rows) {
          uint32_t o[8];
          dequant16(c[i], sc, o);
          store32(out + (r0 + i) * (N >> 3) + 2 * v, o, v32);
        }
      }
    }
  }
}

}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_dequant)

cudaError_t fp8moe_launch_dequantize(const uint8_t* codes, const float* scale, int E, int64_t K,
                                     int64_t N, void* out, int num_sms, cudaStream_t s) {
  const int64_t rows = (int64_t)E * K;
  const int64_t blocks = (rows + fp8moe::kRows - 1) / fp8moe::kRows;
  const int64_t cap = (int64_t)num_sms * 3;   // the 3 CTAs of 256 threads resident per SM
  int grid = (int)(blocks < cap ? blocks : cap);
  if (grid < 1) grid = 1;
  if (N <= 16 * fp8moe::kDqThreads)
    fp8moe::dequantize_kernel<true><<<grid, fp8moe::kDqThreads, 0, s>>>(
        codes, scale, rows, K, N, static_cast<uint4*>(out));
  else
    fp8moe::dequantize_kernel<false><<<grid, fp8moe::kDqThreads, 0, s>>>(
        codes, scale, rows, K, N, static_cast<uint4*>(out));
  return cudaGetLastError();
}
