// dequant.cu -- dequantize_fp8_codes: w[e, k, n] = bf16(f32(code[e, k, n]) * scale[e, n]),
// one f32 multiply then round-to-nearest-even to bf16 ("MoE: native FP8 QAT for
// routed-expert GMMs", Implementation: dequantize_fp8_codes, bit-identical to
// the weight dequantization of the fake-QAT path).
//
// HBM-bound: 1 byte read + 2 bytes written per element. Each thread converts 16
// codes (one 16-byte load, two 16-byte stores); the grid is a multiple of the SM
// count and strides over the tensor.
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "kernels.h"

namespace fp8moe {

__global__ void __launch_bounds__(256) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                         const float* __restrict__ scale, int64_t K,
                                                         int64_t N, int64_t nvec,
                                                         uint4* __restrict__ out) {
  const int64_t vpr = N >> 4;   // 16-code vectors per row (N % 16 == 0)
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
       v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = v / vpr;            // row of [E*K, N]
    const int64_t n0 = (v - row * vpr) << 4;
    const int64_t e = row / K;
    const uint4 c = __ldg(reinterpret_cast<const uint4*>(codes) + v);
    const float4* sp = reinterpret_cast<const float4*>(scale + e * N + n0);
    float sc[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 f = __ldg(sp + i);
      sc[4 * i] = f.x; sc[4 * i + 1] = f.y; sc[4 * i + 2] = f.z; sc[4 * i + 3] = f.w;
    }
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f0, f1, f2, f3;
      half2_to_f32(e4m3x2_to_f16x2((uint16_t)(cw[i] & 0xFFFFu)), f0, f1);
      half2_to_f32(e4m3x2_to_f16x2((uint16_t)(cw[i] >> 16)), f2, f3);
      o[2 * i] = f32x2_to_bf16x2(__fmul_rn(f0, sc[4 * i]), __fmul_rn(f1, sc[4 * i + 1]));
      o[2 * i + 1] = f32x2_to_bf16x2(__fmul_rn(f2, sc[4 * i + 2]), __fmul_rn(f3, sc[4 * i + 3]));
    }
    out[2 * v] = make_uint4(o[0], o[1], o[2], o[3]);
    out[2 * v + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_dequant)

cudaError_t fp8moe_launch_dequantize(const uint8_t* codes, const float* scale, int E, int64_t K,
                                     int64_t N, void* out, int num_sms, cudaStream_t s) {
  const int64_t nvec = (int64_t)E * K * N / 16;
  int64_t blocks = (nvec + 255) / 256;
  int64_t cap = (int64_t)num_sms * 8;
  int grid = (int)(blocks < cap ? blocks : cap);
  if (grid < 1) grid = 1;
  fp8moe::dequantize_kernel<<<grid, 256, 0, s>>>(codes, scale, K, N, nvec,
                                                 static_cast<uint4*>(out));
  return cudaGetLastError();
}
