// kernels.h -- internal launchers of the CUDA library (host side).  The public
// C ABI lives in include/fp8moe.h; these are the per-file entry points that
// api.cu calls after validating arguments and building tensor maps.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

// Rows of experts [e0, e1); ctas_per_sm bounds the grid (resident CTAs per SM).
cudaError_t fp8moe_launch_quantize_rows(const void* lhs, int64_t M, int K, const int32_t* gs,
                                        int E, int e0, int e1, uint8_t* q, float* sx, int num_sms,
                                        int ctas_per_sm, int report, cudaStream_t s);
// Per-512-column block quantization: codes q [M, K], bf16-valued scales sb [M, ceil(K/512)].
cudaError_t fp8moe_launch_quantize_rows_block(const void* lhs, int64_t M, int K, const int32_t* gs,
                                              int E, uint8_t* q, float* sb, int num_sms, int report,
                                              cudaStream_t s);
cudaError_t fp8moe_launch_tgmm_quantize_tiles(const void* lhs, const void* dout, int64_t M, int K,
                                              int N, const int32_t* gs, int E, int64_t Smax,
                                              uint8_t* qx, float* sx, uint8_t* qd, float* sd,
                                              int num_sms, int report, int d_fmt,
                                              cudaStream_t s);
cudaError_t fp8moe_launch_dequantize(const uint8_t* codes, const float* scale, int E, int64_t K,
                                     int64_t N, void* out, int num_sms, cudaStream_t s);

// Forward grouped matmul (FP8 x FP8 or the BF16 comparison arm).
struct GmmFwdArgs {
  CUtensorMap tmA;        // A operand tiles (codes [M, K] u8, or lhs [M, K] bf16)
  CUtensorMap tmB;        // B operand tiles (weights [E, K, N], N contiguous)
  const float* sx;        // [M] row scales (FP8 arm) or nullptr
  const float* scale;     // [E, N] channel scales (FP8 arm) or nullptr
  const int32_t* gs;      // [E]
  void* out;              // bf16 [M, Nout]
  int64_t M;
  int K, N, E, swiglu;
  int e0, e1;             // only the units of experts [e0, e1)
  int blk;                // 1: sx holds per-512-column block scales [M, ceil(K/512)] and the
                          //    accumulation across blocks is bf16 (FP8 arm only)
};
cudaError_t fp8moe_launch_gmm_fp8_fwd(const GmmFwdArgs& a, int num_sms, cudaStream_t s);
cudaError_t fp8moe_launch_gmm_bf16_fwd(const GmmFwdArgs& a, int num_sms, cudaStream_t s);

struct GmmDlhsArgs {
  CUtensorMap tmA;        // dout [M, N] bf16 tiles
  CUtensorMap tmC;        // codes [E, K, N] u8 tiles [256 k x 64 n], no swizzle
  CUtensorMap tmCp;       // the same codes as [128 k x 64 n] tiles, 64-byte swizzle (pair path)
  const float* scale;     // [E, N]
  const int32_t* gs;
  const void* gu;         // bf16 [M, 2K] wi output (gate | up) for the dSwiGLU epilogue, or null
  void* dlhs;             // bf16 [M, K], or [M, 2K] dgu with the dSwiGLU epilogue
  int64_t M;
  int N, K, E;
};
// path: 0 streaming, 1 on-chip weight cache (N <= 256), 2 CTA pairs with the
// dequantized weight in tensor memory.
cudaError_t fp8moe_launch_gmm_dlhs(const GmmDlhsArgs& a, int num_sms, int path, cudaStream_t s);
// The pair kernel alone (gmm_dlhs_pair.cu); fp8moe_launch_gmm_dlhs routes path 2 here.
cudaError_t fp8moe_launch_gmm_dlhs_pair(const GmmDlhsArgs& a, int num_sms, cudaStream_t s);

struct TgmmArgs {
  CUtensorMap tmX;        // qx slots [S, 128, K] u8
  CUtensorMap tmD;        // qd slots [S, 128, N] u8
  CUtensorMap tmW;        // dW [E, K, N] f32 (store)
  const float* sx;        // [S, K]
  const float* sd;        // [S, N]
  const int32_t* gs;
  float* dW;              // [E, K, N]
  int64_t M;
  int K, N, E;
  int d_fmt;              // qd codes: 0 e4m3, 1 e5m2
};
cudaError_t fp8moe_launch_tgmm(const TgmmArgs& a, int num_sms, cudaStream_t s);

// Records the CUDA error that fp8moe_last_cuda_error() reports (api.cu).
extern "C" void fp8moe_internal_set_cuda_error(int e);
extern "C" int fp8moe_internal_check_fwd_args(const void* lhs, int64_t M, int64_t K,
                                              const uint8_t* codes, const float* scale, int32_t E,
                                              int64_t N, const int32_t* gs, const void* out,
                                              int swiglu, int* empty);

uint32_t fp8moe_status_take_quant(cudaStream_t s);
uint32_t fp8moe_status_take_dequant(cudaStream_t s);
uint32_t fp8moe_status_take_gmm_fwd(cudaStream_t s);
uint32_t fp8moe_status_take_dlhs(cudaStream_t s);
uint32_t fp8moe_status_take_dlhs_pair(cudaStream_t s);
uint32_t fp8moe_status_take_tgmm(cudaStream_t s);
uint32_t fp8moe_status_take_selftest(cudaStream_t s);

// One thread waits on an mbarrier that nothing completes for limit_ns, then
// records a wait timeout (selftest.cu).
cudaError_t fp8moe_launch_selftest_wait(uint64_t limit_ns, cudaStream_t s);
// Converts n f32 values to fp8 codes (fmt 0 e4m3, 1 e5m2) with the quantizers'
// cast (selftest.cu).
cudaError_t fp8moe_launch_selftest_cast(const float* x, int64_t n, int fmt, uint8_t* out,
                                        int num_sms, cudaStream_t s);
