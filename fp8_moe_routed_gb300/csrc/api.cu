// api.cu -- the C ABI of libfp8moe.so (declared in include/fp8moe.h): argument
// checks, workspace carving, TMA tensor maps and kernel launches.  Every step of
// the path runs in the kernels of this library; there is no host fallback.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fp8moe.h"
#include "kernels.h"

namespace {

thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  int ready = 0;
  int num_sms = 0;
  int supported = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  (void)cudaGetLastError();   // do not leave a non-sticky error for the caller's next call
  return FP8MOE_ECUDA;
}

// Lazy per-device set-up: SM count, architecture check, the driver's tensor-map
// encoder.  Returns FP8MOE_OK or an error code; *sms receives the SM count.
int device_init(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FP8MOE_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp p;
    e = cudaGetDeviceProperties(&p, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    d.num_sms = p.multiProcessorCount;
    d.supported = (p.major == 10 && p.minor == 3);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return cuda_fail(e != cudaSuccess ? e : cudaErrorNotSupported);
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = 1;
  }
  if (!d.supported) return FP8MOE_EUNSUPPORTED;
  *sms = d.num_sms;
  return FP8MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t segment_bound(int64_t M, int32_t E) { return (M + 127) / 128 + E; }

// rank-2 or rank-3 tiled tensor map; dims[0] is the contiguous one.
int make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
              const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
              CUtensorMapSwizzle sw) {
  cuuint64_t gd[3];
  cuuint64_t gs[2];
  cuuint32_t bx[3];
  cuuint32_t es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = g_encode(m, dt, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = (int)r;
    return FP8MOE_ECUDA;
  }
  return FP8MOE_OK;
}

int check_common(int64_t M, int64_t K, int64_t N, int32_t E) {
  if (M < 0 || M >= (int64_t(1) << 31)) return FP8MOE_EINVAL;
  if (K <= 0 || N <= 0 || K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return FP8MOE_EINVAL;
  if (E < 1 || E > 1024) return FP8MOE_EINVAL;
  if (K % 16 != 0 || N % 16 != 0) return FP8MOE_EALIGN;
  return FP8MOE_OK;
}

struct FwdWorkspace {
  uint8_t* q;
  float* sx;
};

size_t fwd_ws_bytes(int64_t M, int64_t K) {
  return round_up((size_t)M * (size_t)K, 256) + round_up((size_t)M * 4, 256);
}

constexpr int64_t kQuantBlock = 512;
size_t fwd_block_ws_bytes(int64_t M, int64_t K) {
  const int64_t nb = (K + kQuantBlock - 1) / kQuantBlock;
  return round_up((size_t)M * (size_t)K, 256) + round_up((size_t)M * (size_t)nb * 4, 256);
}

struct TgmmWorkspace {
  uint8_t* qx;
  uint8_t* qd;
  float* sx;
  float* sd;
};

size_t tgmm_ws_bytes(int64_t M, int64_t K, int64_t N, int32_t E) {
  const size_t S = (size_t)segment_bound(M, E);
  return round_up(S * 128 * (size_t)K, 256) + round_up(S * 128 * (size_t)N, 256) +
         round_up(S * (size_t)K * 4, 256) + round_up(S * (size_t)N * 4, 256);
}

TgmmWorkspace carve_tgmm(void* ws, int64_t M, int64_t K, int64_t N, int32_t E) {
  const size_t S = (size_t)segment_bound(M, E);
  uint8_t* p = static_cast<uint8_t*>(ws);
  TgmmWorkspace w;
  w.qx = p;
  p += round_up(S * 128 * (size_t)K, 256);
  w.qd = p;
  p += round_up(S * 128 * (size_t)N, 256);
  w.sx = reinterpret_cast<float*>(p);
  p += round_up(S * (size_t)K * 4, 256);
  w.sd = reinterpret_cast<float*>(p);
  return w;
}

int gmm_fp8_fwd_impl(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                     const float* scale, int32_t E, int64_t N, const int32_t* gs, void* out,
                     void* ws, size_t ws_bytes, cudaStream_t stream, int swiglu) {
  int rc = check_common(M, K, N, E);
  if (rc) return rc;
  // SwiGLU: the up half starts at byte N/2 of each weight row, and a TMA copy's
  // inner coordinate must be a multiple of 16 bytes.
  if (swiglu && (N % 32 != 0)) return FP8MOE_EALIGN;
  if (M == 0) return FP8MOE_OK;
  if (!lhs || !codes || !scale || !gs || !out || !ws) return ws ? FP8MOE_EINVAL : FP8MOE_EWORKSPACE;
  if (!aligned16(lhs) || !aligned16(codes) || !aligned16(scale) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u) || (reinterpret_cast<uintptr_t>(gs) & 3u))
    return FP8MOE_EALIGN;
  if (ws_bytes < fwd_ws_bytes(M, K)) return FP8MOE_EWORKSPACE;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  uint8_t* q = static_cast<uint8_t*>(ws);
  float* sx = reinterpret_cast<float*>(q + round_up((size_t)M * (size_t)K, 256));
  GmmFwdArgs a;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)K};
    const uint32_t box[2] = {128, 128};
    rc = make_tmap(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)E};
    const uint64_t st[2] = {(uint64_t)N, (uint64_t)N * (uint64_t)K};
    const uint32_t box[3] = {128, 128, 1};
    rc = make_tmap(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, codes, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  a.sx = sx;
  a.scale = scale;
  a.gs = gs;
  a.out = out;
  a.M = M;
  a.K = (int)K;
  a.N = (int)N;
  a.E = E;
  a.swiglu = swiglu;
  cudaError_t e = fp8moe_launch_quantize_rows(lhs, M, (int)K, gs, E, 0, E, q, sx, sms, 8, 1,
                                              stream);
  if (e != cudaSuccess) return cuda_fail(e);
  a.e0 = 0;
  a.e1 = E;
  a.blk = 0;
  e = fp8moe_launch_gmm_fp8_fwd(a, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

// gu != nullptr selects the dSwiGLU epilogue: dlhs is then dgu [M, 2K].
int dlhs_impl(const void* dout, int64_t M, int64_t N, const uint8_t* codes, const float* scale,
              int32_t E, int64_t K, const int32_t* gs, const void* gu, void* dlhs, int path,
              cudaStream_t stream) {
  int rc = check_common(M, K, N, E);
  if (rc) return rc;
  if (path == 1 && N > 256) return FP8MOE_EINVAL;
  if (M == 0) return FP8MOE_OK;
  if (!dout || !codes || !scale || !gs || !dlhs) return FP8MOE_EINVAL;
  if (!aligned16(dout) || !aligned16(codes) || !aligned16(scale) || !aligned16(dlhs) ||
      (gu && !aligned16(gu)) || (reinterpret_cast<uintptr_t>(gs) & 3u))
    return FP8MOE_EALIGN;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  GmmDlhsArgs a;
  a.gu = gu;
  {
    const uint64_t dims[2] = {(uint64_t)N, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)N * 2};
    const uint32_t box[2] = {64, 128};
    rc = make_tmap(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dout, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)E};
    const uint64_t st[2] = {(uint64_t)N, (uint64_t)N * (uint64_t)K};
    const uint32_t box[3] = {64, 256, 1};
    rc = make_tmap(&a.tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, codes, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
    // pair path: 128 k rows x 64 bytes, 64-byte swizzle (conflict-free row reads)
    const uint32_t box_p[3] = {64, 128, 1};
    rc = make_tmap(&a.tmCp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, codes, dims, st, box_p,
                   CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc) return rc;
  }
  a.scale = scale;
  a.gs = gs;
  a.dlhs = dlhs;
  a.M = M;
  a.N = (int)N;
  a.K = (int)K;
  a.E = E;
  cudaError_t e = fp8moe_launch_gmm_dlhs(a, sms, path, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int tgmm_quantize_impl(const void* lhs, const void* dout, int64_t M, int64_t K, int64_t N,
                       int32_t E, const int32_t* gs, uint8_t* qx, float* sx, uint8_t* qd,
                       float* sd, cudaStream_t stream, int sms, int d_fmt) {
  cudaError_t e = fp8moe_launch_tgmm_quantize_tiles(lhs, dout, M, (int)K, (int)N, gs, E,
                                                    segment_bound(M, E), qx, sx, qd, sd, sms, 1,
                                                    d_fmt, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

}  // namespace

extern "C" {

size_t fp8moe_workspace_size(int op, int64_t M, int64_t K, int64_t N, int32_t E) {
  if (M < 0 || K < 0 || N < 0 || E < 0) return 0;
  switch (op) {
    case FP8MOE_OP_GMM_FP8_FWD:
    case FP8MOE_OP_GMM_SILU_FP8_FWD:
      return fwd_ws_bytes(M, K);
    case FP8MOE_OP_TGMM_DRHS_QUANT:
      return tgmm_ws_bytes(M, K, N, E);
    case FP8MOE_OP_GMM_FP8_FWD_BLOCK:
      return fwd_block_ws_bytes(M, K);
    default:
      return 0;
  }
}

int fp8moe_gmm_fp8_fwd(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                       const float* scale, int32_t E, int64_t N, const int32_t* group_sizes,
                       void* out, void* workspace, size_t workspace_bytes,
                       fp8moe_stream_t stream) {
  return gmm_fp8_fwd_impl(lhs, M, K, codes, scale, E, N, group_sizes, out, workspace,
                          workspace_bytes, stream, 0);
}

int fp8moe_gmm_silu_fp8_fwd(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                            const float* scale, int32_t E, int64_t N,
                            const int32_t* group_sizes, void* out, void* workspace,
                            size_t workspace_bytes, fp8moe_stream_t stream) {
  return gmm_fp8_fwd_impl(lhs, M, K, codes, scale, E, N, group_sizes, out, workspace,
                          workspace_bytes, stream, 1);
}

int fp8moe_gmm_dlhs_fp8(const void* dout, int64_t M, int64_t N, const uint8_t* codes,
                        const float* scale, int32_t E, int64_t K, const int32_t* group_sizes,
                        void* dlhs, void* workspace, size_t workspace_bytes,
                        fp8moe_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  // the on-chip cache path when the whole contraction fits one cached block,
  // otherwise CTA pairs with the dequantized weight in tensor memory
  const int path = (N <= 256) ? 1 : 2;
  return dlhs_impl(dout, M, N, codes, scale, E, K, group_sizes, nullptr, dlhs, path, stream);
}

int fp8moe_gmm_dlhs_fp8_path(const void* dout, int64_t M, int64_t N, const uint8_t* codes,
                             const float* scale, int32_t E, int64_t K,
                             const int32_t* group_sizes, void* dlhs, int32_t path,
                             fp8moe_stream_t stream) {
  if (path < 0 || path > 2) return FP8MOE_EINVAL;
  return dlhs_impl(dout, M, N, codes, scale, E, K, group_sizes, nullptr, dlhs, path, stream);
}

int fp8moe_gmm_dlhs_dswiglu_fp8(const void* dout, int64_t M, int64_t N, const uint8_t* codes,
                                const float* scale, int32_t E, int64_t F, const void* gu,
                                const int32_t* group_sizes, void* dgu, void* workspace,
                                size_t workspace_bytes, fp8moe_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (M > 0 && !gu) return FP8MOE_EINVAL;
  // the pair path has one accumulator and must hold it through the SwiGLU
  // backward, which stalls its MMAs; the streaming path is the faster one here
  const int path = (N <= 256) ? 1 : 0;
  return dlhs_impl(dout, M, N, codes, scale, E, F, group_sizes, gu, dgu, path, stream);
}

int fp8moe_gmm_dlhs_dswiglu_fp8_path(const void* dout, int64_t M, int64_t N, const uint8_t* codes,
                                     const float* scale, int32_t E, int64_t F, const void* gu,
                                     const int32_t* group_sizes, void* dgu, int32_t path,
                                     fp8moe_stream_t stream) {
  if (path < 0 || path > 2) return FP8MOE_EINVAL;
  if (M > 0 && !gu) return FP8MOE_EINVAL;
  return dlhs_impl(dout, M, N, codes, scale, E, F, group_sizes, gu, dgu, path, stream);
}

static int tgmm_drhs_impl(const void* lhs, const void* dout, int64_t M, int64_t K, int64_t N,
                          int32_t E, const int32_t* group_sizes, float* dW, void* workspace,
                          size_t workspace_bytes, int d_fmt, fp8moe_stream_t stream) {
  int rc = check_common(M, K, N, E);
  if (rc) return rc;
  if (d_fmt != FP8MOE_FMT_E4M3 && d_fmt != FP8MOE_FMT_E5M2) return FP8MOE_EINVAL;
  if (!dW || !group_sizes) return FP8MOE_EINVAL;
  if (M > 0 && (!lhs || !dout)) return FP8MOE_EINVAL;
  if (!workspace) return FP8MOE_EWORKSPACE;
  if (!aligned16(lhs) || !aligned16(dout) || !aligned16(dW) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
    return FP8MOE_EALIGN;
  if (workspace_bytes < tgmm_ws_bytes(M, K, N, E)) return FP8MOE_EWORKSPACE;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  TgmmWorkspace w = carve_tgmm(workspace, M, K, N, E);
  const int64_t S = segment_bound(M, E);
  if (M > 0) {
    rc = tgmm_quantize_impl(lhs, dout, M, K, N, E, group_sizes, w.qx, w.sx, w.qd, w.sd, stream, sms,
                            d_fmt);
    if (rc) return rc;
  }
  TgmmArgs a;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)(S * 128)};
    const uint64_t st[1] = {(uint64_t)K};
    const uint32_t box[2] = {128, 128};
    rc = make_tmap(&a.tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, w.qx, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  {
    const uint64_t dims[2] = {(uint64_t)N, (uint64_t)(S * 128)};
    const uint64_t st[1] = {(uint64_t)N};
    const uint32_t box[2] = {128, 128};
    rc = make_tmap(&a.tmD, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, w.qd, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  {
    // dW as [E][K][N] so that a box's rows past K (ragged k tile) are clipped
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)E};
    const uint64_t st[2] = {(uint64_t)N * 4, (uint64_t)K * (uint64_t)N * 4};
    const uint32_t box[3] = {32, 32, 1};
    rc = make_tmap(&a.tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dW, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  a.sx = w.sx;
  a.sd = w.sd;
  a.gs = group_sizes;
  a.dW = dW;
  a.M = M;
  a.K = (int)K;
  a.N = (int)N;
  a.E = E;
  a.d_fmt = d_fmt;
  cudaError_t e = fp8moe_launch_tgmm(a, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int fp8moe_tgmm_drhs_quant(const void* lhs, const void* dout, int64_t M, int64_t K, int64_t N,
                           int32_t E, const int32_t* group_sizes, float* dW, void* workspace,
                           size_t workspace_bytes, fp8moe_stream_t stream) {
  return tgmm_drhs_impl(lhs, dout, M, K, N, E, group_sizes, dW, workspace, workspace_bytes,
                        FP8MOE_FMT_E4M3, stream);
}

int fp8moe_tgmm_drhs_quant_fmt(const void* lhs, const void* dout, int64_t M, int64_t K, int64_t N,
                               int32_t E, const int32_t* group_sizes, float* dW, void* workspace,
                               size_t workspace_bytes, int32_t dout_fmt, fp8moe_stream_t stream) {
  return tgmm_drhs_impl(lhs, dout, M, K, N, E, group_sizes, dW, workspace, workspace_bytes,
                        dout_fmt, stream);
}

int fp8moe_dequantize_fp8_codes(const uint8_t* codes, const float* scale, int32_t E, int64_t K,
                                int64_t N, void* out, fp8moe_stream_t stream) {
  int rc = check_common(0, K, N, E);
  if (rc) return rc;
  if (!codes || !scale || !out) return FP8MOE_EINVAL;
  if (!aligned16(codes) || !aligned16(scale) || !aligned16(out)) return FP8MOE_EALIGN;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  cudaError_t e = fp8moe_launch_dequantize(codes, scale, E, K, N, out, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int fp8moe_gmm_bf16_fwd(const void* lhs, int64_t M, int64_t K, const void* w, int32_t E,
                        int64_t N, const int32_t* group_sizes, int32_t swiglu, void* out,
                        fp8moe_stream_t stream) {
  int rc = check_common(M, K, N, E);
  if (rc) return rc;
  if (M == 0) return FP8MOE_OK;
  if (!lhs || !w || !group_sizes || !out) return FP8MOE_EINVAL;
  if (!aligned16(lhs) || !aligned16(w) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
    return FP8MOE_EALIGN;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  GmmFwdArgs a;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {64, 128};
    rc = make_tmap(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lhs, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)E};
    const uint64_t st[2] = {(uint64_t)N * 2, (uint64_t)N * (uint64_t)K * 2};
    const uint32_t box[3] = {64, 64, 1};
    rc = make_tmap(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  a.sx = nullptr;
  a.scale = nullptr;
  a.gs = group_sizes;
  a.out = out;
  a.M = M;
  a.K = (int)K;
  a.N = (int)N;
  a.E = E;
  a.swiglu = swiglu ? 1 : 0;
  a.e0 = 0;
  a.e1 = E;
  a.blk = 0;
  cudaError_t e = fp8moe_launch_gmm_bf16_fwd(a, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int fp8moe_gmm_fp8_fwd_block(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                             const float* scale, int32_t E, int64_t N,
                             const int32_t* group_sizes, void* out, void* workspace,
                             size_t workspace_bytes, int32_t block, int32_t swiglu,
                             fp8moe_stream_t stream) {
  int rc = check_common(M, K, N, E);
  if (rc) return rc;
  if (block != kQuantBlock || (swiglu != 0 && swiglu != 1)) return FP8MOE_EINVAL;
  if (swiglu && (N % 32 != 0)) return FP8MOE_EALIGN;
  if (M == 0) return FP8MOE_OK;
  if (!workspace) return FP8MOE_EWORKSPACE;
  if (!lhs || !codes || !scale || !group_sizes || !out) return FP8MOE_EINVAL;
  if (!aligned16(lhs) || !aligned16(codes) || !aligned16(scale) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
    return FP8MOE_EALIGN;
  if (workspace_bytes < fwd_block_ws_bytes(M, K)) return FP8MOE_EWORKSPACE;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  uint8_t* q = static_cast<uint8_t*>(workspace);
  float* sb = reinterpret_cast<float*>(q + round_up((size_t)M * (size_t)K, 256));
  cudaError_t e = fp8moe_launch_quantize_rows_block(lhs, M, (int)K, group_sizes, E, q, sb, sms, 1,
                                                    stream);
  if (e != cudaSuccess) return cuda_fail(e);
  GmmFwdArgs a;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)K};
    const uint32_t box[2] = {128, 128};
    rc = make_tmap(&a.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  {
    const uint64_t dims[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)E};
    const uint64_t st[2] = {(uint64_t)N, (uint64_t)N * (uint64_t)K};
    const uint32_t box[3] = {128, 128, 1};
    rc = make_tmap(&a.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, codes, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  a.sx = sb;
  a.scale = scale;
  a.gs = group_sizes;
  a.out = out;
  a.M = M;
  a.K = (int)K;
  a.N = (int)N;
  a.E = E;
  a.swiglu = swiglu;
  a.e0 = 0;
  a.e1 = E;
  a.blk = 1;
  e = fp8moe_launch_gmm_fp8_fwd(a, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int fp8moe_quantize_rows_block(const void* lhs, int64_t M, int64_t K, const int32_t* group_sizes,
                               int32_t E, int32_t block, uint8_t* q, float* sb,
                               fp8moe_stream_t stream) {
  int rc = check_common(M, K, 16, E);
  if (rc) return rc;
  if (block != kQuantBlock) return FP8MOE_EINVAL;
  if (M == 0) return FP8MOE_OK;
  if (!lhs || !group_sizes || !q || !sb) return FP8MOE_EINVAL;
  if (!aligned16(lhs) || !aligned16(q) || (reinterpret_cast<uintptr_t>(sb) & 3u) ||
      (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
    return FP8MOE_EALIGN;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  cudaError_t e = fp8moe_launch_quantize_rows_block(lhs, M, (int)K, group_sizes, E, q, sb, sms, 1,
                                                    stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int fp8moe_quantize_rows(const void* lhs, int64_t M, int64_t K, const int32_t* group_sizes,
                         int32_t E, uint8_t* q, float* sx, fp8moe_stream_t stream) {
  int rc = check_common(M, K, 16, E);
  if (rc) return rc;
  if (M == 0) return FP8MOE_OK;
  if (!lhs || !group_sizes || !q || !sx) return FP8MOE_EINVAL;
  if (!aligned16(lhs) || !aligned16(q) || (reinterpret_cast<uintptr_t>(sx) & 3u) ||
      (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
    return FP8MOE_EALIGN;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  cudaError_t e = fp8moe_launch_quantize_rows(lhs, M, (int)K, group_sizes, E, 0, E, q, sx, sms, 8,
                                              1, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int fp8moe_tgmm_quantize_tiles(const void* lhs, const void* dout, int64_t M, int64_t K,
                               int64_t N, int32_t E, const int32_t* group_sizes, uint8_t* qx,
                               float* sx, uint8_t* qd, float* sd, fp8moe_stream_t stream) {
  return fp8moe_tgmm_quantize_tiles_fmt(lhs, dout, M, K, N, E, group_sizes, qx, sx, qd, sd,
                                        FP8MOE_FMT_E4M3, stream);
}

int fp8moe_tgmm_quantize_tiles_fmt(const void* lhs, const void* dout, int64_t M, int64_t K,
                                   int64_t N, int32_t E, const int32_t* group_sizes, uint8_t* qx,
                                   float* sx, uint8_t* qd, float* sd, int32_t dout_fmt,
                                   fp8moe_stream_t stream) {
  int rc = check_common(M, K, N, E);
  if (rc) return rc;
  if (dout_fmt != FP8MOE_FMT_E4M3 && dout_fmt != FP8MOE_FMT_E5M2) return FP8MOE_EINVAL;
  if (M == 0) return FP8MOE_OK;
  if (!lhs || !dout || !group_sizes || !qx || !sx || !qd || !sd) return FP8MOE_EINVAL;
  if (!aligned16(lhs) || !aligned16(dout) || !aligned16(qx) || !aligned16(qd) ||
      !aligned16(sx) || !aligned16(sd) || (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
    return FP8MOE_EALIGN;
  int sms = 0;
  rc = device_init(&sms);
  if (rc) return rc;
  return tgmm_quantize_impl(lhs, dout, M, K, N, E, group_sizes, qx, sx, qd, sd, stream, sms,
                            dout_fmt);
}

int fp8moe_selftest_wait_timeout(uint32_t limit_us, fp8moe_stream_t stream) {
  if (limit_us == 0 || limit_us > 2000000u) return FP8MOE_EINVAL;
  int sms = 0;
  int rc = device_init(&sms);
  if (rc) return rc;
  cudaError_t e = fp8moe_launch_selftest_wait((uint64_t)limit_us * 1000u, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int fp8moe_selftest_cast_f32(const float* x, int64_t n, int32_t fmt, uint8_t* codes,
                             fp8moe_stream_t stream) {
  if (n < 0 || (fmt != FP8MOE_FMT_E4M3 && fmt != FP8MOE_FMT_E5M2)) return FP8MOE_EINVAL;
  if (n == 0) return FP8MOE_OK;
  if (!x || !codes) return FP8MOE_EINVAL;
  if (reinterpret_cast<uintptr_t>(x) & 3u) return FP8MOE_EALIGN;
  int sms = 0;
  int rc = device_init(&sms);
  if (rc) return rc;
  cudaError_t e = fp8moe_launch_selftest_cast(x, n, fmt, codes, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FP8MOE_OK;
}

int fp8moe_read_status(fp8moe_stream_t stream, uint32_t* flags) {
  if (!flags) return FP8MOE_EINVAL;
  uint32_t v = 0;
  uint32_t (*takes[])(cudaStream_t) = {fp8moe_status_take_quant, fp8moe_status_take_dequant,
                                       fp8moe_status_take_gmm_fwd, fp8moe_status_take_dlhs,
                                       fp8moe_status_take_dlhs_pair, fp8moe_status_take_tgmm,
                                       fp8moe_status_take_selftest};
  for (auto take : takes) {
    uint32_t x = take(stream);
    if (x == 0xFFFFFFFFu) return cuda_fail(cudaGetLastError());
    v |= x;
  }
  *flags = v;
  return FP8MOE_OK;
}

const char* fp8moe_status_string(int code) {
  switch (code) {
    case FP8MOE_OK: return "ok";
    case FP8MOE_EINVAL: return "invalid argument";
    case FP8MOE_EALIGN: return "misaligned pointer or dimension (16-byte rule)";
    case FP8MOE_EWORKSPACE: return "workspace missing or too small";
    case FP8MOE_ECUDA: return "CUDA error (see fp8moe_last_cuda_error)";
    case FP8MOE_EUNSUPPORTED: return "device is not sm_103";
    default: return "unknown status";
  }
}

int fp8moe_last_cuda_error(void) { return t_last_cuda_error; }

void fp8moe_internal_set_cuda_error(int e) { t_last_cuda_error = e; }

// The forward's argument checks that come before its workspace check, in the
// same order and with the same codes (for callers that supply the workspace
// themselves). FP8MOE_OK with *empty = 1: M == 0, nothing to do.
int fp8moe_internal_check_fwd_args(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                                   const float* scale, int32_t E, int64_t N, const int32_t* gs,
                                   const void* out, int swiglu, int* empty) {
  *empty = 0;
  int rc = check_common(M, K, N, E);
  if (rc) return rc;
  if (swiglu && (N % 32 != 0)) return FP8MOE_EALIGN;
  if (M == 0) {
    *empty = 1;
    return FP8MOE_OK;
  }
  if (!lhs || !codes || !scale || !gs || !out) return FP8MOE_EINVAL;
  if (!aligned16(lhs) || !aligned16(codes) || !aligned16(scale) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(gs) & 3u))
    return FP8MOE_EALIGN;
  return FP8MOE_OK;
}

int fp8moe_num_sms(void) {
  int sms = 0;
  if (device_init(&sms) != FP8MOE_OK) return 0;
  return sms;
}

}  // extern "C"
