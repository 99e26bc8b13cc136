// quant.cu -- activation quantization kernels.
//
//  * quantize_rows_kernel: the forward GMM's A operand. One f32 absmax scale per
//    row over the whole K, scale = max(amax, 1e-12) / 448, codes = e4m3(x / scale)
//    ("MoE: native FP8 QAT for routed-expert GMMs", Description and
//    Implementation: in-kernel full-K activation quantization with an f32 scale).
//    One CTA per row, the row held in registers between the amax pass and the
//    cast pass; rows at or past T = sum(group_sizes) are never read.
//
//  * tgmm_quantize_tiles_kernel: the weight-gradient operands, per 128-row tile
//    (the dout operand optionally e5m2, the configurable gradient dtype of
//    "MoE fp8 backward: in-kernel drhs operand quantization", What: scale =
//    max(amax, 1e-12) / 57344, codes = e5m2(x / scale))
//    and per channel, over the rows of one group only ("MoE fp8 backward:
//    in-kernel drhs operand quantization", What). Codes go to 128-row slots, one
//    per (tile, group) segment, rows outside the segment zeroed, so the
//    contraction kernel can TMA whole slots without masking.
//
// Both produce exactly the codes of RN_fp8(RN_f32(x / scale)) (see quotient_x2:
// two reciprocal multiplies that bracket the quotient, with the IEEE division
// taken when their codes differ) cast with cvt.rn.satfinite, so codes and
// scales are bit-exact with a plain f32 reading of the definition. The scale
// itself is always an IEEE division.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "groups.cuh"
#include "kernels.h"
#include "quantize.cuh"

namespace fp8moe {

// ------------------------------------------------------------------------ a1
// One CTA of 256 threads per row (grid-stride over rows): each thread holds CPT
// 16-byte chunks of the row in registers, the row amax is reduced across the
// CTA, then every thread casts its own chunks. Few registers per thread keep
// many rows in flight per SM, which is what an HBM-bound pass needs.
constexpr int kQThreads = 256;

// Rows of at most 2048 columns: a warp per row, the row in the registers of its
// 32 lanes, so the amax needs only shuffles (no block barrier) and dozens of rows
// per SM are in flight. Same arithmetic as quantize_rows_kernel.
template <int CPL>
__global__ void __launch_bounds__(kQThreads) quantize_rows_warp_kernel(
    const __nv_bfloat16* __restrict__ lhs, int64_t M, int K, const int32_t* __restrict__ gs,
    int E, int e0, int e1, uint8_t* __restrict__ q, float* __restrict__ sx, int report) {
  __shared__ int32_t s_lo, s_hi;
  group_row_range_warp0(gs, E, M, e0, e1, &s_lo, &s_hi, report && blockIdx.x == 0);
  __syncthreads();
  const int64_t lo = s_lo, T = s_hi;   // rows [lo, T) of experts [e0, e1)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = K >> 3;           // K % 8 == 0
  constexpr int kWarps = kQThreads / 32;
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  for (int64_t m = lo + (int64_t)blockIdx.x * kWarps + warp; m < T; m += stride) {
    const uint4* row = reinterpret_cast<const uint4*>(lhs + m * K);
    uint4 v[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      v[i] = c < nchunk ? __ldg(row + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t amax2 = 0;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      amax2 = bf16x2_absmax(amax2, v[i].x);
      amax2 = bf16x2_absmax(amax2, v[i].y);
      amax2 = bf16x2_absmax(amax2, v[i].z);
      amax2 = bf16x2_absmax(amax2, v[i].w);
    }
    float amax = bf16x2_hmax_to_f32(amax2);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float s = __fdiv_rn(fmaxf(amax, kEps), kE4m3Max);
    float rl, rh;
    bracket(s, rl, rh);
    uint2* qrow = reinterpret_cast<uint2*>(q + m * K);
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int c = lane + 32 * i;
      if (c < nchunk) qrow[c] = quant8(v[i], s, rl, rh);
    }
    if (lane == 0) sx[m] = s;
  }
}

template <int CPT>
__global__ void __launch_bounds__(kQThreads) quantize_rows_kernel(
    const __nv_bfloat16* __restrict__ lhs, int64_t M, int K, const int32_t* __restrict__ gs,
    int E, int e0, int e1, uint8_t* __restrict__ q, float* __restrict__ sx, int report) {
  __shared__ int32_t s_lo, s_hi;
  __shared__ float s_red[2][kQThreads / 32];
  group_row_range_warp0(gs, E, M, e0, e1, &s_lo, &s_hi, report && blockIdx.x == 0);
  __syncthreads();
  const int64_t lo = s_lo, T = s_hi;   // rows [lo, T) of experts [e0, e1)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = K >> 3;   // K % 8 == 0
  int buf = 0;
  // The next row's loads are issued before this row's cast, so the HBM latency
  // of one row overlaps the arithmetic of the previous one.
  uint4 nxt[CPT];
#pragma unroll
  for (int i = 0; i < CPT; ++i) nxt[i] = make_uint4(0u, 0u, 0u, 0u);
  if (lo + blockIdx.x < T) {
    const uint4* row = reinterpret_cast<const uint4*>(lhs + (lo + blockIdx.x) * K);
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = threadIdx.x + kQThreads * i;
      if (c < nchunk) nxt[i] = __ldg(row + c);
    }
  }
  for (int64_t m = lo + blockIdx.x; m < T; m += gridDim.x) {
    uint4 v[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) v[i] = nxt[i];
    if (m + gridDim.x < T) {
      const uint4* row = reinterpret_cast<const uint4*>(lhs + (m + gridDim.x) * K);
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = threadIdx.x + kQThreads * i;
        if (c < nchunk) nxt[i] = __ldg(row + c);
      }
    }
    uint32_t amax2 = 0;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = threadIdx.x + kQThreads * i;
      if (c < nchunk) {
        amax2 = bf16x2_absmax(amax2, v[i].x);
        amax2 = bf16x2_absmax(amax2, v[i].y);
        amax2 = bf16x2_absmax(amax2, v[i].z);
        amax2 = bf16x2_absmax(amax2, v[i].w);
      }
    }
    float amax = bf16x2_hmax_to_f32(amax2);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if (lane == 0) s_red[buf][warp] = amax;
    __syncthreads();
    amax = s_red[buf][0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_red[buf][w]);
    buf ^= 1;   // the next row reduces into the other buffer: no second barrier needed
    const float s = __fdiv_rn(fmaxf(amax, kEps), kE4m3Max);
    float rl, rh;
    bracket(s, rl, rh);
    uint2* qrow = reinterpret_cast<uint2*>(q + m * K);
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int c = threadIdx.x + kQThreads * i;
      if (c < nchunk) qrow[c] = quant8(v[i], s, rl, rh);
    }
    if (threadIdx.x == 0) sx[m] = s;
  }
}

// Rows longer than the register cache (K > 8192): the cast pass re-reads the
// row (L2 hit).
__global__ void __launch_bounds__(kQThreads) quantize_rows_stream_kernel(
    const __nv_bfloat16* __restrict__ lhs, int64_t M, int K, const int32_t* __restrict__ gs,
    int E, int e0, int e1, uint8_t* __restrict__ q, float* __restrict__ sx, int report) {
  __shared__ int32_t s_lo, s_hi;
  __shared__ float s_red[2][kQThreads / 32];
  group_row_range_warp0(gs, E, M, e0, e1, &s_lo, &s_hi, report && blockIdx.x == 0);
  __syncthreads();
  const int64_t lo = s_lo, T = s_hi;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = K >> 3;
  int buf = 0;
  for (int64_t m = lo + blockIdx.x; m < T; m += gridDim.x) {
    const uint4* row = reinterpret_cast<const uint4*>(lhs + m * K);
    uint32_t amax2 = 0;
    for (int c = threadIdx.x; c < nchunk; c += kQThreads) {
      uint4 v = __ldg(row + c);
      amax2 = bf16x2_absmax(amax2, v.x);
      amax2 = bf16x2_absmax(amax2, v.y);
      amax2 = bf16x2_absmax(amax2, v.z);
      amax2 = bf16x2_absmax(amax2, v.w);
    }
    float amax = bf16x2_hmax_to_f32(amax2);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if (lane == 0) s_red[buf][warp] = amax;
    __syncthreads();
    amax = s_red[buf][0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_red[buf][w]);
    buf ^= 1;
    const float s = __fdiv_rn(fmaxf(amax, kEps), kE4m3Max);
    uint2* qrow = reinterpret_cast<uint2*>(q + m * K);
    float rl, rh;
    bracket(s, rl, rh);
    for (int c = threadIdx.x; c < nchunk; c += kQThreads) qrow[c] = quant8(__ldg(row + c), s, rl, rh);
    if (threadIdx.x == 0) sx[m] = s;
  }
}

// ------------------------------------------- per-512-column block quantization
// The ops-level option of "MoE: native FP8 QAT for routed-expert GMMs"
// (Implementation, lhs_quant_block_size = 512): one bf16 scale per row and
// 512-column block, s = bf16(max(amax over the block, 1e-12) / 448) (IEEE f32
// division, then round to nearest even to bf16), codes = e4m3(x / s). One warp
// per (row, block): 64 16-byte pieces, two per lane; the grid strides over the
// (row, block) pairs of rows < T.
constexpr int kBlockCols = 512;

__global__ void __launch_bounds__(kQThreads) quantize_rows_block_kernel(
    const __nv_bfloat16* __restrict__ lhs, int64_t M, int K, const int32_t* __restrict__ gs,
    int E, uint8_t* __restrict__ q, float* __restrict__ sb, int report) {
  __shared__ int32_t s_lo, s_hi;
  group_row_range_warp0(gs, E, M, 0, E, &s_lo, &s_hi, report && blockIdx.x == 0);
  __syncthreads();
  const int64_t T = s_hi;
  const int lane = threadIdx.x & 31;
  const int nb = (K + kBlockCols - 1) / kBlockCols;
  const int64_t nwarps = (int64_t)gridDim.x * (kQThreads / 32);
  for (int64_t w = (int64_t)blockIdx.x * (kQThreads / 32) + (threadIdx.x >> 5); w < T * nb;
       w += nwarps) {
    const int64_t m = w / nb;
    const int b = (int)(w - m * nb);
    const int k0 = b * kBlockCols;
    const int nchunk = (min(K, k0 + kBlockCols) - k0) >> 3;   // 16-byte pieces, K % 16 == 0
    const uint4* src = reinterpret_cast<const uint4*>(lhs + m * K + k0);
    uint4 v[2];
    uint32_t amax2 = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = lane + 32 * i;
      v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (c < nchunk) {
        v[i] = __ldg(src + c);
        amax2 = bf16x2_absmax(amax2, v[i].x);
        amax2 = bf16x2_absmax(amax2, v[i].y);
        amax2 = bf16x2_absmax(amax2, v[i].z);
        amax2 = bf16x2_absmax(amax2, v[i].w);
      }
    }
    float amax = bf16x2_hmax_to_f32(amax2);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float s = __bfloat162float(__float2bfloat16_rn(__fdiv_rn(fmaxf(amax, kEps), kE4m3Max)));
    float rl, rh;
    bracket(s, rl, rh);
    uint2* dst = reinterpret_cast<uint2*>(q + m * K + k0);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int c = lane + 32 * i;
      if (c < nchunk) dst[c] = quant8(v[i], s, rl, rh);
    }
    if (lane == 0) sb[m * nb + b] = s;
  }
}

// ------------------------------------------------------------------------ a7
// Segment table: nseg[e] = number of 128-row tiles touched by group e, seg_base =
// exclusive prefix (segments numbered expert by expert, tiles ascending).
__device__ __forceinline__ void build_segments_warp0(const int32_t* s_begin, const int32_t* s_end,
                                                     int E, int32_t* s_segbase) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int32_t carry = 0;
  for (int base = 0; base < E; base += 32) {
    int e = base + lane;
    int32_t n = 0;
    if (e < E && s_end[e] > s_begin[e]) n = (s_end[e] - 1) / 128 - s_begin[e] / 128 + 1;
    int32_t incl = n;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    if (e < E) s_segbase[e] = carry + incl - n;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) s_segbase[E] = carry;
}

// Work unit = (segment, 128-column chunk) over the columns of lhs then dout.
// The segment's rows of the chunk are staged once in shared memory by cp.async
// (one HBM read, no staging registers), the per-column amax comes from there,
// then every thread casts its own 16-byte pieces into the zero-padded slot.
// Shared memory is the staged tile plus per-expert bounds sized by E, so that
// several CTAs per SM keep loads in flight while others compute.
constexpr int kTQThreads = 256;
constexpr int kTQMinBlocks = 4;            // CTAs per SM the register budget allows
constexpr int kTQCols = 128;
constexpr int kTQRowBytes = kTQCols * 2;   // 256 B of bf16 per staged row
constexpr size_t kTQTileBytes = 128 * (size_t)kTQRowBytes;      // 32 KB
constexpr int kTQPieces = kTQCols / 8;                         // 16-byte pieces per staged row
constexpr int kTQRowStep = kTQThreads / kTQPieces;              // rows between a thread's rows
constexpr int kTQRowsPer = 128 / kTQRowStep;                    // rows per thread
constexpr size_t kTQPartBytes = (kTQThreads / 32) * kTQPieces * 16;   // per warp and piece: 4 bf16x2 amax
static_assert(kTQPieces <= 32 && kTQRowsPer * kTQRowStep == 128, "tile geometry");
// dynamic shared memory: [tile][part][scale][rl][rh][begin E][end E][segbase E + 1]
__host__ __device__ constexpr size_t tq_smem_bytes(int E) {
  return kTQTileBytes + kTQPartBytes + 3 * kTQCols * 4 + (size_t)(3 * E + 1) * 4;
}

__global__ void __launch_bounds__(kTQThreads, kTQMinBlocks) tgmm_quantize_tiles_kernel(
    const __nv_bfloat16* __restrict__ lhs, const __nv_bfloat16* __restrict__ dout, int64_t M,
    int K, int N, const int32_t* __restrict__ gs, int E, int64_t Smax,
    uint8_t* __restrict__ qx, float* __restrict__ sx, uint8_t* __restrict__ qd,
    float* __restrict__ sd, int report, int d_fmt) {
  extern __shared__ __align__(16) uint8_t tq_smem[];
  uint8_t* s_tile = tq_smem;                                     // [row][128 bf16]
  uint4* s_part = reinterpret_cast<uint4*>(tq_smem + kTQTileBytes);   // [warp][piece]
  float* s_scale = reinterpret_cast<float*>(tq_smem + kTQTileBytes + kTQPartBytes);
  float* s_rl = s_scale + kTQCols;                               // quotient brackets per column
  float* s_rh = s_rl + kTQCols;
  int32_t* s_begin = reinterpret_cast<int32_t*>(s_rh + kTQCols);
  int32_t* s_end = s_begin + E;
  int32_t* s_segbase = s_end + E;
  __shared__ int32_t s_T;
  load_groups_warp0(gs, E, M, s_begin, s_end, &s_T, report && blockIdx.x == 0);
  __syncthreads();
  build_segments_warp0(s_begin, s_end, E, s_segbase);
  __syncthreads();
  const int S = s_segbase[E];
  if (S > Smax) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(kStatusTooManySegments);
    return;
  }
  const int ck = (K + kTQCols - 1) / kTQCols, cn = (N + kTQCols - 1) / kTQCols, cpq = ck + cn;
  const int64_t units = (int64_t)S * cpq;
  const int tid = threadIdx.x;
  const int piece = tid % kTQPieces;  // 16-byte piece (8 columns) of a staged row
  const int prow = tid / kTQPieces;   // first row of this thread, step kTQRowStep
  const int warp = tid >> 5, lane = tid & 31;
  const bool small = units < (int64_t(1) << 31);   // 32-bit unit arithmetic
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int qi = small ? (int)((uint32_t)u / (uint32_t)cpq) : (int)(u / cpq);
    const int ch = (int)(u - (int64_t)qi * cpq);
    const int e = find_bucket(s_segbase, E, qi);
    const int t = s_begin[e] / 128 + (qi - s_segbase[e]);
    const int r0 = max(s_begin[e], t * 128), r1 = min(s_end[e], t * 128 + 128);
    const int lo = r0 - t * 128, hi = r1 - t * 128;            // slot rows of the segment
    const bool is_x = ch < ck;
    const bool e5 = !is_x && d_fmt == 1;                        // e5m2 codes
    const float fmax = e5 ? kE5m2Max : kE4m3Max;
    const int C = is_x ? K : N;
    const int c0 = (is_x ? ch : ch - ck) * kTQCols;
    const int ncols = min(kTQCols, C - c0);                     // multiple of 16
    const __nv_bfloat16* src = is_x ? lhs : dout;
    uint8_t* qo = (is_x ? qx : qd) + (int64_t)qi * 128 * C + c0 + piece * 8;
    float* so = (is_x ? sx : sd) + (int64_t)qi * C;
    const bool pin = piece * 8 < ncols;
    // stage: rows [lo, hi) of the slot, 16 threads per 256-byte row
    if (pin) {
      const __nv_bfloat16* sp = src + (int64_t)(t * 128 + prow) * C + c0 + piece * 8;
#pragma unroll
      for (int i = 0; i < kTQRowsPer; ++i) {
        const int rr = prow + kTQRowStep * i;
        if (rr >= lo && rr < hi)
          cp_async16(s_tile + rr * kTQRowBytes + piece * 16, sp + (int64_t)kTQRowStep * i * C, 16u);
      }
    }
    cp_async_wait_all();
    __syncthreads();
    // column amax over the segment rows (exact): each thread reduces the rows
    // of its 16-byte piece that it casts later, the row sets of a warp meet by
    // shuffle and the warps' partials in shared memory
    {
      uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
      if (pin) {
#pragma unroll
        for (int i = 0; i < kTQRowsPer; ++i) {
          const int rr = prow + kTQRowStep * i;
          if (rr >= lo && rr < hi) {
            const uint4 x = *reinterpret_cast<const uint4*>(s_tile + rr * kTQRowBytes + piece * 16);
            m0 = bf16x2_absmax(m0, x.x);
            m1 = bf16x2_absmax(m1, x.y);
            m2 = bf16x2_absmax(m2, x.z);
            m3 = bf16x2_absmax(m3, x.w);
          }
        }
      }
#pragma unroll
      for (int o = kTQPieces; o < 32; o <<= 1) {
        m0 = bf16x2_absmax(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = bf16x2_absmax(m1, __shfl_xor_sync(0xffffffffu, m1, o));
        m2 = bf16x2_absmax(m2, __shfl_xor_sync(0xffffffffu, m2, o));
        m3 = bf16x2_absmax(m3, __shfl_xor_sync(0xffffffffu, m3, o));
      }
      if (lane < kTQPieces) s_part[warp * kTQPieces + lane] = make_uint4(m0, m1, m2, m3);
    }
    __syncthreads();
    if (tid < kTQCols / 2) {   // column pair tid = word tid % 4 of piece tid / 4
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(s_part) + (tid >> 2) * 4 + (tid & 3);
      uint32_t m2 = 0;
#pragma unroll
      for (int w = 0; w < kTQThreads / 32; ++w) m2 = bf16x2_absmax(m2, pw[w * kTQPieces * 4]);
      const float s0 = __fdiv_rn(fmaxf(bf16lo_to_f32(m2), kEps), fmax);
      const float s1 = __fdiv_rn(fmaxf(bf16hi_to_f32(m2), kEps), fmax);
      s_scale[2 * tid] = s0;
      s_scale[2 * tid + 1] = s1;
      bracket(s0, s_rl[2 * tid], s_rh[2 * tid]);
      bracket(s1, s_rl[2 * tid + 1], s_rh[2 * tid + 1]);
      if (2 * tid < ncols) {
        so[c0 + 2 * tid] = s0;
        so[c0 + 2 * tid + 1] = s1;
      }
    }
    __syncthreads();
    // cast: every slot row is written, rows outside the segment as zeros
    if (pin) {
      float sc[8], rl[8], rh[8];
#pragma unroll
      for (int j = 0; j < 8; j += 4) {
        const float4 a = *reinterpret_cast<const float4*>(s_scale + piece * 8 + j);
        const float4 b = *reinterpret_cast<const float4*>(s_rl + piece * 8 + j);
        const float4 c = *reinterpret_cast<const float4*>(s_rh + piece * 8 + j);
        sc[j] = a.x; sc[j + 1] = a.y; sc[j + 2] = a.z; sc[j + 3] = a.w;
        rl[j] = b.x; rl[j + 1] = b.y; rl[j + 2] = b.z; rl[j + 3] = b.w;
        rh[j] = c.x; rh[j + 1] = c.y; rh[j + 2] = c.z; rh[j + 3] = c.w;
      }
#pragma unroll
      for (int i = 0; i < kTQRowsPer; ++i) {
        const int rr = prow + kTQRowStep * i;
        uint2 o = make_uint2(0u, 0u);
        if (rr >= lo && rr < hi) {
          const uint4 x = *reinterpret_cast<const uint4*>(s_tile + rr * kTQRowBytes + piece * 16);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
          uint16_t c[4];
          if (e5) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              c[j] = quotient_x2<true>(bf16lo_to_f32(w[j]), bf16hi_to_f32(w[j]), sc[2 * j],
                                       sc[2 * j + 1], rl[2 * j], rl[2 * j + 1], rh[2 * j],
                                       rh[2 * j + 1]);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              c[j] = quotient_x2<false>(bf16lo_to_f32(w[j]), bf16hi_to_f32(w[j]), sc[2 * j],
                                        sc[2 * j + 1], rl[2 * j], rl[2 * j + 1], rh[2 * j],
                                        rh[2 * j + 1]);
          }
          o.x = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
          o.y = (uint32_t)c[2] | ((uint32_t)c[3] << 16);
        }
        *reinterpret_cast<uint2*>(qo + (int64_t)rr * C) = o;
      }
    }
    __syncthreads();   // the tile and scales are reused by the next unit
  }
}

}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_quant)

// ------------------------------------------------------------------ launchers
cudaError_t fp8moe_launch_quantize_rows(const void* lhs, int64_t M, int K, const int32_t* gs,
                                        int E, int e0, int e1, uint8_t* q, float* sx, int num_sms,
                                        int ctas_per_sm, int report, cudaStream_t s) {
  using namespace fp8moe;
  // Up to ctas_per_sm row-CTAs resident per SM; the grid strides over the rows.
  int64_t cap = (int64_t)num_sms * ctas_per_sm;
  int grid = (int)(M < cap ? M : cap);
  if (grid < 1) grid = 1;
  const auto* x = static_cast<const __nv_bfloat16*>(lhs);
  const int cpl = (K / 8 + 31) / 32;   // 16-byte chunks per lane of a warp-per-row kernel
  if (cpl <= 8) {
    // a warp per row; one resident wave of CTAs (at most ctas_per_sm per SM)
    // strides over the rows by warps
    auto run = [&](auto kern) -> cudaError_t {
      int per_sm = 0;
      cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kQThreads, 0);
      if (err != cudaSuccess) return err;
      per_sm = per_sm < 1 ? 1 : (per_sm > ctas_per_sm ? ctas_per_sm : per_sm);
      const int64_t need = (M + kQThreads / 32 - 1) / (kQThreads / 32);
      const int64_t wave = (int64_t)num_sms * per_sm;
      const int g = (int)(need < wave ? (need < 1 ? 1 : need) : wave);
      kern<<<g, kQThreads, 0, s>>>(x, M, K, gs, E, e0, e1, q, sx, report);
      return cudaGetLastError();
    };
    if (cpl <= 1) return run(quantize_rows_warp_kernel<1>);
    if (cpl <= 2) return run(quantize_rows_warp_kernel<2>);
    if (cpl <= 4) return run(quantize_rows_warp_kernel<4>);
    return run(quantize_rows_warp_kernel<8>);
  }
  const int cpt = (K / 8 + kQThreads - 1) / kQThreads;
  if (cpt <= 1)
    quantize_rows_kernel<1><<<grid, kQThreads, 0, s>>>(x, M, K, gs, E, e0, e1, q, sx, report);
  else if (cpt <= 2)
    quantize_rows_kernel<2><<<grid, kQThreads, 0, s>>>(x, M, K, gs, E, e0, e1, q, sx, report);
  else if (cpt <= 4)
    quantize_rows_kernel<4><<<grid, kQThreads, 0, s>>>(x, M, K, gs, E, e0, e1, q, sx, report);
  else
    quantize_rows_stream_kernel<<<grid, kQThreads, 0, s>>>(x, M, K, gs, E, e0, e1, q, sx, report);
  return cudaGetLastError();
}

cudaError_t fp8moe_launch_quantize_rows_block(const void* lhs, int64_t M, int K, const int32_t* gs,
                                              int E, uint8_t* q, float* sb, int num_sms, int report,
                                              cudaStream_t s) {
  using namespace fp8moe;
  const int64_t warps = M * ((K + kBlockCols - 1) / kBlockCols);
  const int64_t need = (warps + kQThreads / 32 - 1) / (kQThreads / 32);
  const int64_t cap = (int64_t)num_sms * 8;
  int grid = (int)(need < cap ? need : cap);
  if (grid < 1) grid = 1;
  quantize_rows_block_kernel<<<grid, kQThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(lhs), M,
                                                        K, gs, E, q, sb, report);
  return cudaGetLastError();
}

cudaError_t fp8moe_launch_tgmm_quantize_tiles(const void* lhs, const void* dout, int64_t M, int K,
                                              int N, const int32_t* gs, int E, int64_t Smax,
                                              uint8_t* qx, float* sx, uint8_t* qd, float* sd,
                                              int num_sms, int report, int d_fmt, cudaStream_t s) {
  using namespace fp8moe;
  const size_t smem = tq_smem_bytes(E);   // < 48 KB for any E <= kMaxExperts
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, tgmm_quantize_tiles_kernel, kTQThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int grid = num_sms * per_sm;   // one resident wave, grid-stride over units
  tgmm_quantize_tiles_kernel<<<grid, kTQThreads, smem, s>>>(
      static_cast<const __nv_bfloat16*>(lhs), static_cast<const __nv_bfloat16*>(dout), M, K, N,
      gs, E, Smax, qx, sx, qd, sd, report, d_fmt);
  return cudaGetLastError();
}
