// tgmm.cu -- weight-gradient grouped matmul over in-kernel quantized operands.
//
//   dW[e, k, n] = sum over the segments q of expert e of
//                 sx[q, k] * sd[q, n] * sum_{rows m of q} qx[m, k] * qd[m, n]
//
// "MoE fp8 backward: in-kernel drhs operand quantization", What: the drhs tgmm
// quantizes both operands per gm tile and per channel inside the kernel and
// touches only the tiles that group_sizes covers, so no reduction ever reads
// the tail of a dropless buffer. Segments are the global 128-row tiles
// intersected with each group; tgmm_quantize_tiles_kernel (quant.cu) wrote each
// segment's codes to a 128-row slot with the rows outside the segment zeroed
// and the per-channel scales next to it. This kernel never looks at a buffer
// row: it reads slots only.
//
// Design (one CTA per SM, persistent). Work unit = (expert, 128-wide k tile,
// 256-wide n tile); n tiles of one k tile are adjacent so the A slots are
// shared through L2.
//   warp 0      TMA: qx slot [128 rows x 128 k] and qd slot [128 rows x 128 n],
//               both row-major = MN-major operands, 128-byte swizzle; and the
//               segment's 128 + 128 channel scales by bulk copy into a scale
//               ring that the rescale warps release.
//   warp 1      tcgen05.mma kind::f8f6f4, M=128 (k), N=128 (n), K=32 rows, four
//               per segment, into one of two TMEM partial buffers.
//   warps 2..17 rescale: each thread owns one k row and 32 n columns of the
//               f32 accumulator in registers, acc += (sx * sd[n]) * P[n]; the
//               partial products sit in four TMEM buffers so the MMA runs up
//               to four segments ahead. At the end of the unit the accumulator
//               goes to dW through a per-warp shared-memory transpose
//               (128-byte coalesced stores).
// The 128-wide n tile and four rescale warps per SM sub-partition keep the
// accumulator in registers (Blackwell budgets registers per group of four warps)
// and give the rescale enough warps to hide the TMEM and shared-memory latency.
// The dout operand's codes may be e5m2 (the configurable gradient dtype of the
// same page); the MMA then reads B as e5m2 (kind::f8f6f4 takes mixed fp8 types).
// An expert without rows writes zeros.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace fp8moe {
namespace tg {

constexpr int kBK = 128;     // k per tile (MMA M)
constexpr int kBN = 128;     // n per tile (MMA N)
constexpr int kStages = 4;
constexpr int kXBytes = 128 * 128;
constexpr int kDBytes = 128 * 128;
constexpr int kStageBytes = kXBytes + kDBytes;    // 32 KB
constexpr int kEpiWarps = 16;                     // 4 per TMEM lane quarter
constexpr int kCols = kBN * 4 / kEpiWarps;        // 32 accumulator columns per thread
constexpr int kTBufs = 4;                         // TMEM partial buffers of kBN columns
constexpr int kThreads = (2 + kEpiWarps) * 32;    // 576
constexpr int kTmemCols = 512;
constexpr int kXpose = 32 * 32 * 4;               // per-warp transpose buffer
constexpr int kSRing = 16;                        // scale ring slots (1 KB each)

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[kTBufs];
  uint64_t tempty[kTBufs];
  uint64_t sfull[kSRing];
  uint64_t sempty[kSRing];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t T;
  int32_t total_units;
  alignas(16) float sring[kSRing][2][128];   // [slot][0: sx over k, 1: sd over n]
  int32_t begin[kMaxExperts];
  int32_t end[kMaxExperts];
  int32_t segbase[kMaxExperts + 1];
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kEpiWarps * kXpose + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");

__global__ void __launch_bounds__(kThreads, 1)
tgmm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmD,
            const float* __restrict__ sx, const float* __restrict__ sd,
            const int32_t* __restrict__ gs, float* __restrict__ dW, int64_t M, int K, int N, int E,
            int d_fmt) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  float* xpose = reinterpret_cast<float*>(tiles + (size_t)kStages * kStageBytes);
  Smem& s = *reinterpret_cast<Smem*>(tiles + (size_t)kStages * kStageBytes + kEpiWarps * kXpose);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkt = (K + kBK - 1) / kBK, nnt = (N + kBN - 1) / kBN;
  const int units_per_e = nkt * nnt;

  if (warp == 0) {
    load_groups_warp0(gs, E, M, s.begin, s.end, &s.T, blockIdx.x == 0);
    __syncwarp();
    int32_t carry = 0;
    for (int base = 0; base < E; base += 32) {
      int e = base + lane;
      int32_t n = 0;
      if (e < E && s.end[e] > s.begin[e]) n = (s.end[e] - 1) / 128 - s.begin[e] / 128 + 1;
      int32_t incl = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      if (e < E) s.segbase[e] = carry + incl - n;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s.segbase[E] = carry;
      s.total_units = E * units_per_e;
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmD);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(&s.full[i], 1);
        mbar_init(&s.empty[i], 1);
      }
      // released by one elected lane per rescale warp
      for (int i = 0; i < kTBufs; ++i) {
        mbar_init(&s.tfull[i], 1);
        mbar_init(&s.tempty[i], kEpiWarps);
      }
      for (int i = 0; i < kSRing; ++i) {
        mbar_init(&s.sfull[i], 1);
        mbar_init(&s.sempty[i], kEpiWarps);
      }
      mbar_init(&s.drain, 1);
      fence_mbar_init();
    }
    __syncwarp();
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const int total = s.total_units;
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const int e = u / units_per_e, rem = u - e * units_per_e;
        const int kt = rem / nnt, ntile = rem - kt * nnt;
        const int q0 = s.segbase[e], q1 = s.segbase[e + 1];
        // K, N % 16 == 0: the valid part of a 128-wide scale row is a multiple
        // of 64 bytes, so both bulk copies keep 16-byte alignment and size.
        const uint32_t kbytes = (uint32_t)min(kBK, K - kt * kBK) * 4u;
        const uint32_t nbytes = (uint32_t)min(kBN, N - ntile * kBN) * 4u;
        for (int q = q0; q < q1; ++q) {
          if (!mbar_wait(&s.empty[st], ph ^ 1, kWhereProducer)) { ok = false; break; }
          const int ss = (int)(issued % kSRing);
          if (!mbar_wait(&s.sempty[ss], (uint32_t)(((issued / kSRing) & 1) ^ 1), kWhereProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.full[st], kStageBytes);
          uint8_t* a = tiles + st * kStageBytes;
          tma_load_2d(a, &tmX, &s.full[st], kt * kBK, q * 128);
          tma_load_2d(a + kXBytes, &tmD, &s.full[st], ntile * kBN, q * 128);
          mbar_arrive_expect_tx(&s.sfull[ss], kbytes + nbytes);
          bulk_load(s.sring[ss][0], sx + (int64_t)q * K + kt * kBK, kbytes, &s.sfull[ss]);
          bulk_load(s.sring[ss][1], sd + (int64_t)q * N + ntile * kBN, nbytes, &s.sfull[ss]);
          ++issued;
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
      }
      int64_t n_last = issued < kStages ? issued : kStages;
      for (int64_t i = 1; i <= n_last; ++i) {
        int64_t idx = issued - i;
        mbar_wait(&s.full[idx % kStages], (uint32_t)((idx / kStages) & 1), kWhereDrain);
      }
      n_last = issued < kSRing ? issued : kSRing;
      for (int64_t i = 1; i <= n_last; ++i) {
        int64_t idx = issued - i;
        mbar_wait(&s.sfull[idx % kSRing], (uint32_t)((idx / kSRing) & 1), kWhereDrain);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // A = qx slot, [K_mma = 128 rows][M_mma = 128 k] -> MN-major, one atom;
      // B = qd slot, [K_mma = 128 rows][N_mma = 128 n] -> MN-major, one atom.
      // B (qd) is e5m2 when the gradient dtype is e5m2; A (qx) is always e4m3
      const uint32_t idesc = make_idesc(0, d_fmt == 1 ? 1u : 0u, 1, 1, kBK, kBN);
      int st = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const int e = u / units_per_e;
        const int q0 = s.segbase[e], q1 = s.segbase[e + 1];
        for (int q = q0; q < q1; ++q) {
          if (!mbar_wait(&s.tempty[acc], aph ^ 1, kWhereMma)) { ok = false; break; }
          if (!mbar_wait(&s.full[st], ph, kWhereMma)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(acc * kBN);
          const uint32_t a_addr = smem_u32(tiles + st * kStageBytes);
          const uint32_t b_addr = a_addr + kXBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = make_desc(a_addr + kk * 4096, 16384, 1024, kSwizzle128B);
            const uint64_t bd = make_desc(b_addr + kk * 4096, 16384, 1024, kSwizzle128B);
            mma_f8f6f4(d, ad, bd, idesc, kk != 0);
          }
          mma_commit(&s.empty[st]);
          mma_commit(&s.tfull[acc]);
          if (++st == kStages) { st = 0; ph ^= 1; }
          if (++acc == kTBufs) { acc = 0; aph ^= 1; }
        }
      }
      mma_commit(&s.drain);
      mbar_wait(&s.drain, 0, kWhereDrain);
    }
  } else {
    // ============================ rescale + store ===========================
    const int ew = warp - 2;                 // 0..15
    const int quarter = warp & 3;            // TMEM lanes 32*quarter ..
    const int cg = ew >> 2;                  // columns [kCols*cg, kCols*cg + kCols)
    const int r = quarter * 32 + lane;       // k row inside the tile
    float* xp = xpose + ew * (kXpose / 4);
    int acc = 0;
    uint32_t aph = 0;
    int64_t used = 0;                        // scale ring position
    bool failed = false;
    for (int u = blockIdx.x; u < total && !failed; u += gridDim.x) {
      const int e = u / units_per_e, rem = u - e * units_per_e;
      const int kt = rem / nnt, ntile = rem - kt * nnt;
      const int q0 = s.segbase[e], q1 = s.segbase[e + 1];
      float a[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) a[i] = 0.0f;
      for (int q = q0; q < q1; ++q) {
        const int ss = (int)(used % kSRing);
        if (!mbar_wait_warp(&s.sfull[ss], (uint32_t)((used / kSRing) & 1), kWhereEpilogue) ||
            !mbar_wait_warp(&s.tfull[acc], aph, kWhereEpilogue)) {
          failed = true;
          break;
        }
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN + cg * kCols), v);
        const float sxk = s.sring[ss][0][r];
        const float4* sdv = reinterpret_cast<const float4*>(&s.sring[ss][1][cg * kCols]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.tempty[acc]);   // TMEM buffer free once in registers
#pragma unroll
        for (int i = 0; i < kCols / 4; ++i) {
          const float4 d4 = sdv[i];
          a[4 * i] = __fmaf_rn(__fmul_rn(sxk, d4.x), __uint_as_float(v[4 * i]), a[4 * i]);
          a[4 * i + 1] = __fmaf_rn(__fmul_rn(sxk, d4.y), __uint_as_float(v[4 * i + 1]), a[4 * i + 1]);
          a[4 * i + 2] = __fmaf_rn(__fmul_rn(sxk, d4.z), __uint_as_float(v[4 * i + 2]), a[4 * i + 2]);
          a[4 * i + 3] = __fmaf_rn(__fmul_rn(sxk, d4.w), __uint_as_float(v[4 * i + 3]), a[4 * i + 3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sempty[ss]);
        ++used;
        if (++acc == kTBufs) { acc = 0; aph ^= 1; }
      }
      if (failed) break;
      // store the [32 k rows x 32 n] block through the per-warp transpose buffer
      // (16-byte chunk c4 of row i stored at chunk c4 ^ (i & 7)).
      const int k_warp0 = kt * kBK + quarter * 32;
      const int n_cg0 = ntile * kBN + cg * kCols;
      __syncwarp();
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const int pc = c4 ^ (lane & 7);
        *reinterpret_cast<float4*>(xp + lane * 32 + pc * 4) =
            make_float4(a[c4 * 4], a[c4 * 4 + 1], a[c4 * 4 + 2], a[c4 * 4 + 3]);
      }
      __syncwarp();
#pragma unroll 1
      for (int it = 0; it < 8; ++it) {
        const int i = it * 4 + (lane >> 3);       // row within the 32-row block
        const int c4 = lane & 7;
        const float4 v = *reinterpret_cast<const float4*>(xp + i * 32 + ((c4 ^ (i & 7)) * 4));
        const int kk = k_warp0 + i;
        const int nn = n_cg0 + c4 * 4;
        if (kk < K && nn < N)   // N % 16 == 0: a 4-column group is all in or all out
          *reinterpret_cast<float4*>(dW + ((int64_t)e * K + kk) * N + nn) = v;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tg
}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_tgmm)

cudaError_t fp8moe_launch_tgmm(const TgmmArgs& a, int num_sms, cudaStream_t s) {
  using namespace fp8moe::tg;
  cudaError_t err = cudaFuncSetAttribute(tgmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  tgmm_kernel<<<num_sms, kThreads, kSmemBytes, s>>>(a.tmX, a.tmD, a.sx, a.sd, a.gs, a.dW, a.M,
                                                    a.K, a.N, a.E, a.d_fmt);
  return cudaGetLastError();
}
