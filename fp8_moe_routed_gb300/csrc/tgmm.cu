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
//   warp 0      lane 0: TMA of the qx slot [128 rows x 128 k] and the qd slot
//               [128 rows x 256 n] (two 128-column boxes), row-major =
//               MN-major operands, 128-byte swizzle. All 32 lanes: the
//               segment's 128 + 256 channel scales by 16-byte cp.async into a
//               scale ring (load/store unit, so the TMA unit only moves tiles).
//   warp 1      tcgen05.mma kind::f8f6f4, M=128 (k), N=256 (n), K=32 rows, four
//               per segment, into one of two TMEM partial buffers.
//   warps 4..19 rescale: each thread owns one k row and 64 n columns of the f32
//               accumulator in registers, acc += (sx * sd[n]) * P[n] in packed
//               f32x2 instructions, reading the partial product from TMEM 16
//               columns at a time. At the end of the unit each warp writes its
//               [32 x 64] block to dW: the second 32 columns by coalesced
//               stores through a swizzled shared-memory buffer, then the first
//               32 columns by a TMA tensor store from the same buffer, which
//               drains while the next unit computes.
// The per-segment rescale costs as many FP32 lane operations as the FP8 MMA
// takes tensor cycles, so the tile is as wide as the registers allow (64
// accumulators a thread; warpgroup 0 of producer, MMA and two idle warps gives
// registers to the rescale warpgroups with setmaxnreg); the wide
// tile halves the TMA operations and barrier rounds per FLOP against a 128 x 128
// tile. The dout operand's codes may be e5m2 (the configurable gradient dtype of
// the same page); the MMA then reads B as e5m2 (kind::f8f6f4 takes mixed fp8
// types). An expert without rows writes zeros.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace fp8moe {
namespace tg {

constexpr int kBK = 128;                          // k per tile (MMA M)
constexpr int kBN = 256;                          // n per tile (MMA N)
constexpr int kStages = 3;
constexpr int kXBytes = 128 * kBK;                // qx tile, 16 KB
constexpr int kDChunk = 128 * 128;                // one 128-column qd box, 16 KB
constexpr int kDBytes = 128 * kBN;                // qd tile, two boxes
constexpr int kStageBytes = kXBytes + kDBytes;    // 48 KB
constexpr int kEpiWarps = 16;                     // 4 per TMEM lane quarter
constexpr int kCols = kBN * 4 / kEpiWarps;        // 64 accumulator columns per thread
constexpr int kChunk = 16;                        // columns per TMEM load
constexpr int kTBufs = 2;                         // TMEM partial buffers of kBN columns
constexpr int kCtlWarps = 4;                      // producer, MMA, two idle: one warpgroup
constexpr int kThreads = (kCtlWarps + kEpiWarps) * 32;   // 640
constexpr int kCtlRegs = 32, kEpiRegs = 112;       // per thread after the register hand-over
static_assert(kCtlRegs * kCtlWarps + kEpiRegs * kEpiWarps <= (65536 / kThreads / 8 * 8) * (kThreads / 32),
              "register split exceeds the launch allocation");
constexpr int kTmemCols = kTBufs * kBN;           // 512
constexpr int kXpose = 32 * 32 * 4;               // per-warp transpose buffer (32 x 32 f32)
constexpr int kSRing = 8;                         // scale ring slots
static_assert((kSRing & (kSRing - 1)) == 0 && (kTBufs & (kTBufs - 1)) == 0, "rings of 2^n");

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
  alignas(16) float sx[kSRing][kBK];
  alignas(16) float sd[kSRing][kBN];
  int32_t segbase[kMaxExperts + 1];
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kEpiWarps * kXpose + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");
// the group bounds are staged in the transpose buffers before the first unit
static_assert(kEpiWarps * kXpose >= 2 * kMaxExperts * 4, "transpose buffers too small for groups");

// a0 += (s * d0) * p0 and a1 += (s * d1) * p1 as packed f32x2 instructions (one
// multiply and one fused multiply-add per column, both round-to-nearest: the
// same bits as the scalar form, in half the issue slots)
__device__ __forceinline__ void rescale_pair(float& a0, float& a1, float s, float d0, float d1,
                                             uint32_t p0, uint32_t p1) {
  asm("{\n\t.reg .b64 t, p, acc, sd, dd;\n\t"
      "mov.b64 sd, {%2, %2};\n\t"
      "mov.b64 dd, {%3, %4};\n\t"
      "mul.rn.f32x2 t, sd, dd;\n\t"
      "mov.b64 p, {%5, %6};\n\t"
      "mov.b64 acc, {%0, %1};\n\t"
      "fma.rn.f32x2 acc, t, p, acc;\n\t"
      "mov.b64 {%0, %1}, acc;\n\t}"
      : "+f"(a0), "+f"(a1) : "f"(s), "f"(d0), "f"(d1), "r"(p0), "r"(p1));
}

__global__ void __launch_bounds__(kThreads, 1)
tgmm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmD,
            const __grid_constant__ CUtensorMap tmW,
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
    int32_t* g_begin = reinterpret_cast<int32_t*>(xpose);
    int32_t* g_end = g_begin + kMaxExperts;
    load_groups_warp0(gs, E, M, g_begin, g_end, &s.T, blockIdx.x == 0);
    __syncwarp();
    int32_t carry = 0;
    for (int base = 0; base < E; base += 32) {
      int e = base + lane;
      int32_t n = 0;
      if (e < E && g_end[e] > g_begin[e]) n = (g_end[e] - 1) / 128 - g_begin[e] / 128 + 1;
      int32_t incl = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      if (e < E) s.segbase[e] = carry + incl - n;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    fence_proxy_async_smem();   // the staged group bounds precede TMA use of the buffers
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
      // filled by the 32 lanes of the producer warp (one cp.async arrival each)
      for (int i = 0; i < kSRing; ++i) {
        mbar_init(&s.sfull[i], 32);
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

  // warpgroup 0 hands registers to the four rescale warpgroups
  if (warp < kCtlWarps) {
    setmaxnreg_dec<kCtlRegs>();
  if (warp == 0) {
    // ============================== producer ================================
    int st = 0;
    uint32_t ph = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const int e = u / units_per_e, rem = u - e * units_per_e;
      const int kt = rem / nnt, ntile = rem - kt * nnt;
      const int q0 = s.segbase[e], q1 = s.segbase[e + 1];
      // scale columns of this lane: sx [4 lane, 4 lane + 4) of the k tile, sd
      // the same and 128 further of the n tile; columns past K or N are zero-filled
      // (K, N % 16 == 0, so a 16-byte piece is all in or all out)
      const int kc = kt * kBK + lane * 4, nc0 = ntile * kBN + lane * 4, nc1 = nc0 + 128;
      const uint32_t bx = kc < K ? 16u : 0u, b0 = nc0 < N ? 16u : 0u, b1 = nc1 < N ? 16u : 0u;
      for (int q = q0; q < q1; ++q) {
        if (!mbar_wait_warp(&s.empty[st], ph ^ 1, kWhereProducer)) { ok = false; break; }
        const int ss = (int)(issued % kSRing);
        if (!mbar_wait_warp(&s.sempty[ss], (uint32_t)(((issued / kSRing) & 1) ^ 1), kWhereProducer)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&s.full[st], kStageBytes);
          uint8_t* a = tiles + st * kStageBytes;
          tma_load_2d(a, &tmX, &s.full[st], kt * kBK, q * 128);
          tma_load_2d(a + kXBytes, &tmD, &s.full[st], ntile * kBN, q * 128);
          tma_load_2d(a + kXBytes + kDChunk, &tmD, &s.full[st], ntile * kBN + 128, q * 128);
        }
        const float* sxq = sx + (int64_t)q * K;
        const float* sdq = sd + (int64_t)q * N;
        cp_async16(&s.sx[ss][lane * 4], bx ? sxq + kc : sxq, bx);
        cp_async16(&s.sd[ss][lane * 4], b0 ? sdq + nc0 : sdq, b0);
        cp_async16(&s.sd[ss][128 + lane * 4], b1 ? sdq + nc1 : sdq, b1);
        cp_async_mbar_arrive(&s.sfull[ss]);
        ++issued;
        if (++st == kStages) { st = 0; ph ^= 1; }
      }
    }
    cp_async_wait_all();
    if (lane == 0) {
      const int64_t n_last = issued < kStages ? issued : kStages;
      for (int64_t i = 1; i <= n_last; ++i) {
        const int64_t idx = issued - i;
        mbar_wait(&s.full[idx % kStages], (uint32_t)((idx / kStages) & 1), kWhereDrain);
      }
    }
  } else if (warp == 1) {
    // ================================ MMA ===================================
    if (lane == 0) {
      // A = qx slot, [K_mma = 128 rows][M_mma = 128 k] -> MN-major, one atom;
      // B = qd slot, [K_mma = 128 rows][N_mma = 256 n] -> MN-major, two atoms of
      // 128 columns, 16 KB apart (leading-dimension offset).
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
            const uint64_t ad = make_desc(a_addr + kk * 4096, kDChunk, 1024, kSwizzle128B);
            const uint64_t bd = make_desc(b_addr + kk * 4096, kDChunk, 1024, kSwizzle128B);
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
  }
  } else {
    setmaxnreg_inc<kEpiRegs>();
    // ============================ rescale + store ===========================
    const int ew = warp - kCtlWarps;         // 0..15
    const int quarter = warp & 3;            // TMEM lanes 32*quarter ..
    const int cg = ew >> 2;                  // columns [kCols*cg, kCols*cg + kCols)
    const int r = quarter * 32 + lane;       // k row inside the tile
    float* xp = xpose + ew * (kXpose / 4);
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(cg * kCols);
    // segments consumed so far: TMEM buffer used % kTBufs, scale slot used % kSRing
    // (both powers of two, so one counter gives buffers, slots and phases)
    uint32_t used = 0;
    bool failed = false;
    for (int u = blockIdx.x; u < total && !failed; u += gridDim.x) {
      const int e = u / units_per_e, rem = u - e * units_per_e;
      const int kt = rem / nnt, ntile = rem - kt * nnt;
      const int q0 = s.segbase[e], q1 = s.segbase[e + 1];
      float a[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) a[i] = 0.0f;
      for (int q = q0; q < q1; ++q) {
        const int ss = (int)(used % kSRing), acc = (int)(used % kTBufs);
        if (!mbar_wait_warp(&s.sfull[ss], (used / kSRing) & 1, kWhereEpilogue) ||
            !mbar_wait_warp(&s.tfull[acc], (used / kTBufs) & 1, kWhereEpilogue)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const float sxk = s.sx[ss][r];
        const float4* sdv = reinterpret_cast<const float4*>(&s.sd[ss][cg * kCols]);
#pragma unroll
        for (int c = 0; c < kCols / kChunk; ++c) {
          uint32_t v[kChunk];
          tmem_ld16(tl + (uint32_t)(acc * kBN + c * kChunk), v);
          tmem_ld_wait();
          if (c == kCols / kChunk - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(&s.tempty[acc]);   // TMEM buffer free once in registers
          }
#pragma unroll
          for (int i = 0; i < kChunk / 4; ++i) {
            const float4 d4 = sdv[c * (kChunk / 4) + i];
            float* ap = a + c * kChunk + 4 * i;
            rescale_pair(ap[0], ap[1], sxk, d4.x, d4.y, v[4 * i], v[4 * i + 1]);
            rescale_pair(ap[2], ap[3], sxk, d4.z, d4.w, v[4 * i + 2], v[4 * i + 3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sempty[ss]);   // scale slot free
        ++used;
      }
      if (failed) break;
      // store the [32 k rows x 64 n] block through the per-warp buffer, kept in
      // the 128-byte swizzled layout (16-byte chunk c4 of row i at chunk
      // c4 ^ (i & 7)): columns 32..63 first by coalesced 128-byte row stores,
      // then columns 0..31 by a TMA tensor store (rows past K and columns past
      // N clipped) that leaves the buffer while the next unit computes.
      const int k_warp0 = kt * kBK + quarter * 32;
      const int n_w0 = ntile * kBN + cg * kCols;
      if (lane == 0) bulk_wait_read();   // the previous unit's box has left the buffer
      __syncwarp();
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const int pc = c4 ^ (lane & 7);
        *reinterpret_cast<float4*>(xp + lane * 32 + pc * 4) =
            make_float4(a[32 + c4 * 4], a[32 + c4 * 4 + 1], a[32 + c4 * 4 + 2], a[32 + c4 * 4 + 3]);
      }
      __syncwarp();
#pragma unroll 1
      for (int it = 0; it < 8; ++it) {
        const int i = it * 4 + (lane >> 3);       // row within the 32-row block
        const int c4 = lane & 7;
        const float4 v = *reinterpret_cast<const float4*>(xp + i * 32 + ((c4 ^ (i & 7)) * 4));
        const int kk = k_warp0 + i;
        const int nn = n_w0 + 32 + c4 * 4;
        if (kk < K && nn < N)   // N % 16 == 0: a 4-column group is all in or all out
          *reinterpret_cast<float4*>(dW + ((int64_t)e * K + kk) * N + nn) = v;
      }
      __syncwarp();
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const int pc = c4 ^ (lane & 7);
        *reinterpret_cast<float4*>(xp + lane * 32 + pc * 4) =
            make_float4(a[c4 * 4], a[c4 * 4 + 1], a[c4 * 4 + 2], a[c4 * 4 + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && k_warp0 < K && n_w0 < N) {
        tma_store_3d(&tmW, xp, n_w0, k_warp0, e);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait();
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
  // the register hand-over needs the full launch allocation: refuse a build whose
  // kernel was compiled with fewer registers than the split assumes
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, tgmm_kernel);
  if (err != cudaSuccess) return err;
  if (fa.numRegs * (kThreads / 32) < kCtlRegs * kCtlWarps + kEpiRegs * kEpiWarps)
    return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(tgmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  tgmm_kernel<<<num_sms, kThreads, kSmemBytes, s>>>(a.tmX, a.tmD, a.tmW, a.sx, a.sd, a.gs, a.dW, a.M,
                                                    a.K, a.N, a.E, a.d_fmt);
  return cudaGetLastError();
}
