// gmm_fwd.cu -- ragged grouped matmul forward on tcgen05 tensor cores.
//
//   out[m, n] = sx[m] * sw[e(m), n] * sum_k qx[m, k] * qw[e(m), k, n]       (FP8 arm)
//   out[m, j] = silu(g) * u, g = y[m, j], u = y[m, N/2 + j]                  (SwiGLU)
//
// "MoE: native FP8 QAT for routed-expert GMMs", Description and Implementation:
// the wi/wo forward GMMs run FP8 x FP8 from the FP8 weight codes and per-channel
// scales, with the activation quantized per row over the full K (quant.cu writes
// the codes this kernel reads), f32 accumulation, and SwiGLU fused into wi.
// The same kernel, instantiated with bf16 operands and no scales, is the BF16
// grouped matmul used as the fake-QAT comparison arm ("... Tests": the BF16 GMM
// gets a weight dequantized beforehand).
//
// Design (one CTA per SM, persistent):
//   warp 0      TMA producer: A tile [128 rows x 128 bytes of K] (K-major,
//               128-byte swizzle) and the B tile, 256 columns of the
//               N-contiguous weight by 128 bytes of K (MN-major, 128-byte
//               swizzle); 4-stage ring of 48 KB stages.
//   warp 1      TMEM allocation (512 columns = two 128x256 f32 accumulators) and
//               the single thread that issues tcgen05.mma (M=128, N=256).
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator, scales,
//               SwiGLU, bf16 rounding, row-masked 16-byte stores. The second
//               accumulator lets the next tile's MMAs run meanwhile.
// Work units are (expert, 128-row m tile, 256-column n tile), enumerated expert
// by expert, n tile by n tile, m tiles fastest, so that concurrently running
// CTAs share weight tiles through L2. Each CTA derives the ragged layout from
// group_sizes itself; tiles begin at their group's first row and rows past the
// group end are computed but never stored.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace fp8moe {
namespace fwd {

constexpr int kStages = 4;
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kABytes = kBM * 128;          // 16 KB
constexpr int kBBytes = kBN * 128;          // 32 KB: 256 columns x 128 bytes of K
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t T;
  int32_t total_units;
  int32_t abort_flag;
  float sw[2][kBN];
  int32_t begin[kMaxExperts];
  int32_t end[kMaxExperts];
  int32_t prefix[kMaxExperts + 1];
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

struct Unit {
  int e, row0, rows, j;
};

__device__ __forceinline__ Unit decode_unit(const Smem& s, int E, int nt, int u) {
  Unit r;
  r.e = find_bucket(s.prefix, E, u);
  const int mt = (s.end[r.e] - s.begin[r.e] + kBM - 1) / kBM;
  const int local = u - s.prefix[r.e];
  r.j = local / mt;
  const int i = local - r.j * mt;
  r.row0 = s.begin[r.e] + i * kBM;
  r.rows = min(kBM, s.end[r.e] - r.row0);
  return r;
}

// FP8: operands are 1 byte, a 128-byte swizzle row holds 128 K values of A (or
// 128 N values of B); BF16: 64.
template <bool FP8, bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
gmm_fwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const float* __restrict__ sx, const float* __restrict__ scale,
               const int32_t* __restrict__ gs, __nv_bfloat16* __restrict__ out, int64_t M, int K,
               int N, int E) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  Smem& s = *reinterpret_cast<Smem*>(tiles + (size_t)kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  constexpr int kElemsPerRow = FP8 ? 128 : 64;        // elements per 128-byte row
  const int Nout = SWIGLU ? N / 2 : N;
  const int nt = SWIGLU ? (Nout + 127) / 128 : (N + kBN - 1) / kBN;
  const int nkb = (K + kElemsPerRow - 1) / kElemsPerRow;

  // ---- set-up: ragged layout, unit prefix, barriers, TMEM
  if (warp == 0) {
    load_groups_warp0(gs, E, M, s.begin, s.end, &s.T, blockIdx.x == 0);
    __syncwarp();
    int32_t carry = 0;
    for (int base = 0; base < E; base += 32) {
      int e = base + lane;
      int32_t n = 0;
      if (e < E) n = ((s.end[e] - s.begin[e] + kBM - 1) / kBM) * nt;
      int32_t incl = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
      }
      if (e < E) s.prefix[e] = carry + incl - n;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      s.prefix[E] = carry;
      s.total_units = carry;
      s.abort_flag = 0;
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(&s.full[i], 1);
        mbar_init(&s.empty[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.tfull[i], 1);
        mbar_init(&s.tempty[i], 4);   // one elected lane per epilogue warp
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
    // ============================ TMA producer ============================
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit t = decode_unit(s, E, nt, u);
        int nb0, nb1;
        if (SWIGLU) { nb0 = t.j * 128; nb1 = Nout + t.j * 128; }
        else { nb0 = t.j * kBN; nb1 = t.j * kBN + 128; }
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&s.empty[st], ph ^ 1, kWhereProducer)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.full[st], kStageBytes);
          uint8_t* a = tiles + st * kStageBytes;
          uint8_t* b = a + kABytes;
          const int k0 = kb * kElemsPerRow;
          tma_load_2d(a, &tmA, &s.full[st], k0, t.row0);
          if (FP8) {
            tma_load_3d(b, &tmB, &s.full[st], nb0, k0, t.e);
            tma_load_3d(b + 16384, &tmB, &s.full[st], nb1, k0, t.e);
          } else {
            // bf16: four 64-column boxes of 64 K rows (8 KB each)
            tma_load_3d(b, &tmB, &s.full[st], nb0, k0, t.e);
            tma_load_3d(b + 8192, &tmB, &s.full[st], nb0 + 64, k0, t.e);
            tma_load_3d(b + 16384, &tmB, &s.full[st], nb1, k0, t.e);
            tma_load_3d(b + 24576, &tmB, &s.full[st], nb1 + 64, k0, t.e);
          }
          ++issued;
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
      }
      if (!ok) s.abort_flag = 1;
      // drain: every load issued must have landed before the CTA may exit
      int64_t n_last = issued < kStages ? issued : kStages;
      for (int64_t i = 1; i <= n_last; ++i) {
        int64_t idx = issued - i;
        mbar_wait(&s.full[idx % kStages], (uint32_t)((idx / kStages) & 1), kWhereDrain);
      }
    }
  } else if (warp == 1) {
    // ============================== MMA issuer ============================
    if (lane == 0) {
      constexpr uint32_t idesc = FP8 ? make_idesc(0, 0, 0, 1, kBM, kBN)
                                     : make_idesc(1, 1, 0, 1, kBM, kBN);
      // B (MN-major): atoms of 128 bytes along N; FP8 atom = 128 columns with
      // the second half 16 KB further; BF16 atom = 64 columns, 8 KB apart.
      constexpr uint32_t kBLbo = FP8 ? 16384 : 8192;
      // one MMA consumes 32 bytes of K: FP8 32 K values (= 32 B-rows), BF16 16
      constexpr uint32_t kBStep = FP8 ? 32 * 128 : 16 * 128;
      int st = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        if (!mbar_wait(&s.tempty[acc], aph ^ 1, kWhereMma)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&s.full[st], ph, kWhereMma)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + st * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = make_desc(a_addr + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = make_desc(b_addr + kk * kBStep, kBLbo, 1024, kSwizzle128B);
            if (FP8) mma_f8f6f4(d, ad, bd, idesc, (kb | kk) != 0);
            else mma_f16(d, ad, bd, idesc, (kb | kk) != 0);
          }
          mma_commit(&s.empty[st]);
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
        if (!ok) break;
        mma_commit(&s.tfull[acc]);
        acc ^= 1;
        if (acc == 0) aph ^= 1;
      }
      if (!ok) s.abort_flag = 1;
      // all MMAs of this thread complete before TMEM may be released
      mma_commit(&s.drain);
      mbar_wait(&s.drain, 0, kWhereDrain);
    }
  } else {
    // =============================== epilogue =============================
    const int et = threadIdx.x - 64;                 // 0..127
    const int quarter = warp & 3;                    // TMEM lanes 32*quarter ..
    const int r = quarter * 32 + lane;               // row inside the tile
    int acc = 0;
    uint32_t aph = 0;
    int sb = 0;
    // A timed-out wait marks the thread failed; it keeps iterating (without
    // touching TMEM) so that every epilogue thread passes the same named barriers.
    bool failed = false;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit t = decode_unit(s, E, nt, u);
      // per-column scales of this tile's 256 accumulator columns
      if (FP8) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = et + 128 * h;
          int col;
          bool in;
          if (SWIGLU) {
            col = (c < 128 ? 0 : Nout) + t.j * 128 + (c & 127);
            in = (t.j * 128 + (c & 127)) < Nout;
          } else {
            col = t.j * kBN + c;
            in = col < N;
          }
          s.sw[sb][c] = in ? __ldg(scale + (int64_t)t.e * N + col) : 0.0f;
        }
      }
      named_bar_sync(1, 128);
      const bool row_ok = r < t.rows;
      const int64_t row = (int64_t)t.row0 + r;
      const float sxr = (FP8 && row_ok) ? __ldg(sx + row) : 1.0f;
      if (!failed && !mbar_wait_warp(&s.tfull[acc], aph, kWhereEpilogue)) failed = true;
      if (failed) {
        acc ^= 1;
        if (acc == 0) aph ^= 1;
        sb ^= 1;
        continue;
      }
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
      __nv_bfloat16* orow = out + row * Nout;
      constexpr int kChunks = SWIGLU ? 4 : 8;
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c) {
        uint32_t o[16];
        int col0;
        if (SWIGLU) {
          uint32_t g[32], v[32];
          tmem_ld32(tbase + c * 32, g);
          tmem_ld32(tbase + 128 + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float y[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float gg = __uint_as_float(g[i + h]);
              float uu = __uint_as_float(v[i + h]);
              if (FP8) {
                gg = __fmul_rn(__fmul_rn(gg, sxr), s.sw[sb][c * 32 + i + h]);
                uu = __fmul_rn(__fmul_rn(uu, sxr), s.sw[sb][128 + c * 32 + i + h]);
              }
              const float sg = __fdiv_rn(gg, __fadd_rn(1.0f, expf(-gg)));
              y[h] = __fmul_rn(sg, uu);
            }
            o[i / 2] = f32x2_to_bf16x2(y[0], y[1]);
          }
          col0 = t.j * 128 + c * 32;
        } else {
          uint32_t v[32];
          tmem_ld32(tbase + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float y0 = __uint_as_float(v[i]), y1 = __uint_as_float(v[i + 1]);
            if (FP8) {
              y0 = __fmul_rn(__fmul_rn(y0, sxr), s.sw[sb][c * 32 + i]);
              y1 = __fmul_rn(__fmul_rn(y1, sxr), s.sw[sb][c * 32 + i + 1]);
            }
            o[i / 2] = f32x2_to_bf16x2(y0, y1);
          }
          col0 = t.j * kBN + c * 32;
        }
        if (row_ok) {
          if (col0 + 32 <= Nout) {
            uint4* dst = reinterpret_cast<uint4*>(orow + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          } else {
            uint16_t* dst = reinterpret_cast<uint16_t*>(orow);
#pragma unroll
            for (int q = 0; q < 32; ++q)
              if (col0 + q < Nout) dst[col0 + q] = (uint16_t)(o[q / 2] >> (16 * (q & 1)));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.tempty[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1;
      sb ^= 1;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool FP8, bool SWIGLU>
cudaError_t launch(const GmmFwdArgs& a, int num_sms, cudaStream_t s) {
  auto kern = gmm_fwd_kernel<FP8, SWIGLU>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  kern<<<num_sms, kThreads, kSmemBytes, s>>>(a.tmA, a.tmB, a.sx, a.scale, a.gs,
                                             static_cast<__nv_bfloat16*>(a.out), a.M, a.K, a.N,
                                             a.E);
  return cudaGetLastError();
}

}  // namespace fwd
}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_gmm_fwd)

cudaError_t fp8moe_launch_gmm_fp8_fwd(const GmmFwdArgs& a, int num_sms, cudaStream_t s) {
  return a.swiglu ? fp8moe::fwd::launch<true, true>(a, num_sms, s)
                  : fp8moe::fwd::launch<true, false>(a, num_sms, s);
}

cudaError_t fp8moe_launch_gmm_bf16_fwd(const GmmFwdArgs& a, int num_sms, cudaStream_t s) {
  return a.swiglu ? fp8moe::fwd::launch<false, true>(a, num_sms, s)
                  : fp8moe::fwd::launch<false, false>(a, num_sms, s);
}
