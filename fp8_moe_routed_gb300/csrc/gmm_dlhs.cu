// gmm_dlhs.cu -- backward dLHS grouped matmul reading FP8 weight codes.
//
//   dlhs[m, k] = sum_n dout[m, n] * bf16(f32(code[e(m), k, n]) * scale[e(m), n])
//
// "MoE: native FP8 QAT for routed-expert GMMs", Description and Implementation
// (the rhs_contract_dequant path): the dLHS GMM reads the FP8 codes, dequantizes
// each weight tile on chip and feeds it straight to the matmul, so no BF16 copy
// of the weight is written to HBM; the result is bit-identical to running the
// BF16 GMM on the dequantized weight. With a single contraction tile the
// dequantized block is also kept on chip across the expert's m tiles (the
// review thread on the cache: it only hits with one K tile).
//
// Three kernels, all giving the same bits:
//   gmm_dlhs_pair_kernel (gmm_dlhs_pair.cu) -- the default for contractions
//     past 256: CTA pairs, the product transposed, the dequantized weight tile
//     written into tensor memory as the MMA's A operand;
//   gmm_dlhs_kernel<CACHED = true> -- contractions up to 256: the dequantized
//     weight block cached in shared memory across a run of m tiles;
//   gmm_dlhs_kernel<CACHED = false> -- streaming, kept as the dSwiGLU default
//     (two accumulators let its SwiGLU epilogue overlap the next tile's MMAs;
//     the pair kernel has one and must hold it through the SwiGLU math) and as
//     a forced path.
//
// GB300 design (one CTA per SM, persistent), per 128-row x 256-column output
// tile and 64-wide contraction step:
//   warp 0       TMA: dout tiles [128 x 64] bf16 (K-major, 128-byte swizzle) and
//                the codes tile [256 x 64] u8 (no swizzle) into a 3-deep ring.
//                Streaming units cover two m tiles of one expert, so every
//                dequantized weight tile feeds two accumulators (half the
//                dequantization per FLOP).
//   warps 6..13  dequant: e4m3 -> f32, x scale (one f32 multiply), round to
//                bf16, write the [256 x 64] bf16 B operand in the K-major
//                128-byte-swizzle layout the tensor core reads (2-deep ring).
//   warp 1       tcgen05.mma kind::f16 (M=128, N=256, K=16) into TMEM.
//   warps 2..5,  epilogue: TMEM -> bf16 -> row-masked stores, two warps per
//   14..17       TMEM lane quarter, each one half of the columns. TMEM holds two
//                accumulators: the two m tiles of a streaming unit, or (cached)
//                consecutive m tiles so that the epilogue overlaps the MMAs.
// dSwiGLU variant (DSW): the wo dLHS of "gmm_dswiglu_fp8" ([NQ] Implementation)
// with the SwiGLU backward in the epilogue. The accumulator is dh = dL/dh for
// h = silu(g) * u; the epilogue reads g and u from the wi output gu [M, 2F] and
// writes dgu [M, 2F]: dg = dh * u * sig(g) * (1 + g * (1 - sig(g))) in columns
// [0, F) and du = dh * g * sig(g) in [F, 2F), so dh itself never reaches HBM.
// Cached variant (the contraction fits in <= 4 steps, i.e. N <= 256): a work
// unit is (expert, k tile, run of m tiles); the whole dequantized
// [256 x N] block stays in shared memory and only dout tiles stream. Both
// variants issue the same MMA sequence per output tile, so their results are
// bit-identical.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace fp8moe {
namespace dlhs {

constexpr int kBM = 128;
constexpr int kBN = 256;                 // output columns (k) per tile = MMA N
constexpr int kBK = 64;                  // contraction (n) per step
constexpr int kLdStages = 4;            // ring slots (cached: A tiles)
constexpr int kLdStagesStream = 3;      // streaming: 3 slots of [A0 | A1 | C]
constexpr int kBStages = 2;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB dout tile
constexpr int kCBytes = kBN * kBK;       // 16 KB codes tile
constexpr int kBBytes = kBN * kBK * 2;   // 32 KB bf16 operand
constexpr int kDqWarps = 8;
constexpr int kEpiWarps = 8;                    // two per TMEM lane quarter
constexpr int kThreads = (2 + kEpiWarps + kDqWarps) * 32;   // 576
// Registers are budgeted per SM sub-partition: 18 warps put 5 on two of them,
// so a thread may hold 16384 / (5 * 32) -> 96 registers; launch bounds of 640
// threads give the compiler that cap.
constexpr int kRegBudgetThreads = 640;
constexpr int kTmemCols = 512;
constexpr int kMaxCachedSteps = 4;       // cached variant: N <= 256
constexpr int kCachedRun = 8;            // m tiles per cached work unit

// Streaming layout: ld ring [A0 | A1 | C] 3 x 48 KB, B ring 2 x 32 KB = 208 KB.
// Cached layout: B cache 4 x 32 KB, A ring 4 x 16 KB, C staging 16 KB = 208 KB.
constexpr int kStreamStage = 2 * kABytes + kCBytes;
constexpr size_t kTileBytesStream = (size_t)kLdStagesStream * kStreamStage + kBStages * kBBytes;
constexpr size_t kTileBytesCached = (size_t)kMaxCachedSteps * kBBytes + kLdStages * kABytes + kCBytes;

struct Smem {
  uint64_t ld_full[kLdStages];
  uint64_t ld_empty[kLdStages];
  uint64_t b_full[kMaxCachedSteps];
  uint64_t b_empty[kMaxCachedSteps];
  uint64_t c_full, c_empty;
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t T;
  int32_t total_units;
  int32_t begin[kMaxExperts];
  int32_t end[kMaxExperts];
  int32_t prefix[kMaxExperts + 1];
};

template <bool CACHED>
constexpr size_t smem_bytes() {
  return 1024 + (CACHED ? kTileBytesCached : kTileBytesStream) + sizeof(Smem);
}
static_assert(smem_bytes<true>() <= 232448 && smem_bytes<false>() <= 232448,
              "shared memory per CTA exceeds 227 KB");

struct Unit {
  int e, row0, rows_total, mtiles, j;   // mtiles: m tiles in this unit (streaming: 1)
};

// Streaming: (e, j, pair of m tiles), pairs fastest.
// Cached:    (e, j, run) with runs of up to kCachedRun m tiles.
template <bool CACHED>
__device__ __forceinline__ int unit_run(int mt) {
  return CACHED ? kCachedRun : 2;
}

template <bool CACHED>
__device__ __forceinline__ Unit decode_unit(const Smem& s, int E, int nt, int u) {
  Unit r;
  r.e = find_bucket(s.prefix, E, u);
  const int mt = (s.end[r.e] - s.begin[r.e] + kBM - 1) / kBM;
  const int run = unit_run<CACHED>(mt);
  const int nruns = (mt + run - 1) / run;
  const int local = u - s.prefix[r.e];
  r.j = local / nruns;
  const int i = local - r.j * nruns;
  const int first_tile = i * run;
  r.row0 = s.begin[r.e] + first_tile * kBM;
  r.mtiles = min(run, mt - first_tile);
  r.rows_total = s.end[r.e] - r.row0;
  return r;
}

// Dequantize a [256 x 64] codes tile (row r at r*64 bytes) into the K-major
// 128-byte-swizzled bf16 operand (row r at r*128 bytes, 16-byte chunk c stored at
// chunk c ^ (r & 7)). Thread t of the 256 dequant threads converts the 16-code
// chunks t, t + 256, t + 512, t + 768; all four share the same 16 columns.
__device__ __forceinline__ void dequant_tile(const uint8_t* __restrict__ csm, uint8_t* __restrict__ bsm,
                                             const float* __restrict__ sc16, int t) {
  const int sub = t & 3;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int c = t + 256 * it;
    const int r = c >> 2;
    const uint4 cw = *reinterpret_cast<const uint4*>(csm + r * 64 + sub * 16);
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f0, f1, f2, f3;
      half2_to_f32(e4m3x2_to_f16x2((uint16_t)(w[i] & 0xFFFFu)), f0, f1);
      half2_to_f32(e4m3x2_to_f16x2((uint16_t)(w[i] >> 16)), f2, f3);
      o[2 * i] = f32x2_to_bf16x2(__fmul_rn(f0, sc16[4 * i]), __fmul_rn(f1, sc16[4 * i + 1]));
      o[2 * i + 1] = f32x2_to_bf16x2(__fmul_rn(f2, sc16[4 * i + 2]), __fmul_rn(f3, sc16[4 * i + 3]));
    }
    uint8_t* rowp = bsm + r * 128;
    const int x = r & 7;
    *reinterpret_cast<uint4*>(rowp + (((2 * sub) ^ x) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(rowp + (((2 * sub + 1) ^ x) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

__device__ __forceinline__ void load_scales16(const float* __restrict__ scale, int64_t base, int n0,
                                              int N, float* sc16) {
#pragma unroll
  for (int i = 0; i < 16; ++i) sc16[i] = 0.0f;
  if (n0 + 16 <= N) {
    const float4* p = reinterpret_cast<const float4*>(scale + base + n0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4 f = __ldg(p + i);
      sc16[4 * i] = f.x; sc16[4 * i + 1] = f.y; sc16[4 * i + 2] = f.z; sc16[4 * i + 3] = f.w;
    }
  }
  // N % 16 == 0, so a 16-column group is either fully in range or fully out.
}

// Epilogue of one finished accumulator: 128 rows x 256 columns f32 -> bf16.
__device__ __forceinline__ void store_tile(uint32_t tbase, int r, bool row_ok,
                                           __nv_bfloat16* __restrict__ orow, int col_base, int K,
                                           int nchunks) {
#pragma unroll 1
  for (int c = 0; c < nchunks; ++c) {
    uint32_t v[32];
    tmem_ld32(tbase + c * 32, v);
    tmem_ld_wait();
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) o[i / 2] = f32x2_to_bf16x2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
    const int col0 = col_base + c * 32;
    if (row_ok) {
      if (col0 + 32 <= K) {
        st_global_64B(orow + col0, o);
      } else {
        uint16_t* dst = reinterpret_cast<uint16_t*>(orow);
#pragma unroll
        for (int q = 0; q < 32; ++q)
          if (col0 + q < K) dst[col0 + q] = (uint16_t)(o[q / 2] >> (16 * (q & 1)));
      }
    }
  }
}

// dSwiGLU epilogue of one finished accumulator (dh, 128 rows x 256 columns of
// F): g = gurow[f], u = gurow[F + f] -> dgu row: dg at f, du at F + f.
__device__ __forceinline__ void dswiglu8(const uint4& gw, const uint4& uw, const uint32_t* v,
                                         uint32_t* og, uint32_t* ou) {
  const uint32_t gg[4] = {gw.x, gw.y, gw.z, gw.w};
  const uint32_t uu[4] = {uw.x, uw.y, uw.z, uw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float dg[2], du[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float g = __uint_as_float((gg[i] >> (16 * h)) << 16);
      const float u = __uint_as_float((uu[i] >> (16 * h)) << 16);
      const float d = __uint_as_float(v[2 * i + h]);
      // sig(g) from the hardware exponential and an IEEE reciprocal: relative
      // error ~1e-6 against bf16 outputs (2^-9 relative half-ulp)
      const float sg = __frcp_rn(__fadd_rn(1.0f, __expf(-g)));
      const float dsilu = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sg))));
      dg[h] = __fmul_rn(__fmul_rn(d, u), dsilu);
      du[h] = __fmul_rn(d, __fmul_rn(g, sg));
    }
    og[i] = f32x2_to_bf16x2(dg[0], dg[1]);
    ou[i] = f32x2_to_bf16x2(du[0], du[1]);
  }
}

__device__ __forceinline__ void store_tile_dswiglu(uint32_t tbase, bool row_ok,
                                                   const __nv_bfloat16* __restrict__ gurow,
                                                   __nv_bfloat16* __restrict__ orow, int col_base,
                                                   int F, int nchunks) {
#pragma unroll 1
  for (int c = 0; c < nchunks; ++c) {
    uint32_t v[32];
    tmem_ld32(tbase + c * 32, v);
    tmem_ld_wait();
    const int col0 = col_base + c * 32;
    if (!row_ok || col0 >= F) continue;
    // F % 16 == 0: the valid part of a chunk is whole 8-column groups
    uint4 g[4], u[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (col0 + 8 * q < F) {
        g[q] = __ldg(reinterpret_cast<const uint4*>(gurow + col0 + 8 * q));
        u[q] = __ldg(reinterpret_cast<const uint4*>(gurow + F + col0 + 8 * q));
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (col0 + 8 * q < F) {
        uint32_t og[4], ou[4];
        dswiglu8(g[q], u[q], v + 8 * q, og, ou);
        *reinterpret_cast<uint4*>(orow + col0 + 8 * q) = make_uint4(og[0], og[1], og[2], og[3]);
        *reinterpret_cast<uint4*>(orow + F + col0 + 8 * q) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
      }
    }
  }
}

template <bool CACHED, bool DSW>
__global__ void __launch_bounds__(kRegBudgetThreads, 1)
gmm_dlhs_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC,
                const float* __restrict__ scale, const int32_t* __restrict__ gs,
                const __nv_bfloat16* __restrict__ gu, __nv_bfloat16* __restrict__ dlhs, int64_t M,
                int N, int K, int E) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  Smem& s = *reinterpret_cast<Smem*>(tiles + (CACHED ? kTileBytesCached : kTileBytesStream));
  // Streaming: [ld slot i: A0 (16 KB) | A1 (16 KB) | C (16 KB)] x 3, then B x 2.
  // Cached:    B cache x 4, A x 4, C staging x 1.
  constexpr int kSlots = CACHED ? kLdStages : kLdStagesStream;
  uint8_t* const ringA = tiles + (CACHED ? kMaxCachedSteps * kBBytes : 0);
  uint8_t* const ringB = tiles + (CACHED ? 0 : kLdStagesStream * kStreamStage);
  uint8_t* const stageC = tiles + kMaxCachedSteps * kBBytes + kLdStages * kABytes;   // cached only
  auto a_tile = [&](int i, int mi) -> uint8_t* {
    return CACHED ? ringA + i * kABytes : tiles + i * kStreamStage + mi * kABytes;
  };
  auto c_tile = [&](int i) -> uint8_t* { return CACHED ? stageC : tiles + i * kStreamStage + 2 * kABytes; };
  auto b_tile = [&](int i) -> uint8_t* { return ringB + i * kBBytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = (K + kBN - 1) / kBN;
  const int nkb = (N + kBK - 1) / kBK;

  if (warp == 0) {
    load_groups_warp0(gs, E, M, s.begin, s.end, &s.T, blockIdx.x == 0);
    __syncwarp();
    int32_t carry = 0;
    for (int base = 0; base < E; base += 32) {
      int e = base + lane;
      int32_t n = 0;
      if (e < E) {
        int mt = (s.end[e] - s.begin[e] + kBM - 1) / kBM;
        const int run = CACHED ? kCachedRun : 2;
        n = ((mt + run - 1) / run) * nt;
      }
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
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmC);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < kLdStages; ++i) {
        mbar_init(&s.ld_full[i], 1);
        // streaming: freed by the MMA commit (A) and each dequant warp (C)
        mbar_init(&s.ld_empty[i], CACHED ? 1 : 1 + kDqWarps);
      }
      for (int i = 0; i < kMaxCachedSteps; ++i) {
        mbar_init(&s.b_full[i], kDqWarps);
        mbar_init(&s.b_empty[i], 1);
      }
      mbar_init(&s.c_full, 1);
      mbar_init(&s.c_empty, kDqWarps);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.tfull[i], 1);
        mbar_init(&s.tempty[i], kEpiWarps);   // one elected lane per epilogue warp
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
      int64_t issued = 0, c_issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit t = decode_unit<CACHED>(s, E, nt, u);
        const int k0 = t.j * kBN;
        if (CACHED) {
          // the unit's whole codes block, one step at a time through the staging slot
          for (int kb = 0; kb < nkb && ok; ++kb) {
            if (!mbar_wait(&s.c_empty, (uint32_t)((c_issued & 1) ^ 1), kWhereProducer)) { ok = false; break; }
            mbar_arrive_expect_tx(&s.c_full, kCBytes);
            tma_load_3d(c_tile(0), &tmC, &s.c_full, kb * kBK, k0, t.e);
            ++c_issued;
          }
        }
        if (CACHED) {
          for (int mi = 0; mi < t.mtiles && ok; ++mi) {
            const int row0 = t.row0 + mi * kBM;
            for (int kb = 0; kb < nkb; ++kb) {
              if (!mbar_wait(&s.ld_empty[st], ph ^ 1, kWhereProducer)) { ok = false; break; }
              mbar_arrive_expect_tx(&s.ld_full[st], kABytes);
              tma_load_2d(a_tile(st, 0), &tmA, &s.ld_full[st], kb * kBK, row0);
              ++issued;
              if (++st == kSlots) { st = 0; ph ^= 1; }
            }
          }
        } else {
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&s.ld_empty[st], ph ^ 1, kWhereProducer)) { ok = false; break; }
            mbar_arrive_expect_tx(&s.ld_full[st], t.mtiles * kABytes + kCBytes);
            for (int mi = 0; mi < t.mtiles; ++mi)
              tma_load_2d(a_tile(st, mi), &tmA, &s.ld_full[st], kb * kBK, t.row0 + mi * kBM);
            tma_load_3d(c_tile(st), &tmC, &s.ld_full[st], kb * kBK, k0, t.e);
            ++issued;
            if (++st == kSlots) { st = 0; ph ^= 1; }
          }
        }
      }
      // drain outstanding copies before the CTA may exit
      int64_t n_last = issued < kSlots ? issued : kSlots;
      for (int64_t i = 1; i <= n_last; ++i) {
        int64_t idx = issued - i;
        mbar_wait(&s.ld_full[idx % kSlots], (uint32_t)((idx / kSlots) & 1), kWhereDrain);
      }
      if (CACHED && c_issued > 0) mbar_wait(&s.c_full, (uint32_t)((c_issued - 1) & 1), kWhereDrain);
    }
  } else if (warp == 1) {
    // ============================== MMA issuer ============================
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(1, 1, 0, 0, kBM, kBN);
      int st = 0;
      uint32_t ph = 0;
      int bst = 0;
      uint32_t bph = 0;
      int64_t cached_fills = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      auto issue = [&](uint32_t d, uint32_t a_addr, uint32_t b_addr, int kb) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = make_desc(a_addr + kk * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = make_desc(b_addr + kk * 32, 16, 1024, kSwizzle128B);
          mma_f16(d, ad, bd, idesc, (kb | kk) != 0);
        }
      };
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit t = decode_unit<CACHED>(s, E, nt, u);
        if (CACHED) {
          // one m tile per accumulator, accumulators alternate (epilogue overlaps)
          for (int mi = 0; mi < t.mtiles && ok; ++mi) {
            if (!mbar_wait(&s.tempty[acc], aph ^ 1, kWhereMma)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * kBN);
            for (int kb = 0; kb < nkb; ++kb) {
              if (!mbar_wait(&s.ld_full[st], ph, kWhereMma)) { ok = false; break; }
              // the cache slot kb is (re)filled once per unit
              if (mi == 0 && !mbar_wait(&s.b_full[kb], (uint32_t)(cached_fills & 1), kWhereMma)) { ok = false; break; }
              tc_fence_after();
              issue(d, smem_u32(a_tile(st, 0)), smem_u32(b_tile(kb)), kb);
              mma_commit(&s.ld_empty[st]);
              if (mi + 1 == t.mtiles) mma_commit(&s.b_empty[kb]);   // slot refillable by the next unit
              if (++st == kSlots) { st = 0; ph ^= 1; }
            }
            if (!ok) break;
            mma_commit(&s.tfull[acc]);
            acc ^= 1;
            if (acc == 0) aph ^= 1;
          }
          ++cached_fills;
        } else {
          // both m tiles of the unit share each dequantized B tile
          if (!mbar_wait(&s.tempty[0], aph ^ 1, kWhereMma)) { ok = false; break; }
          tc_fence_after();
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&s.ld_full[st], ph, kWhereMma)) { ok = false; break; }
            if (!mbar_wait(&s.b_full[bst], bph, kWhereMma)) { ok = false; break; }
            tc_fence_after();
            const uint32_t b_addr = smem_u32(b_tile(bst));
            for (int mi = 0; mi < t.mtiles; ++mi)
              issue(tmem + (uint32_t)(mi * kBN), smem_u32(a_tile(st, mi)), b_addr, kb);
            mma_commit(&s.ld_empty[st]);
            mma_commit(&s.b_empty[bst]);
            if (++bst == kBStages) { bst = 0; bph ^= 1; }
            if (++st == kSlots) { st = 0; ph ^= 1; }
          }
          if (!ok) break;
          mma_commit(&s.tfull[0]);
          aph ^= 1;
        }
      }
      mma_commit(&s.drain);
      mbar_wait(&s.drain, 0, kWhereDrain);
    }
  } else if (warp < 6 || warp >= 6 + kDqWarps) {
    // =============================== epilogue =============================
    // two warps per TMEM lane quarter: each drains one half of the 256 columns
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int half = warp >= 6 + kDqWarps ? 1 : 0;
    constexpr int kHalfCols = kBN / 2;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit t = decode_unit<CACHED>(s, E, nt, u);
      if (!CACHED) {
        if (!mbar_wait_warp(&s.tfull[0], aph, kWhereEpilogue)) { ok = false; break; }
        tc_fence_after();
      }
      for (int mi = 0; mi < t.mtiles; ++mi) {
        const int rows = min(kBM, t.rows_total - mi * kBM);
        const bool row_ok = r < rows;
        const int64_t row = (int64_t)t.row0 + mi * kBM + r;
        int col_acc = mi;
        if (CACHED) {
          if (!mbar_wait_warp(&s.tfull[acc], aph, kWhereEpilogue)) { ok = false; break; }
          tc_fence_after();
          col_acc = acc;
        }
        const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) +
                               (uint32_t)(col_acc * kBN + half * kHalfCols);
        const int col_base = t.j * kBN + half * kHalfCols;
        if (DSW)
          store_tile_dswiglu(tbase, row_ok, gu + row * 2 * K, dlhs + row * 2 * K, col_base, K,
                             kHalfCols / 32);
        else
          store_tile(tbase, r, row_ok, dlhs + row * K, col_base, K, kHalfCols / 32);
        if (CACHED) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_relaxed(&s.tempty[acc]);
          acc ^= 1;
          if (acc == 0) aph ^= 1;
        }
      }
      if (!CACHED && ok) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&s.tempty[0]);
        aph ^= 1;
      }
    }
  } else {
    // ========================== dequant warps ============================
    const int t = threadIdx.x - 192;          // 0..255
    const int sub = t & 3;
    int st = 0;
    uint32_t ph = 0;
    int bst = 0;
    uint32_t bph = 0;
    int64_t c_used = 0, fills = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit un = decode_unit<CACHED>(s, E, nt, u);
      const int64_t sbase = (int64_t)un.e * N;
      if (CACHED) {
        for (int kb = 0; kb < nkb; ++kb) {
          float sc16[16];
          load_scales16(scale, sbase, kb * kBK + sub * 16, N, sc16);
          if (!mbar_wait(&s.c_full, (uint32_t)(c_used & 1), kWhereDequant)) { ok = false; break; }
          // the previous unit's MMAs must be done with cache slot kb
          if (!mbar_wait(&s.b_empty[kb], (uint32_t)((fills & 1) ^ 1), kWhereDequant)) { ok = false; break; }
          dequant_tile(c_tile(0), b_tile(kb), sc16, t);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&s.b_full[kb]);
            mbar_arrive(&s.c_empty);
          }
          ++c_used;
        }
        ++fills;
      } else {
        for (int kb = 0; kb < nkb; ++kb) {
          float sc16[16];
          load_scales16(scale, sbase, kb * kBK + sub * 16, N, sc16);
          if (!mbar_wait(&s.ld_full[st], ph, kWhereDequant)) { ok = false; break; }
          if (!mbar_wait(&s.b_empty[bst], bph ^ 1, kWhereDequant)) { ok = false; break; }
          dequant_tile(c_tile(st), b_tile(bst), sc16, t);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&s.b_full[bst]);
            mbar_arrive(&s.ld_empty[st]);
          }
          if (++st == kSlots) { st = 0; ph ^= 1; }
          if (++bst == kBStages) { bst = 0; bph ^= 1; }
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool CACHED, bool DSW>
cudaError_t launch(const GmmDlhsArgs& a, int num_sms, cudaStream_t s) {
  auto kern = gmm_dlhs_kernel<CACHED, DSW>;
  constexpr size_t bytes = smem_bytes<CACHED>();
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (err != cudaSuccess) return err;
  kern<<<num_sms, kThreads, bytes, s>>>(a.tmA, a.tmC, a.scale, a.gs,
                                        static_cast<const __nv_bfloat16*>(a.gu),
                                        static_cast<__nv_bfloat16*>(a.dlhs), a.M, a.N, a.K, a.E);
  return cudaGetLastError();
}

}  // namespace dlhs
}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_dlhs)

cudaError_t fp8moe_launch_gmm_dlhs(const GmmDlhsArgs& a, int num_sms, int path, cudaStream_t s) {
  using namespace fp8moe::dlhs;
  if (path == 2) return fp8moe_launch_gmm_dlhs_pair(a, num_sms, s);
  const bool cached = path == 1;
  if (a.gu)
    return cached ? launch<true, true>(a, num_sms, s) : launch<false, true>(a, num_sms, s);
  return cached ? launch<true, false>(a, num_sms, s) : launch<false, false>(a, num_sms, s);
}
