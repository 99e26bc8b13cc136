// gmm_fwd.cu -- ragged grouped matmul forward on tcgen05 tensor cores, CTA pairs.
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
// Design: persistent clusters of two CTAs (one CTA per SM). A work unit is
// (expert, pair of 128-row m tiles, 256-column n tile); the pair computes the
// 256 x 256 tile with tcgen05.mma.cta_group::2 (M = 256, N = 256) issued by the
// even CTA. Each CTA loads only its own 128 A rows and one 128-column half of
// the B tile, so a CTA moves 32 KB per 128-byte K step instead of the 48 KB a
// single-CTA 128 x 256 tile needs: the tensor cores stay fed from L2.
//   warp 0      TMA producer of this CTA's A rows (K-major, 128-byte swizzle)
//               and B half (MN-major, 128-byte swizzle), 6 stages of 32 KB;
//               completion is counted on the even CTA's barrier.
//   warp 1      TMEM allocation for the pair (512 columns = two 128 x 256 f32
//               accumulators per CTA); in the even CTA, the MMA-issuing thread.
//   warps 2..    epilogue of this CTA's 128 rows: tcgen05.ld, scales, SwiGLU,
//               bf16, row-masked 32-byte stores; the second accumulator lets
//               the next tile's MMAs run meanwhile. Four warps (one per TMEM
//               lane quarter) for the plain forward; eight (two per quarter,
//               half the columns each) for SwiGLU and the block mode, whose
//               heavier epilogues would otherwise hold up the MMAs.
// SwiGLU: the even CTA's B half is the gate columns, the odd CTA's the matching
// up columns, so accumulator columns [0, 128) are gate and [128, 256) up.
// Units are enumerated expert by expert, n tile by n tile, pairs fastest, so
// that concurrently running clusters share weight tiles through L2. Each CTA
// derives the ragged layout from group_sizes itself; tiles begin at their
// group's first row and rows past the group end are computed but never stored.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "groups.cuh"
#include "kernels.h"

namespace fp8moe {
namespace fwd {

constexpr int kStages = 6;
constexpr int kBM = 128;                    // rows per CTA (M = 256 per pair)
constexpr int kBN = 256;                    // accumulator columns (MMA N)
constexpr int kABytes = kBM * 128;          // 16 KB: 128 rows x 128 bytes of K
constexpr int kBBytes = 128 * 128;          // 16 KB: this CTA's 128 columns x 128 bytes of K
constexpr int kStageBytes = kABytes + kBBytes;
// Epilogue warps: one per TMEM lane quarter (4), or two per quarter with half the
// columns each (8) where the epilogue is heavy enough to hold up the MMAs
// otherwise (SwiGLU; the block mode's per-block folding). Registers are budgeted
// per SM sub-partition: 10 warps put 3 on two of them, so a thread may hold
// 16384 / (3 * 32) -> 168 registers (launch bounds of 384 threads give the
// compiler that cap); 6 warps put at most 2 on one, which leaves the cap at 255.
template <bool SWIGLU, bool BLK>
struct Epi {
  static constexpr int kWarps = (SWIGLU || BLK) ? 8 : 4;
  static constexpr int kHalves = kWarps / 4;
  static constexpr int kThreads = (2 + kWarps) * 32;
  static constexpr int kRegBudgetThreads = kWarps == 8 ? 384 : 192;
};
constexpr int kTmemCols = 512;

struct Smem {
  uint64_t full[kStages];      // even CTA: both CTAs' tiles of the stage landed
  uint64_t empty[kStages];     // both CTAs: the stage's MMAs completed
  uint64_t tfull[2];           // both CTAs: accumulator ready
  uint64_t tempty[2];          // even CTA: both CTAs' epilogues drained it
  uint64_t drain;
  uint32_t tmem_base;
  int32_t T;
  int32_t total_units;
  float sw[2][kBN];
  int32_t begin[kMaxExperts];
  int32_t end[kMaxExperts];
  int32_t prefix[kMaxExperts + 1];
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");

struct Unit {
  int e, row0, rows, j;   // row0 / rows: this CTA's m tile (rows may be <= 0)
};

__device__ __forceinline__ Unit decode_unit(const Smem& s, int E, int nt, int u, int rank) {
  Unit r;
  r.e = find_bucket(s.prefix, E, u);
  const int mt = (s.end[r.e] - s.begin[r.e] + kBM - 1) / kBM;
  const int mtp = (mt + 1) / 2;
  const int local = u - s.prefix[r.e];
  r.j = local / mtp;
  const int p = local - r.j * mtp;
  r.row0 = s.begin[r.e] + (2 * p + rank) * kBM;
  r.rows = min(kBM, s.end[r.e] - r.row0);
  return r;
}

// Block mode (BLK, FP8 only): per-512-column block activation scales sx [M, nblk]
// and bf16 accumulation across blocks (the ops-level lhs_quant_block_size = 512
// option of "MoE: native FP8 QAT for routed-expert GMMs", Implementation). The
// MMA starts a fresh TMEM accumulator every 512 K columns (four 128-column
// steps) and alternates the two accumulators block by block; the epilogue warps
// fold each block into a bf16 register accumulator, acc = bf16(acc + P * s_b),
// and apply the channel scales (and SwiGLU) once at the end of the unit.
constexpr int kBlkSteps = 4;      // 128-column K steps per 512-column block

// 16 bf16 values (8 words) of one output row, 16-byte stores; columns past
// Nout are skipped.
__device__ __forceinline__ void store_row_chunk(const uint32_t* o, bool row_ok,
                                                __nv_bfloat16* __restrict__ orow, int col0,
                                                int Nout) {
  if (!row_ok) return;
  if (col0 + 32 <= Nout) {
    st_global_64B(orow + col0, o);
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(orow);
#pragma unroll
    for (int q = 0; q < 32; ++q)
      if (col0 + q < Nout) dst[col0 + q] = (uint16_t)(o[q / 2] >> (16 * (q & 1)));
  }
}

// FP8: a 128-byte swizzle row holds 128 K values of A (or 128 N values of B);
// BF16: 64.
template <bool FP8, bool SWIGLU, bool BLK>
__global__ void __launch_bounds__(Epi<SWIGLU, BLK>::kRegBudgetThreads, 1)
gmm_fwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const float* __restrict__ sx, const float* __restrict__ scale,
               const int32_t* __restrict__ gs, __nv_bfloat16* __restrict__ out, int64_t M, int K,
               int N, int E, int e0, int e1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  Smem& s = *reinterpret_cast<Smem*>(tiles + (size_t)kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

  constexpr int kElemsPerRow = FP8 ? 128 : 64;        // elements per 128-byte row
  const int Nout = SWIGLU ? N / 2 : N;
  const int nt = SWIGLU ? (Nout + 127) / 128 : (N + kBN - 1) / kBN;
  const int nkb = (K + kElemsPerRow - 1) / kElemsPerRow;

  // ---- set-up: ragged layout, unit prefix (units = m-tile pairs), barriers, TMEM
  if (warp == 0) {
    load_groups_warp0(gs, E, M, s.begin, s.end, &s.T, blockIdx.x == 0);
    __syncwarp();
    int32_t carry = 0;
    for (int base = 0; base < E; base += 32) {
      int e = base + lane;
      int32_t n = 0;
      if (e >= e0 && e < e1) n = (((s.end[e] - s.begin[e] + kBM - 1) / kBM + 1) / 2) * nt;
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
        mbar_init(&s.tempty[i], 2 * Epi<SWIGLU, BLK>::kWarps);   // one lane per epilogue warp, both CTAs
      }
      mbar_init(&s.drain, 1);
      fence_mbar_init();
    }
    __syncwarp();
    tmem_alloc_pair(&s.tmem_base, kTmemCols);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync();      // the peer's barriers exist before anyone signals them
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
      for (int u = cluster; u < total && ok; u += nclusters) {
        const Unit t = decode_unit(s, E, nt, u, rank);
        int nb;
        if (SWIGLU) nb = (rank ? Nout : 0) + t.j * 128;
        else nb = t.j * kBN + rank * 128;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(&s.empty[st], ph ^ 1, kWhereProducer)) { ok = false; break; }
          // the even CTA's barrier counts the bytes of both CTAs
          if (rank == 0) mbar_arrive_expect_tx(&s.full[st], 2 * kStageBytes);
          const uint32_t bar = mapa_shared(smem_u32(&s.full[st]), 0);
          uint8_t* a = tiles + st * kStageBytes;
          uint8_t* b = a + kABytes;
          const int k0 = kb * kElemsPerRow;
          tma_load_2d_pair(a, &tmA, bar, k0, t.row0);
          if (FP8) {
            tma_load_3d_pair(b, &tmB, bar, nb, k0, t.e);
          } else {
            // bf16: two 64-column boxes of 64 K rows (8 KB each)
            tma_load_3d_pair(b, &tmB, bar, nb, k0, t.e);
            tma_load_3d_pair(b + 8192, &tmB, bar, nb + 64, k0, t.e);
          }
          ++issued;
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
      }
      // drain (even CTA): every load of both CTAs landed before either may exit
      if (rank == 0) {
        int64_t n_last = issued < kStages ? issued : kStages;
        for (int64_t i = 1; i <= n_last; ++i) {
          int64_t idx = issued - i;
          mbar_wait_cluster(&s.full[idx % kStages], (uint32_t)((idx / kStages) & 1), kWhereDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ============================== MMA issuer ============================
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = FP8 ? make_idesc(0, 0, 0, 1, 2 * kBM, kBN)
                                     : make_idesc(1, 1, 0, 1, 2 * kBM, kBN);
      // B (MN-major), this CTA's 128 columns: FP8 one 128-column atom; BF16
      // two 64-column atoms 8 KB apart.
      constexpr uint32_t kBLbo = FP8 ? 16384 : 8192;
      // one MMA consumes 32 bytes of K: FP8 32 K values (= 32 B-rows), BF16 16
      constexpr uint32_t kBStep = FP8 ? 32 * 128 : 16 * 128;
      int st = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (int u = cluster; u < total && ok; u += nclusters) {
        if (!BLK) {
          if (!mbar_wait_cluster(&s.tempty[acc], aph ^ 1, kWhereMma)) { ok = false; break; }
          tc_fence_after();
        }
        uint32_t d = tmem + (uint32_t)(acc * kBN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (BLK && kb % kBlkSteps == 0) {   // a fresh accumulator per 512-column block
            if (!mbar_wait_cluster(&s.tempty[acc], aph ^ 1, kWhereMma)) { ok = false; break; }
            tc_fence_after();
            d = tmem + (uint32_t)(acc * kBN);
          }
          if (!mbar_wait_cluster(&s.full[st], ph, kWhereMma)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + st * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = make_desc(a_addr + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = make_desc(b_addr + kk * kBStep, kBLbo, 1024, kSwizzle128B);
            const bool accumulate = BLK ? ((kb % kBlkSteps) | kk) != 0 : (kb | kk) != 0;
            if (FP8) mma_f8f6f4_pair(d, ad, bd, idesc, accumulate);
            else mma_f16_pair(d, ad, bd, idesc, accumulate);
          }
          mma_commit_pair(&s.empty[st]);
          if (++st == kStages) { st = 0; ph ^= 1; }
          if (BLK && (kb % kBlkSteps == kBlkSteps - 1 || kb == nkb - 1)) {
            mma_commit_pair(&s.tfull[acc]);
            acc ^= 1;
            if (acc == 0) aph ^= 1;
          }
        }
        if (!ok) break;
        if (!BLK) {
          mma_commit_pair(&s.tfull[acc]);
          acc ^= 1;
          if (acc == 0) aph ^= 1;
        }
      }
      // all MMAs complete (in both CTAs' TMEM) before TMEM may be released
      mma_commit_pair(&s.drain);
    }
    if (lane == 0) mbar_wait_cluster(&s.drain, 0, kWhereDrain);
  } else {
    // =============================== epilogue =============================
    const int et = threadIdx.x - 64;                 // epilogue thread
    const int quarter = warp & 3;                    // TMEM lanes 32*quarter ..
    constexpr int kEpiThreads = Epi<SWIGLU, BLK>::kWarps * 32;
    constexpr int kHalves = Epi<SWIGLU, BLK>::kHalves;
    const int half = (warp - 2) >> 2;                // which half of the columns (8 warps)
    const int r = quarter * 32 + lane;               // row inside this CTA's tile
    int acc = 0;
    uint32_t aph = 0;
    int sb = 0;
    // A timed-out wait marks the warp failed; it keeps iterating (without
    // touching TMEM) so that every epilogue thread passes the same named barriers.
    bool failed = false;
    for (int u = cluster; u < total; u += nclusters) {
      const Unit t = decode_unit(s, E, nt, u, rank);
      // per-column scales of this tile's 256 accumulator columns
      if (FP8) {
#pragma unroll
        for (int c = et; c < kBN; c += kEpiThreads) {
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
      named_bar_sync(1, kEpiThreads);
      const bool row_ok = r < t.rows;
      const int64_t row = (int64_t)t.row0 + r;
      if (BLK) {
        // ---- block mode: fold every block's accumulator into bf16 registers
        // bf16 pairs of this thread's 128 columns: SwiGLU gate chunks 2 half,
        // 2 half + 1 in accb[0..31] and the matching up chunks in accb[32..63];
        // otherwise chunks 4 half .. 4 half + 3
        uint32_t accb[kBN / 4];
#pragma unroll
        for (int i = 0; i < kBN / 4; ++i) accb[i] = 0u;
        const int nblk = (nkb + kBlkSteps - 1) / kBlkSteps;
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        for (int b = 0; b < nblk; ++b) {
          const float sbk = row_ok ? __ldg(sx + row * nblk + b) : 0.0f;
          if (!failed && !mbar_wait_warp_cluster(&s.tfull[acc], aph, kWhereEpilogue)) failed = true;
          if (!failed) {
            tc_fence_after();
            if (t.rows > 0) {
              const uint32_t tbase = trow + (uint32_t)(acc * kBN);
#pragma unroll
              for (int c = 0; c < kBN / 64; ++c) {
                const int tc = SWIGLU ? (c < 2 ? 2 * half + c : 4 + 2 * half + (c - 2)) : 4 * half + c;
                uint32_t v[32];
                tmem_ld32(tbase + tc * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  float f0 = bf16lo_to_f32(accb[c * 16 + i]), f1 = bf16hi_to_f32(accb[c * 16 + i]);
                  f0 = __fmaf_rn(__uint_as_float(v[2 * i]), sbk, f0);
                  f1 = __fmaf_rn(__uint_as_float(v[2 * i + 1]), sbk, f1);
                  accb[c * 16 + i] = f32x2_to_bf16x2(f0, f1);
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&s.tempty[acc]), 0));
          }
          acc ^= 1;
          if (acc == 0) aph ^= 1;
        }
        if (!failed && t.rows > 0) {
          __nv_bfloat16* orow = out + row * Nout;
          if (SWIGLU) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int oc = 2 * half + c;        // output chunk of 32 columns
              uint32_t o[16];
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float y[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint32_t gw = accb[(c * 32 + i) / 2], uw = accb[32 + (c * 32 + i) / 2];
                  const float gg = __fmul_rn(h ? bf16hi_to_f32(gw) : bf16lo_to_f32(gw),
                                             s.sw[sb][oc * 32 + i + h]);
                  const float uu = __fmul_rn(h ? bf16hi_to_f32(uw) : bf16lo_to_f32(uw),
                                             s.sw[sb][128 + oc * 32 + i + h]);
                  y[h] = __fmul_rn(__fdiv_rn(gg, __fadd_rn(1.0f, expf(-gg))), uu);
                }
                o[i / 2] = f32x2_to_bf16x2(y[0], y[1]);
              }
              store_row_chunk(o, row_ok, orow, t.j * 128 + oc * 32, Nout);
            }
          } else {
#pragma unroll
            for (int c = 0; c < kBN / 64; ++c) {
              const int oc = 4 * half + c;
              uint32_t o[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                o[i] = f32x2_to_bf16x2(__fmul_rn(bf16lo_to_f32(accb[c * 16 + i]), s.sw[sb][oc * 32 + 2 * i]),
                                       __fmul_rn(bf16hi_to_f32(accb[c * 16 + i]),
                                                 s.sw[sb][oc * 32 + 2 * i + 1]));
              store_row_chunk(o, row_ok, orow, t.j * kBN + oc * 32, Nout);
            }
          }
        }
        sb ^= 1;
        continue;
      }
      const float sxr = (FP8 && row_ok) ? __ldg(sx + row) : 1.0f;
      if (!failed && !mbar_wait_warp_cluster(&s.tfull[acc], aph, kWhereEpilogue)) failed = true;
      if (failed) {
        acc ^= 1;
        if (acc == 0) aph ^= 1;
        sb ^= 1;
        continue;
      }
      tc_fence_after();
      if (t.rows > 0) {
        const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
        __nv_bfloat16* orow = out + row * Nout;
        constexpr int kChunks = (SWIGLU ? 4 : 8) / kHalves;   // this warp's columns
#pragma unroll 1
        for (int cc = 0; cc < kChunks; ++cc) {
          const int c = half * kChunks + cc;
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
          store_row_chunk(o, row_ok, orow, col0, Nout);
        }
      }
      tc_fence_before();
      __syncwarp();
      // the even CTA's MMA thread waits for the epilogue warps of both CTAs
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&s.tempty[acc]), 0));
      acc ^= 1;
      if (acc == 0) aph ^= 1;
      sb ^= 1;
    }
  }

  __syncthreads();
  cluster_sync();      // both CTAs done with TMEM, shared memory and barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <bool FP8, bool SWIGLU, bool BLK>
cudaError_t launch(const GmmFwdArgs& a, int num_sms, cudaStream_t s) {
  auto kern = gmm_fwd_kernel<FP8, SWIGLU, BLK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_sms & ~1), 1, 1);   // whole CTA pairs, one CTA per SM
  cfg.blockDim = dim3(Epi<SWIGLU, BLK>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.sx, a.scale, a.gs,
                           static_cast<__nv_bfloat16*>(a.out), a.M, a.K, a.N, a.E, a.e0, a.e1);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace fwd
}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_gmm_fwd)

cudaError_t fp8moe_launch_gmm_fp8_fwd(const GmmFwdArgs& a, int num_sms, cudaStream_t s) {
  using namespace fp8moe::fwd;
  if (a.blk)
    return a.swiglu ? launch<true, true, true>(a, num_sms, s) : launch<true, false, true>(a, num_sms, s);
  return a.swiglu ? launch<true, true, false>(a, num_sms, s) : launch<true, false, false>(a, num_sms, s);
}

cudaError_t fp8moe_launch_gmm_bf16_fwd(const GmmFwdArgs& a, int num_sms, cudaStream_t s) {
  using namespace fp8moe::fwd;
  return a.swiglu ? launch<false, true, false>(a, num_sms, s) : launch<false, false, false>(a, num_sms, s);
}
