// gmm_dlhs_pair.cu -- the default backward dLHS for contractions past 256.
//
//   dlhs[m, k] = sum_n dout[m, n] * bf16(f32(code[e(m), k, n]) * scale[e(m), n])
//
// "MoE: native FP8 QAT for routed-expert GMMs", Description and Implementation
// (the rhs_contract_dequant path): the weight codes are dequantized on chip and
// fed to the matmul, no BF16 weight copy reaches HBM, and the result is
// bit-identical to the BF16 GMM on the dequantized weight (and to the streaming
// and cached kernels of gmm_dlhs.cu).
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "groups.cuh"
#include "kernels.h"

// The dLHS transposed, dlhs^T[k, m] = sum_n w[k, n] * dout[m, n], on
// CTA pairs with the dequantized weight as the MMA's A operand in tensor memory.
//
// The streaming kernel (gmm_dlhs.cu) is bound by shared-memory bandwidth: per MMA
// cycle its tensor core reads the dequantized weight and both dout tiles from
// shared memory while TMA fills it and the dequant warps read codes and write
// BF16 there. Here the weight tile never touches shared memory as BF16: the
// dequant warps write it from registers straight into TMEM (tcgen05.st), where
// tcgen05.mma reads A. A unit is (expert, 256 token rows, 256 weight rows k);
// the pair's MMA is M = 256 (k: 128 per CTA, from each CTA's TMEM) by N = 256
// (token rows: 128 per CTA, from each CTA's shared memory), so each CTA moves
// 16 KB of dout and 8 KB of codes per 64-wide contraction step.
//   warp 0       TMA: this CTA's dout half [128 rows x 64] bf16 (K-major,
//                128-byte swizzle; completion counted on the even CTA's barrier)
//                and its codes [128 k x 64 n] (64-byte swizzle), 8 stages; the
//                step's 64 weight scales ride on the codes' barrier (a bulk
//                copy), so the dequant warps never wait on global loads.
//   warp 1       TMEM (512 columns: accumulator [0, 256), eight 32-column A
//                slots [256, 512)); in the even CTA the MMA-issuing thread.
//   warps 2, 3   idle (they complete the first warpgroup for setmaxnreg).
//   warps 4..11  epilogue: the accumulator holds dlhs^T (lane = k, column =
//                token row); two warps per TMEM lane quarter load 128 columns
//                each into registers, release the accumulator, then store
//                bf16 values (a warp writes 32 consecutive k of one row).
//   warps 12..27 dequant in four groups of four that take every fourth step;
//                in a group, one warp per TMEM lane quarter, each thread
//                converting the step's 64 codes of its k row,
//                bf16(f32(code) * scale[n]), into the A slot. A warp's chain
//                per step (barrier waits, conversions, the TMEM store round
//                trip) is longer than a step of MMAs, so each warp gets four
//                steps' time for it.
// setmaxnreg moves registers from the first warpgroup (32 each) and the dequant
// warps (56) to the epilogue warps (120), which hold a 128-column half of the
// accumulator as bf16 pairs.
// Publishing the odd CTA's A half to the even CTA's MMA: each dequant thread
// blocks in tcgen05.wait::st until its TMEM stores have completed, then its
// warp arrives on the even CTA's barrier. A cluster-scope release on that
// arrive would add about a microsecond per step (the release waits for the
// thread's memory operations at cluster scope) and there is nothing for it to
// publish: the stores are complete before the arrive is issued and the MMA that
// reads them is issued after the arrive is observed, so the arrive is relaxed.
namespace fp8moe {
namespace dlhs_pair {

constexpr int kBK = 64;                       // contraction (n) per step
constexpr int kRows = 128;                    // per CTA: k rows (A) and token rows (B)
constexpr int kUnitRows = 2 * kRows;          // token rows per unit = MMA N
constexpr int kUnitK = 2 * kRows;             // weight rows per unit = MMA M
constexpr int kStages = 8;
constexpr int kBBytes = kRows * kBK * 2;      // 16 KB dout half
constexpr int kCBytes = kRows * kBK;          // 8 KB codes
constexpr int kStageBytes = kBBytes + kCBytes;
constexpr int kScaleBytes = kBK * 4;          // a step's weight scales
constexpr int kASlots = 8;
constexpr int kACols = kBK / 2;               // TMEM columns per A slot (bf16 pairs)
constexpr int kDCols = kUnitRows;             // accumulator columns
constexpr int kTmemCols = 512;
static_assert(kDCols + kASlots * kACols == kTmemCols, "TMEM budget");
static_assert(kStages % 4 == 0 && kASlots % 4 == 0, "a dequant group owns every fourth slot");
constexpr int kCtlWarps = 4;                  // TMA, MMA, two idle: one warpgroup
constexpr int kEpiWarps = 8;                  // two per TMEM lane quarter
constexpr int kDqWarps = 16;                  // four per TMEM lane quarter
constexpr int kFirstEpi = kCtlWarps, kFirstDq = kCtlWarps + kEpiWarps;
constexpr int kThreads = (kCtlWarps + kEpiWarps + kDqWarps) * 32;   // 896
// 72 registers a thread at launch (65536 / 896, rounded down to 8); afterwards
// each SM sub-partition holds one warp of every warpgroup, so the shares must
// stay within 7 x 72 per sub-partition: 32 + 2 x 120 + 4 x 56 = 496.
constexpr int kCtlRegs = 32, kEpiRegs = 120, kDqRegs = 56;
static_assert(kCtlRegs + 2 * kEpiRegs + 4 * kDqRegs <= 7 * 72, "register hand-over");

struct Smem {
  uint64_t bfull[kStages];     // even CTA: both dout halves of the stage landed
  uint64_t cfull[kStages];     // this CTA's codes landed
  uint64_t sempty[kStages];    // this CTA's stage: MMAs done and codes read
  uint64_t afull[kASlots];     // even CTA: both CTAs wrote the A slot
  uint64_t aempty[kASlots];    // the MMAs reading the A slot completed
  uint64_t tfull;              // accumulator complete
  uint64_t tempty;             // even CTA: both CTAs' epilogues loaded it
  uint64_t drain;
  uint32_t tmem_base;
  int32_t T;
  int32_t total_units;
  int32_t begin[kMaxExperts];
  int32_t end[kMaxExperts];
  int32_t prefix[kMaxExperts + 1];
};
constexpr size_t kSmemBytes =
    1024 + (size_t)kStages * (kStageBytes + kScaleBytes) + sizeof(Smem);
static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");

struct Unit {
  int e, m0, rows, k0;    // rows: valid token rows of the unit (<= 256)
};

// Units: expert by expert, 256-row token tiles, weight-row tiles fastest (the
// token tile's dout is reused from L2 by the consecutive units).
__device__ __forceinline__ Unit decode_unit(const Smem& s, int E, int nkt, int u) {
  Unit r;
  r.e = find_bucket(s.prefix, E, u);
  const int local = u - s.prefix[r.e];
  const int mi = local / nkt;
  r.k0 = (local - mi * nkt) * kUnitK;
  r.m0 = s.begin[r.e] + mi * kUnitRows;
  r.rows = min(kUnitRows, s.end[r.e] - r.m0);
  return r;
}

// 16 codes of one k row (one 16-byte chunk) -> 8 bf16 pairs, bf16(f32(code) * scale).
__device__ __forceinline__ void dequant16(const uint4& c, const float* sc, uint32_t (&o)[8]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float f0, f1, f2, f3, p0, p1, p2, p3;
    half2_to_f32(e4m3x2_to_f16x2((uint16_t)(w[i] & 0xFFFFu)), f0, f1);
    half2_to_f32(e4m3x2_to_f16x2((uint16_t)(w[i] >> 16)), f2, f3);
    mul_f32x2(f0, f1, sc[4 * i], sc[4 * i + 1], p0, p1);
    mul_f32x2(f2, f3, sc[4 * i + 2], sc[4 * i + 3], p2, p3);
    o[2 * i] = f32x2_to_bf16x2(p0, p1);
    o[2 * i + 1] = f32x2_to_bf16x2(p2, p3);
  }
}

// dSwiGLU of one element: dh (f32 accumulator), g and u (bf16 bits).
__device__ __forceinline__ void dswiglu1(float d, uint16_t gb, uint16_t ub, uint16_t& dg_out,
                                         uint16_t& du_out) {
  const float g = __uint_as_float((uint32_t)gb << 16);
  const float u = __uint_as_float((uint32_t)ub << 16);
  const float sg = __frcp_rn(__fadd_rn(1.0f, __expf(-g)));
  const float dsilu = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sg))));
  const uint32_t p = f32x2_to_bf16x2(__fmul_rn(__fmul_rn(d, u), dsilu), __fmul_rn(d, __fmul_rn(g, sg)));
  dg_out = (uint16_t)(p & 0xFFFFu);
  du_out = (uint16_t)(p >> 16);
}

template <bool DSW>
__global__ void __launch_bounds__(kThreads, 1)
gmm_dlhs_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmC,
                     const float* __restrict__ scale, const int32_t* __restrict__ gs,
                     const __nv_bfloat16* __restrict__ gu, __nv_bfloat16* __restrict__ dlhs,
                     int64_t M, int N, int K, int E) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  float* const scales = reinterpret_cast<float*>(tiles + (size_t)kStages * kStageBytes);
  Smem& s = *reinterpret_cast<Smem*>(tiles + (size_t)kStages * (kStageBytes + kScaleBytes));
  auto b_tile = [&](int i) -> uint8_t* { return tiles + i * kStageBytes; };
  auto c_tile = [&](int i) -> uint8_t* { return tiles + i * kStageBytes + kBBytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const int nkt = (K + kUnitK - 1) / kUnitK;
  const int nkb = (N + kBK - 1) / kBK;

  if (warp == 0) {
    load_groups_warp0(gs, E, M, s.begin, s.end, &s.T, blockIdx.x == 0);
    __syncwarp();
    int32_t carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int32_t n = 0;
      if (e < E) n = ((s.end[e] - s.begin[e] + kUnitRows - 1) / kUnitRows) * nkt;
      int32_t incl = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
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
      for (int i = 0; i < kStages; ++i) {
        mbar_init(&s.bfull[i], 1);
        mbar_init(&s.cfull[i], 1);
        mbar_init(&s.sempty[i], 1 + kDqWarps / 4);   // the MMA commit + one dequant group
      }
      for (int i = 0; i < kASlots; ++i) {
        mbar_init(&s.afull[i], kDqWarps / 2);    // one dequant group of each CTA
        mbar_init(&s.aempty[i], 1);
      }
      mbar_init(&s.tfull, 1);
      mbar_init(&s.tempty, 2 * kEpiWarps);
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

  if (warp < kCtlWarps) setmaxnreg_dec<kCtlRegs>();
  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int u = cluster; u < total && ok; u += nclusters) {
        const Unit t = decode_unit(s, E, nkt, u);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(&s.sempty[st], ph ^ 1, kWhereProducer)) { ok = false; break; }
          if (rank == 0) mbar_arrive_expect_tx(&s.bfull[st], 2 * kBBytes);
          tma_load_2d_pair(b_tile(st), &tmA, mapa_shared(smem_u32(&s.bfull[st]), 0), kb * kBK,
                           t.m0 + rank * kRows);
          // N % 16 == 0: the in-range scales of a step are a multiple of 64 bytes
          const uint32_t sbytes = (uint32_t)min(kBK, N - kb * kBK) * 4u;
          mbar_arrive_expect_tx(&s.cfull[st], kCBytes + sbytes);
          tma_load_3d(c_tile(st), &tmC, &s.cfull[st], kb * kBK, t.k0 + rank * kRows, t.e);
          bulk_load(scales + st * kBK, scale + (int64_t)t.e * N + kb * kBK, sbytes, &s.cfull[st]);
          ++issued;
          if (++st == kStages) { st = 0; ph ^= 1; }
        }
      }
      // drain: every copy into this CTA (and, for the even CTA, both dout
      // halves) landed before either CTA may exit
      const int64_t n_last = issued < kStages ? issued : kStages;
      for (int64_t i = 1; i <= n_last; ++i) {
        const int64_t idx = issued - i;
        const uint32_t par = (uint32_t)((idx / kStages) & 1);
        mbar_wait(&s.cfull[idx % kStages], par, kWhereDrain);
        if (rank == 0) mbar_wait_cluster(&s.bfull[idx % kStages], par, kWhereDrain);
      }
    }
  } else if (warp == 1) {
    // ============================== MMA issuer ============================
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = make_idesc(1, 1, 0, 0, kUnitK, kUnitRows);
      int st = 0, as = 0;
      uint32_t ph = 0, aph = 0, tph = 0;
      bool ok = true;
      for (int u = cluster; u < total && ok; u += nclusters) {
        if (!mbar_wait_cluster(&s.tempty, tph ^ 1, kWhereMma)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(&s.bfull[st], ph, kWhereMma)) { ok = false; break; }
          if (!mbar_wait_cluster(&s.afull[as], aph, kWhereMma)) { ok = false; break; }
          tc_fence_after();
          const uint32_t b_addr = smem_u32(b_tile(st));
          const uint32_t a_col = tmem + (uint32_t)(kDCols + as * kACols);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = make_desc(b_addr + kk * 32, 16, 1024, kSwizzle128B);
            mma_f16_pair_ts(tmem, a_col + kk * 8, bd, idesc, (kb | kk) != 0);
          }
          mma_commit_pair(&s.sempty[st]);
          mma_commit_pair(&s.aempty[as]);
          if (++st == kStages) { st = 0; ph ^= 1; }
          if (++as == kASlots) { as = 0; aph ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair(&s.tfull);
        tph ^= 1;
      }
      // all MMAs complete (in both CTAs' TMEM) before TMEM may be released
      mma_commit_pair(&s.drain);
    }
    if (lane == 0) mbar_wait_cluster(&s.drain, 0, kWhereDrain);
  } else if (warp < kCtlWarps) {
    // idle
  } else if (warp < kFirstDq) {
    // =============================== epilogue =============================
    setmaxnreg_inc<kEpiRegs>();
    const int quarter = warp & 3;
    const int half = (warp - kFirstEpi) >> 2;      // token-row columns [128 half, +128)
    const int r = quarter * 32 + lane;             // k row inside this CTA's 128
    const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(half * 128);
    uint32_t tph = 0;
    for (int u = cluster; u < total; u += nclusters) {
      const Unit t = decode_unit(s, E, nkt, u);
      const int k = t.k0 + rank * kRows + r;
      const int jn = min(128, t.rows - half * 128);   // valid token rows of this half
      const int64_t row0 = (int64_t)t.m0 + half * 128;
      if (DSW) {
        // dSwiGLU needs the f32 accumulator, 128 values a thread: too many to hold
        // in registers, so the epilogue works through the accumulator 16 columns
        // at a time while holding it, loading each chunk's g and u one chunk ahead
        // (the first chunk's before the accumulator is ready)
        const bool kin = k < K;
        const uint16_t* gub = reinterpret_cast<const uint16_t*>(gu) + row0 * 2 * K + k;
        uint16_t* ob = reinterpret_cast<uint16_t*>(dlhs) + row0 * 2 * K + k;
        auto fetch = [&](int c, uint32_t (&g)[16], uint32_t (&uu)[16]) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int jj = c * 16 + j;
            g[j] = 0u;
            uu[j] = 0u;
            if (kin && jj < jn) {
              g[j] = __ldg(gub + (int64_t)jj * 2 * K);
              uu[j] = __ldg(gub + (int64_t)jj * 2 * K + K);
            }
          }
        };
        uint32_t g0[16], u0[16];
        fetch(0, g0, u0);
        if (!mbar_wait_warp_cluster(&s.tfull, tph, kWhereEpilogue)) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t g1[16], u1[16];
          if (c + 1 < 8) fetch(c + 1, g1, u1);
          uint32_t w[16];
          tmem_ld16(tbase + c * 16, w);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int jj = c * 16 + j;
            if (kin && jj < jn) {
              uint16_t dg, du;
              dswiglu1(__uint_as_float(w[j]), (uint16_t)g0[j], (uint16_t)u0[j], dg, du);
              ob[(int64_t)jj * 2 * K] = dg;
              ob[(int64_t)jj * 2 * K + K] = du;
            }
          }
          if (c + 1 < 8) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              g0[j] = g1[j];
              u0[j] = u1[j];
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&s.tempty), 0));
        tph ^= 1;
        continue;
      }
      if (!mbar_wait_warp_cluster(&s.tfull, tph, kWhereEpilogue)) break;
      tc_fence_after();
      // the whole 128-column half in registers as bf16 pairs
      uint32_t v[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[32];
        tmem_ld32(tbase + c * 32, w);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[c * 16 + i] = f32x2_to_bf16x2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
      }
      tc_fence_before();
      __syncwarp();
      // the even CTA's MMA thread waits for the epilogue warps of both CTAs
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&s.tempty), 0));
      tph ^= 1;
      if (k < K && jn > 0) {
        uint16_t* ob = reinterpret_cast<uint16_t*>(dlhs) + row0 * K + k;
#pragma unroll
        for (int j = 0; j < 128; ++j) {
          if (j < jn) *ob = (uint16_t)(v[j >> 1] >> (16 * (j & 1)));
          ob += K;
        }
      }
    }
  } else {
    // ========================== dequant warps ============================
    setmaxnreg_dec<kDqRegs>();
    const int quarter = warp & 3;
    const int group = (warp - kFirstDq) >> 2;      // takes the steps i with i % 4 == group
    const int r = quarter * 32 + lane;             // k row inside this CTA's 128
    const uint32_t tcol = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)kDCols;
    // 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3)
    const int x = (r >> 1) & 3;
    const uint32_t peer_afull = mapa_shared(smem_u32(&s.afull[0]), 0);
    uint32_t i = 0;                                // global step index (stages and A slots)
    bool ok = true;
    for (int u = cluster; u < total && ok; u += nclusters) {
      for (int kb = 0; kb < nkb; ++kb, ++i) {
        if ((int)(i & 3) != group) continue;
        const int st = (int)(i % kStages), as = (int)(i % kASlots);
        const uint32_t ph = (i / kStages) & 1, aph = (i / kASlots) & 1;
        if (!mbar_wait(&s.cfull[st], ph, kWhereDequant)) { ok = false; break; }
        // the MMAs that read this A slot completed (commit of the even CTA's MMA
        // thread, multicast to both CTAs)
        if (!mbar_wait(&s.aempty[as], aph ^ 1, kWhereDequant)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* crow = c_tile(st) + r * 64;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t o[16];
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = 2 * h + jj;
            const uint4 c = *reinterpret_cast<const uint4*>(crow + ((j ^ x) << 4));
            // N % 16 == 0: a 16-column group is fully in range or fully out (past
            // N the slot holds an earlier step's scales and the codes are zero)
            float sc[16];
            const bool in = kb * kBK + j * 16 < N;
            const float4* p = reinterpret_cast<const float4*>(scales + st * kBK + j * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 f = in ? p[q] : make_float4(0.f, 0.f, 0.f, 0.f);
              sc[4 * q] = f.x; sc[4 * q + 1] = f.y; sc[4 * q + 2] = f.z; sc[4 * q + 3] = f.w;
            }
            uint32_t oj[8];
            dequant16(c, sc, oj);
#pragma unroll
            for (int q = 0; q < 8; ++q) o[8 * jj + q] = oj[q];
          }
          tmem_st16(tcol + (uint32_t)(as * kACols + h * 16), o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sempty[st]);   // codes and scales read
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(&s.afull[as]);
          else mbar_arrive_cluster_relaxed(peer_afull + (uint32_t)(as * sizeof(uint64_t)));
        }
      }
    }
  }

  __syncthreads();
  cluster_sync();      // both CTAs done with TMEM, shared memory and barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <bool DSW>
cudaError_t launch(const GmmDlhsArgs& a, int num_sms, cudaStream_t s) {
  auto kern = gmm_dlhs_pair_kernel<DSW>;
  // the register hand-over needs the full launch allocation: refuse a build whose
  // kernel was compiled with fewer registers than the split assumes
  cudaFuncAttributes fa;
  cudaError_t err = cudaFuncGetAttributes(&fa, kern);
  if (err != cudaSuccess) return err;
  if (fa.numRegs * (kThreads / 32) <
      kCtlRegs * kCtlWarps + kEpiRegs * kEpiWarps + kDqRegs * kDqWarps)
    return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_sms & ~1), 1, 1);   // whole CTA pairs, one CTA per SM
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmCp, a.scale, a.gs,
                           static_cast<const __nv_bfloat16*>(a.gu),
                           static_cast<__nv_bfloat16*>(a.dlhs), a.M, a.N, a.K, a.E);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace dlhs_pair
}  // namespace fp8moe

FP8MOE_DEFINE_STATUS_TAKE(fp8moe_status_take_dlhs_pair)

cudaError_t fp8moe_launch_gmm_dlhs_pair(const GmmDlhsArgs& a, int num_sms, cudaStream_t s) {
  using namespace fp8moe::dlhs_pair;
  return a.gu ? launch<true>(a, num_sms, s) : launch<false>(a, num_sms, s);
}
