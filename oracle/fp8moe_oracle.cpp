// fp8moe_oracle.cpp -- CPU oracle for the native-FP8 MoE grouped-matmul path.
//
// TEST INFRASTRUCTURE ONLY. This file is the slow, plain, obviously-correct
// definition that the CUDA library is checked against. It shares no code, header,
// table or constant generator with the CUDA path, and nothing in the product
// imports it: only the test suite, the smoke check and the benchmark's CPU
// baseline load it.
//
// Sources (web pages; each function names the passage it follows):
//   [NQ]  "MoE: native FP8 QAT for routed-expert GMMs (FP8 forward + FP8-weight
//          backward dLHS)" -- sections Description, Data flow, Implementation,
//          Tests, and its review threads.
//   [DQ]  "MoE fp8 backward: in-kernel drhs operand quantization + configurable
//          gradient dtype" -- section What.
//   [SM]  "Fix fp8 MoE on the sparse_matmul path" -- section Fix (names the
//          forward dtype float8_e4m3fn).
//   [DQ] What also makes the gradient fp8 dtype configurable, e5m2 (the
//   recipe's default) or e4m3: here the tgmm's dout operand may be e5m2.
//   The SwiGLU backward (dSwiGLU) is the derivative of silu(g) * u written out;
//   [NQ] Implementation names the op that fuses it into the wo GMM
//   (gmm_dswiglu_fp8).
//
// Floating point: all sums are taken in double. Products of two e4m3 values are
// multiples of 2^-18 with magnitude <= 448^2, so any sum of up to 2^17 of them is
// exact in double whatever the order; the forward GMM accumulator is therefore the
// exact value, rounded once at the end. With an e5m2 operand (tgmm, multiples of
// 2^-16 up to 57344) a 128-term segment dot product can need more than 53 bits;
// it is then within 128 * 2^-53 relative of the exact value. Quantization decisions (scales, codes) are
// taken in f32, the precision the pages fix for the activation scale.
//
// Data-dependent bounds: group sizes are clamped like the library documents
// (negative sizes count as 0, rows are clipped at the static buffer size M). Every
// read of an input row goes through a guarded accessor that counts reads of rows
// at or past T = sum(group_sizes); each entry point returns that count (0 = the
// tail was never read).
//
// Parity pins: see tests/test_oracle_*.py. Everything here is pinned except the
// model-level relative-error figures quoted on [NQ] (needs the rollout kernel).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <atomic>
#include <thread>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---------------------------------------------------------------------------
// bf16 <-> f32.  bf16 is the top half of an IEEE binary32.
// ---------------------------------------------------------------------------
float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round a double to the nearest bf16, ties to even, in ONE rounding (no detour
// through f32).  NaN -> 0x7FC0 with the sign kept; overflow -> +-Inf.
uint16_t f64_to_bf16_rne(double d) {
  if (std::isnan(d)) return std::signbit(d) ? 0xFFC0 : 0x7FC0;
  uint16_t sign = std::signbit(d) ? 0x8000 : 0;
  double a = std::fabs(d);
  if (a == 0.0) return sign;
  // bf16: 8 significant bits, exponent range of binary32 (min normal 2^-126,
  // subnormal quantum 2^-133, max finite (2 - 2^-7) * 2^127).
  int e;
  std::frexp(a, &e);            // a = f * 2^e, f in [0.5, 1)
  int exp_unbiased = e - 1;     // a in [2^(e-1), 2^e)
  int q_exp = std::max(exp_unbiased, -126) - 7;   // quantum of the bf16 grid here
  double quantum = std::ldexp(1.0, q_exp);
  double n = a / quantum;       // exact: scaling by a power of two
  double fl = std::floor(n);
  double rem = n - fl;
  double r;
  if (rem > 0.5) r = fl + 1.0;
  else if (rem < 0.5) r = fl;
  else r = (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double v = r * quantum;
  const double max_finite = std::ldexp(255.0, 127 - 7);   // 0x7F7F
  if (v > max_finite) return sign | 0x7F80;               // round to Inf
  // Encode v (exactly representable) into bits.
  float vf = (float)v;   // exact: v has <= 8 significant bits and is in f32 range
  uint32_t u;
  std::memcpy(&u, &vf, 4);
  return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

uint16_t f32_to_bf16_rne(float f) { return f64_to_bf16_rne((double)f); }

// ---------------------------------------------------------------------------
// OCP float8 e4m3fn  ([SM] Fix: the forward dtype is float8_e4m3fn; [NQ]
// Implementation: the activation scale divides by 448, the e4m3fn maximum).
// Layout s.eeee.mmm, exponent bias 7, no infinities, S.1111.111 is NaN,
// exponent field 0 holds subnormals m * 2^-9.
// ---------------------------------------------------------------------------
double e4m3_decode(uint8_t c) {
  int s = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return std::nan("");
  if (e == 0) v = std::ldexp((double)m, -9);
  else v = std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

// The 127 non-negative finite values, code 0x00 .. 0x7E, ascending.
struct E4m3Table {
  double v[127];
  E4m3Table() { for (int c = 0; c < 127; ++c) v[c] = e4m3_decode((uint8_t)c); }
};
const E4m3Table& e4m3_table() { static E4m3Table t; return t; }

// Round an f32 to e4m3fn: nearest value, ties to the even code; magnitudes past
// the largest finite value (including infinities) saturate to +-448; NaN -> 0x7F.
uint8_t e4m3_encode(float f) {
  if (std::isnan(f)) return 0x7F;
  uint8_t sign = std::signbit(f) ? 0x80 : 0x00;
  double a = std::fabs((double)f);
  const double* v = e4m3_table().v;
  if (a >= v[126]) return sign | 126;
  // Largest code c with v[c] <= a (binary search over the ascending table).
  int lo = 0, hi = 126;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (v[mid] <= a) lo = mid; else hi = mid;
  }
  int c = lo;
  double below = v[c], above = v[c + 1];
  double d_lo = a - below, d_hi = above - a;
  int pick;
  if (d_lo < d_hi) pick = c;
  else if (d_hi < d_lo) pick = c + 1;
  else pick = (c % 2 == 0) ? c : c + 1;   // tie: even code = even mantissa LSB
  return sign | (uint8_t)pick;
}

// ---------------------------------------------------------------------------
// OCP float8 e5m2 ([DQ] What: the gradient fp8 dtype, e5m2 by default).
// Layout s.eeeee.mm, exponent bias 15, exponent field 0 holds subnormals
// m * 2^-16, exponent field 31 holds +-Inf (m = 0) and NaN (m != 0); largest
// finite value 1.75 * 2^15 = 57344.
// ---------------------------------------------------------------------------
double e5m2_decode(uint8_t c) {
  int s = (c >> 7) & 1;
  int e = (c >> 2) & 0x1F;
  int m = c & 0x3;
  double v;
  if (e == 0x1F) v = m == 0 ? HUGE_VAL : std::nan("");
  else if (e == 0) v = std::ldexp((double)m, -16);
  else v = std::ldexp(1.0 + m / 4.0, e - 15);
  return s ? -v : v;
}

// The 124 non-negative finite values, code 0x00 .. 0x7B, ascending.
struct E5m2Table {
  double v[124];
  E5m2Table() { for (int c = 0; c < 124; ++c) v[c] = e5m2_decode((uint8_t)c); }
};
const E5m2Table& e5m2_table() { static E5m2Table t; return t; }

// Round an f32 to e5m2: nearest value, ties to the even code; magnitudes past
// the largest finite value (including infinities) saturate to +-57344 (the
// finite-saturating conversion: a scaled operand never becomes infinite);
// NaN -> 0x7F.
uint8_t e5m2_encode(float f) {
  if (std::isnan(f)) return 0x7F;
  uint8_t sign = std::signbit(f) ? 0x80 : 0x00;
  double a = std::fabs((double)f);
  const double* v = e5m2_table().v;
  if (a >= v[123]) return sign | 123;
  int lo = 0, hi = 123;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (v[mid] <= a) lo = mid; else hi = mid;
  }
  int c = lo;
  double d_lo = a - v[c], d_hi = v[c + 1] - a;
  int pick;
  if (d_lo < d_hi) pick = c;
  else if (d_hi < d_lo) pick = c + 1;
  else pick = (c % 2 == 0) ? c : c + 1;
  return sign | (uint8_t)pick;
}

// An fp8 format of the tgmm's dout operand: 0 = e4m3fn, 1 = e5m2.
struct Fp8Fmt {
  int32_t id;
  float max() const { return id == 1 ? 57344.0f : 448.0f; }
  uint8_t encode(float f) const { return id == 1 ? e5m2_encode(f) : e4m3_encode(f); }
  double decode(uint8_t c) const { return id == 1 ? e5m2_decode(c) : e4m3_decode(c); }
};

// ---------------------------------------------------------------------------
// Ragged groups.  Rows of expert e are [off[e], off[e] + gs[e]), off = exclusive
// prefix sum, in the static buffer of M rows ([DQ] What: the buffer has a static
// size; only rows covered by group_sizes are valid).  Clamping: negative sizes
// are 0; ranges are clipped at M.  T = end of the last group.
// ---------------------------------------------------------------------------
struct Groups {
  std::vector<int64_t> begin, end;
  int64_t T = 0;
  Groups(const int32_t* gs, int32_t E, int64_t M) : begin(E), end(E) {
    int64_t off = 0;
    for (int32_t e = 0; e < E; ++e) {
      int64_t g = gs[e] < 0 ? 0 : gs[e];
      begin[e] = std::min(off, M);
      end[e] = std::min(off + g, M);
      off += g;
    }
    T = std::min(off, M);
  }
};

// Guarded row access: a read of a row >= T is counted, never silently taken.
struct RowGuard {
  int64_t T;
  std::atomic<int64_t>* bad;
  bool ok(int64_t row) const {
    if (row < 0 || row >= T) { bad->fetch_add(1); return false; }
    return true;
  }
};

const float kEps = 1e-12f;     // [NQ] Implementation: max(amax, 1e-12)
const float kE4m3Max = 448.0f; // e4m3fn largest finite value

// Per-row full-K activation scale and codes ([NQ] Description, Implementation:
// one f32 absmax scale per row over the whole K, scale = max(amax, 1e-12)/448).
void quantize_one_row(const uint16_t* x, int64_t K, uint8_t* q, float* s_out) {
  float amax = 0.0f;
  for (int64_t k = 0; k < K; ++k) amax = std::max(amax, std::fabs(bf16_to_f32(x[k])));
  float s = std::max(amax, kEps) / kE4m3Max;
  for (int64_t k = 0; k < K; ++k) q[k] = e4m3_encode(bf16_to_f32(x[k]) / s);
  *s_out = s;
}

// One row with one bf16-valued scale per block of `block` columns (reading in
// the comment above orc_gmm_fwd_block).
void quantize_one_row_block(const uint16_t* x, int64_t K, int64_t block, uint8_t* q,
                            float* sb) {
  const int64_t nb = (K + block - 1) / block;
  for (int64_t b = 0; b < nb; ++b) {
    const int64_t k0 = b * block, k1 = std::min(K, k0 + block);
    float amax = 0.0f;
    for (int64_t k = k0; k < k1; ++k) amax = std::max(amax, std::fabs(bf16_to_f32(x[k])));
    const float s = bf16_to_f32(f32_to_bf16_rne(std::max(amax, kEps) / kE4m3Max));
    for (int64_t k = k0; k < k1; ++k) q[k] = e4m3_encode(bf16_to_f32(x[k]) / s);
    sb[b] = s;
  }
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

}  // namespace

extern "C" {

// ----- codec access for the pin tests -------------------------------------
double orc_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
double orc_e5m2_decode(uint8_t c) { return e5m2_decode(c); }

void orc_e5m2_encode_f32(const float* x, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = e5m2_encode(x[i]);
}

void orc_e4m3_encode_f32(const float* x, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}

// Encode the f32 whose bit patterns are [lo, lo + n) (brute-force sweeps).
void orc_e4m3_encode_bits(uint32_t lo, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint32_t u = lo + (uint32_t)i;
    float f;
    std::memcpy(&f, &u, 4);
    out[i] = e4m3_encode(f);
  }
}

void orc_f64_to_bf16(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f64_to_bf16_rne(x[i]);
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// ----- a1: activation row quantization --------------------------------------
// lhs bf16 [M, K]; writes q [M, K] and sx [M] for rows < T only.
// Returns the number of reads of rows >= T (always 0 by construction).
int64_t orc_quantize_rows(const uint16_t* lhs, int64_t M, int64_t K,
                          const int32_t* gs, int32_t E, uint8_t* q, float* sx) {
  Groups g(gs, E, M);
  std::atomic<int64_t> bad{0};
  RowGuard guard{g.T, &bad};
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t m = 0; m < g.T; ++m) {
    if (!guard.ok(m)) continue;
    quantize_one_row(lhs + m * K, K, q + m * K, sx + m);
  }
  return bad.load();
}

// ----- a2..a4: ragged FP8 GMM forward (+ SwiGLU) -----------------------------
// [NQ] Description/Implementation: out[m, n] = sx[m] * sw[e, n] *
// sum_k qx[m, k] * qw[e, k, n], f32-or-better accumulation over ragged groups.
// silu != 0: the N columns are gate | up halves; out[m, j] =
// silu(g) * u with g = y[m, j], u = y[m, N/2 + j] ([NQ] Implementation:
// gmm_silu_fp8, wi with fused SwiGLU).  One bf16 rounding at the end.
//
// rows == nullptr: all rows of all groups; otherwise only the listed rows
// (each must be < T; rows >= T are counted as bad reads and skipped).
// out has Nout = (silu ? N/2 : N) columns and is indexed by the row number;
// out_f64 (optional) receives the unrounded value.
int64_t orc_gmm_fwd(const uint16_t* lhs, int64_t M, int64_t K,
                    const uint8_t* codes, const float* scale, int32_t E, int64_t N,
                    const int32_t* gs, int32_t silu_flag,
                    const int64_t* rows, int64_t nrows,
                    uint16_t* out, double* out_f64) {
  Groups g(gs, E, M);
  std::atomic<int64_t> bad{0};
  RowGuard guard{g.T, &bad};
  const int64_t Nout = silu_flag ? N / 2 : N;
  // expert of a row
  auto expert_of = [&](int64_t m) -> int32_t {
    for (int32_t e = 0; e < E; ++e) if (m >= g.begin[e] && m < g.end[e]) return e;
    return -1;
  };
  std::vector<int64_t> all;
  if (!rows) { all.resize(g.T); for (int64_t m = 0; m < g.T; ++m) all[m] = m; rows = all.data(); nrows = g.T; }
#pragma omp parallel
  {
    std::vector<uint8_t> qrow(K);
    std::vector<double> y(N);
#pragma omp for schedule(dynamic, 4)
    for (int64_t i = 0; i < nrows; ++i) {
      int64_t m = rows[i];
      if (!guard.ok(m)) continue;
      int32_t e = expert_of(m);
      if (e < 0) continue;
      float sx;
      quantize_one_row(lhs + m * K, K, qrow.data(), &sx);
      const uint8_t* w = codes + (int64_t)e * K * N;
      for (int64_t n = 0; n < N; ++n) y[n] = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double a = e4m3_decode(qrow[k]);
        if (a == 0.0) continue;       // exact: adds 0 * finite
        const uint8_t* wr = w + k * N;
        for (int64_t n = 0; n < N; ++n) y[n] += a * e4m3_decode(wr[n]);
      }
      for (int64_t n = 0; n < N; ++n) y[n] = y[n] * (double)sx * (double)scale[(int64_t)e * N + n];
      for (int64_t j = 0; j < Nout; ++j) {
        double v = silu_flag ? silu(y[j]) * y[Nout + j] : y[j];
        out[m * Nout + j] = f64_to_bf16_rne(v);
        if (out_f64) out_f64[m * Nout + j] = v;
      }
    }
  }
  return bad.load();
}

// ----- a5: dequantize_fp8_codes ----------------------------------------------
// [NQ] Implementation: dequantize_fp8_codes, bit-identical to the weight
// dequantization: w = bf16(f32(code) * scale[e, n]) -- one f32 multiply, then
// round to bf16.
void orc_dequantize(const uint8_t* codes, const float* scale, int32_t E, int64_t K,
                    int64_t N, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t ek = 0; ek < (int64_t)E * K; ++ek) {
    int64_t e = ek / K;
    for (int64_t n = 0; n < N; ++n) {
      float p = (float)e4m3_decode(codes[ek * N + n]) * scale[e * N + n];
      out[ek * N + n] = f32_to_bf16_rne(p);
    }
  }
}

// ----- a6: dLHS GMM with the dequantized weight ------------------------------
// [NQ] Description/Implementation: the backward dLHS reads the codes and
// dequantizes each tile; bit-identical to the BF16 dequant backward, so
// dlhs[m, k] = sum_n dout[m, n] * bf16(code[e, k, n] * s[e, n]), bf16 x bf16
// products accumulated (here in double), rounded once to bf16.
// dout bf16 [M, N] -> dlhs bf16 [M, K]; rows as in orc_gmm_fwd.
int64_t orc_gmm_dlhs(const uint16_t* dout, int64_t M, int64_t N,
                     const uint8_t* codes, const float* scale, int32_t E, int64_t K,
                     const int32_t* gs, const int64_t* rows, int64_t nrows,
                     uint16_t* dlhs, double* dlhs_f64) {
  Groups g(gs, E, M);
  std::atomic<int64_t> bad{0};
  RowGuard guard{g.T, &bad};
  auto expert_of = [&](int64_t m) -> int32_t {
    for (int32_t e = 0; e < E; ++e) if (m >= g.begin[e] && m < g.end[e]) return e;
    return -1;
  };
  std::vector<int64_t> all;
  if (!rows) { all.resize(g.T); for (int64_t m = 0; m < g.T; ++m) all[m] = m; rows = all.data(); nrows = g.T; }
#pragma omp parallel
  {
    std::vector<double> wrow(N);
#pragma omp for schedule(dynamic, 4)
    for (int64_t i = 0; i < nrows; ++i) {
      int64_t m = rows[i];
      if (!guard.ok(m)) continue;
      int32_t e = expert_of(m);
      if (e < 0) continue;
      const uint16_t* d = dout + m * N;
      for (int64_t k = 0; k < K; ++k) {
        const uint8_t* c = codes + ((int64_t)e * K + k) * N;
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          float w = (float)e4m3_decode(c[n]) * scale[(int64_t)e * N + n];
          double wb = (double)bf16_to_f32(f32_to_bf16_rne(w));
          acc += (double)bf16_to_f32(d[n]) * wb;
        }
        dlhs[m * K + k] = f64_to_bf16_rne(acc);
        if (dlhs_f64) dlhs_f64[m * K + k] = acc;
      }
    }
  }
  return bad.load();
}

// ----- per-512-column block quantization (see quantize_one_row_block) -------
int64_t orc_quantize_rows_block(const uint16_t* lhs, int64_t M, int64_t K, int64_t block,
                                const int32_t* gs, int32_t E, uint8_t* q, float* sb) {
  Groups g(gs, E, M);
  std::atomic<int64_t> bad{0};
  RowGuard guard{g.T, &bad};
  const int64_t nb = (K + block - 1) / block;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t m = 0; m < g.T; ++m) {
    if (!guard.ok(m)) continue;
    quantize_one_row_block(lhs + m * K, K, block, q + m * K, sb + m * nb);
  }
  return bad.load();
}

// ----- per-512-column block activation quantization, bf16 accumulation -------
// [NQ] Implementation and its review thread: an ops-level option quantizes the
// activation with one bf16 scale per 512-column block (lhs_quant_block_size
// 512, the earlier default) and accumulates across K blocks in bf16; the
// production path is the full-K f32 scale with f32 accumulation. The pages do
// not spell out the rounding points; the reading taken here:
//   per row m and block b = columns [512 b, min(512 b + 512, K)):
//     s[m, b] = bf16( max(amax over the block, 1e-12) / 448 )   (f32 division,
//               then round to nearest even to bf16; kept as its f32 value)
//     q[m, k] = e4m3(x[m, k] / s[m, b])                          (f32 division)
//   forward: acc = 0 (bf16); for each block b in order:
//     d_b = RN_f32( sum_{k in b} q[m, k] * w[e, k, n] )  (the f32 block product)
//     acc = bf16( acc + d_b * s[m, b] )                   (one rounding to bf16)
//   y = acc * sw[e, n] (then SwiGLU as the full-K path), rounded once to bf16.
// acc_max (optional, [M, N]) receives max |acc| over the blocks: the scale of
// the rounding steps, from which a tolerance follows.
int64_t orc_gmm_fwd_block(const uint16_t* lhs, int64_t M, int64_t K, int64_t block,
                          const uint8_t* codes, const float* scale, int32_t E, int64_t N,
                          const int32_t* gs, int32_t silu_flag, const int64_t* rows,
                          int64_t nrows, uint16_t* out, double* out_f64, double* acc_max) {
  Groups g(gs, E, M);
  std::atomic<int64_t> bad{0};
  RowGuard guard{g.T, &bad};
  const int64_t Nout = silu_flag ? N / 2 : N;
  const int64_t nb = (K + block - 1) / block;
  auto expert_of = [&](int64_t m) -> int32_t {
    for (int32_t e = 0; e < E; ++e) if (m >= g.begin[e] && m < g.end[e]) return e;
    return -1;
  };
  std::vector<int64_t> all;
  if (!rows) { all.resize(g.T); for (int64_t m = 0; m < g.T; ++m) all[m] = m; rows = all.data(); nrows = g.T; }
#pragma omp parallel
  {
    std::vector<uint8_t> qrow(K);
    std::vector<float> sb(nb);
    std::vector<double> dot(N), y(N), amx(N);
    std::vector<uint16_t> acc(N);
#pragma omp for schedule(dynamic, 4)
    for (int64_t i = 0; i < nrows; ++i) {
      const int64_t m = rows[i];
      if (!guard.ok(m)) continue;
      const int32_t e = expert_of(m);
      if (e < 0) continue;
      quantize_one_row_block(lhs + m * K, K, block, qrow.data(), sb.data());
      const uint8_t* w = codes + (int64_t)e * K * N;
      for (int64_t n = 0; n < N; ++n) { acc[n] = 0; amx[n] = 0.0; }
      for (int64_t b = 0; b < nb; ++b) {
        for (int64_t n = 0; n < N; ++n) dot[n] = 0.0;
        for (int64_t k = b * block; k < std::min(K, b * block + block); ++k) {
          const double a = e4m3_decode(qrow[k]);
          if (a == 0.0) continue;
          const uint8_t* wr = w + k * N;
          for (int64_t n = 0; n < N; ++n) dot[n] += a * e4m3_decode(wr[n]);   // exact
        }
        for (int64_t n = 0; n < N; ++n) {
          const double d = (double)(float)dot[n];                   // f32 block product
          const double v = (double)bf16_to_f32(acc[n]) + d * (double)sb[b];
          acc[n] = f64_to_bf16_rne(v);
          amx[n] = std::max(amx[n], std::fabs((double)bf16_to_f32(acc[n])));
        }
      }
      for (int64_t n = 0; n < N; ++n)
        y[n] = (double)bf16_to_f32(acc[n]) * (double)scale[(int64_t)e * N + n];
      for (int64_t j = 0; j < Nout; ++j) {
        const double v = silu_flag ? silu(y[j]) * y[Nout + j] : y[j];
        out[m * Nout + j] = f64_to_bf16_rne(v);
        if (out_f64) out_f64[m * Nout + j] = v;
      }
      if (acc_max)
        for (int64_t n = 0; n < N; ++n) acc_max[m * N + n] = amx[n];
    }
  }
  return bad.load();
}

// ----- dSwiGLU (backward of the wi SwiGLU, fused into the wo dLHS) ------------
// [NQ] Implementation: gmm_dswiglu_fp8 is the wo op; its backward is the wo dLHS
// followed by the SwiGLU backward. With h = silu(g) * u, silu(z) = z * sig(z),
// sig(z) = 1 / (1 + exp(-z)), and upstream dh = dL/dh:
//   dg = dh * u * silu'(g),   silu'(g) = sig(g) * (1 + g * (1 - sig(g)))
//   du = dh * silu(g)
// g = gu[m, j], u = gu[m, F + j] (gate | up halves of the wi output, bf16); dh is
// taken unrounded (double, e.g. the exact dLHS sum) and each result is rounded
// once to bf16. dgu is [M, 2F] with dg in [0, F) and du in [F, 2F); rows as in
// orc_gmm_fwd (nullptr = every row < M).
void orc_dswiglu(const double* dh, const uint16_t* gu, int64_t M, int64_t F,
                 const int64_t* rows, int64_t nrows, uint16_t* dgu, double* dgu_f64) {
  std::vector<int64_t> all;
  if (!rows) { all.resize(M); for (int64_t m = 0; m < M; ++m) all[m] = m; rows = all.data(); nrows = M; }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t m = rows[i];
    for (int64_t j = 0; j < F; ++j) {
      const double d = dh[m * F + j];
      const double g = (double)bf16_to_f32(gu[m * 2 * F + j]);
      const double u = (double)bf16_to_f32(gu[m * 2 * F + F + j]);
      const double sg = 1.0 / (1.0 + std::exp(-g));
      const double dg = d * u * (sg * (1.0 + g * (1.0 - sg)));
      const double du = d * (g * sg);
      dgu[m * 2 * F + j] = f64_to_bf16_rne(dg);
      dgu[m * 2 * F + F + j] = f64_to_bf16_rne(du);
      if (dgu_f64) {
        dgu_f64[m * 2 * F + j] = dg;
        dgu_f64[m * 2 * F + F + j] = du;
      }
    }
  }
}

// ----- a7: tgmm operand quantization per gm-tile per channel -----------------
// [DQ] What: the drhs tgmm quantizes its operands inside the kernel, per gm tile
// and per channel, e4m3, touching only the tiles covered by group_sizes.
// Reading taken here: gm tiles are the global 128-row tiles [128 t, 128 t + 128)
// of the buffer, intersected with each group (a tile shared by two groups is
// two segments with their own scales).  Per segment and column:
// s = max(amax over the segment's rows, 1e-12) / 448 in f32, codes = e4m3(x / s).
// With d_fmt = 1 the dout operand is e5m2 instead ([DQ] What, the gradient
// dtype): s = max(amax, 1e-12) / 57344 (reading: the same rule with the e5m2
// maximum), codes = e5m2(x / s).
//
// Segments are numbered expert by expert, tiles ascending, empty experts have
// none.  Output layout (the library's debug export uses the same): for segment
// q with tile t, slot row r in [0, 128) holds buffer row 128 t + r if that row is
// in the segment and zero codes otherwise.
//   qx [Smax, 128, K] u8, sx [Smax, K] f32, qd [Smax, 128, N] u8, sd [Smax, N] f32
// Returns the number of reads of rows >= T.  *nseg receives the segment count.
int64_t orc_tgmm_quantize_tiles(const uint16_t* lhs, const uint16_t* dout,
                                int64_t M, int64_t K, int64_t N, int32_t E,
                                const int32_t* gs, int64_t Smax,
                                uint8_t* qx, float* sx, uint8_t* qd, float* sd,
                                int64_t* nseg, int32_t d_fmt) {
  Groups g(gs, E, M);
  std::atomic<int64_t> bad{0};
  RowGuard guard{g.T, &bad};
  // enumerate segments
  std::vector<int32_t> seg_e;
  std::vector<int64_t> seg_t;
  for (int32_t e = 0; e < E; ++e) {
    if (g.end[e] <= g.begin[e]) continue;
    for (int64_t t = g.begin[e] / 128; t <= (g.end[e] - 1) / 128; ++t) {
      seg_e.push_back(e);
      seg_t.push_back(t);
    }
  }
  *nseg = (int64_t)seg_e.size();
  if ((int64_t)seg_e.size() > Smax) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t q = 0; q < (int64_t)seg_e.size(); ++q) {
    int32_t e = seg_e[q];
    int64_t t = seg_t[q];
    int64_t r0 = std::max(g.begin[e], t * 128), r1 = std::min(g.end[e], t * 128 + 128);
    for (int pass = 0; pass < 2; ++pass) {
      const uint16_t* src = pass == 0 ? lhs : dout;
      int64_t C = pass == 0 ? K : N;
      uint8_t* qo = (pass == 0 ? qx : qd) + q * 128 * C;
      float* so = (pass == 0 ? sx : sd) + q * C;
      const Fp8Fmt fmt{pass == 0 ? 0 : d_fmt};
      std::memset(qo, 0, (size_t)(128 * C));
      for (int64_t c = 0; c < C; ++c) {
        float amax = 0.0f;
        for (int64_t m = r0; m < r1; ++m) {
          if (!guard.ok(m)) continue;
          amax = std::max(amax, std::fabs(bf16_to_f32(src[m * C + c])));
        }
        float s = std::max(amax, kEps) / fmt.max();
        so[c] = s;
        for (int64_t m = r0; m < r1; ++m) {
          if (!guard.ok(m)) continue;
          qo[(m - t * 128) * C + c] = fmt.encode(bf16_to_f32(src[m * C + c]) / s);
        }
      }
    }
  }
  return bad.load();
}

// ----- a8: tgmm contraction ---------------------------------------------------
// dW[e, k, n] = sum over the segments of e of sx[q, k] * sd[q, n] *
//               sum_{m in segment} qx[m, k] * qd[m, n]      (double, -> f32)
// An expert with no rows gets dW[e] = 0.  Only the block
// [k0, k1) x [n0, n1) of each listed expert is computed (experts == nullptr:
// all experts in order; k0 = n0 = 0, k1 = K, n1 = N selects the whole matrix).
// dW_blk is [nexperts, k1 - k0, n1 - n0] f32.
int64_t orc_tgmm(const uint16_t* lhs, const uint16_t* dout, int64_t M, int64_t K,
                 int64_t N, int32_t E, const int32_t* gs,
                 const int32_t* experts, int32_t nexperts,
                 int64_t k0, int64_t k1, int64_t n0, int64_t n1, float* dW, int32_t d_fmt) {
  Groups g(gs, E, M);
  std::atomic<int64_t> bad{0};
  RowGuard guard{g.T, &bad};
  std::vector<int32_t> all;
  if (!experts) { all.resize(E); for (int32_t e = 0; e < E; ++e) all[e] = e; experts = all.data(); nexperts = E; }
  const int64_t KB = k1 - k0, NB = n1 - n0;
  for (int32_t ie = 0; ie < nexperts; ++ie) {
    int32_t e = experts[ie];
    std::vector<double> acc((size_t)(KB * NB), 0.0);
    if (g.end[e] > g.begin[e]) {
      for (int64_t t = g.begin[e] / 128; t <= (g.end[e] - 1) / 128; ++t) {
        int64_t r0 = std::max(g.begin[e], t * 128), r1 = std::min(g.end[e], t * 128 + 128);
        int64_t R = r1 - r0;
        // per-channel scales over the segment rows, then codes
        std::vector<float> sxs(KB), sds(NB);
        std::vector<double> qxv((size_t)(R * KB)), qdv((size_t)(R * NB));
        for (int pass = 0; pass < 2; ++pass) {
          const uint16_t* src = pass == 0 ? lhs : dout;
          int64_t C = pass == 0 ? K : N;
          int64_t c0 = pass == 0 ? k0 : n0, CB = pass == 0 ? KB : NB;
          std::vector<float>& s_out = pass == 0 ? sxs : sds;
          std::vector<double>& q_out = pass == 0 ? qxv : qdv;
          const Fp8Fmt fmt{pass == 0 ? 0 : d_fmt};
#pragma omp parallel for schedule(static)
          for (int64_t c = 0; c < CB; ++c) {
            float amax = 0.0f;
            for (int64_t m = r0; m < r1; ++m) {
              if (!guard.ok(m)) continue;
              amax = std::max(amax, std::fabs(bf16_to_f32(src[m * C + c0 + c])));
            }
            float s = std::max(amax, kEps) / fmt.max();
            s_out[c] = s;
            for (int64_t m = r0; m < r1; ++m) {
              if (!guard.ok(m)) continue;
              q_out[(m - r0) * CB + c] = fmt.decode(fmt.encode(bf16_to_f32(src[m * C + c0 + c]) / s));
            }
          }
        }
#pragma omp parallel for schedule(static)
        for (int64_t kk = 0; kk < KB; ++kk) {
          for (int64_t nn = 0; nn < NB; ++nn) {
            double dot = 0.0;
            for (int64_t r = 0; r < R; ++r) dot += qxv[r * KB + kk] * qdv[r * NB + nn];
            acc[kk * NB + nn] += (double)sxs[kk] * (double)sds[nn] * dot;
          }
        }
      }
    }
    for (int64_t kk = 0; kk < KB; ++kk)
      for (int64_t nn = 0; nn < NB; ++nn)
        dW[((int64_t)ie * KB + kk) * NB + nn] = (float)acc[kk * NB + nn];
  }
  return bad.load();
}

}  // extern "C"
