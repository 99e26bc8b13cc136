/* fp8moe.h -- C ABI of libfp8moe.so: native-FP8 grouped matmuls for the routed
 * experts of a mixture-of-experts layer, on one GB300 (sm_103a).
 *
 * Sources (web pages):
 *   [NQ] "MoE: native FP8 QAT for routed-expert GMMs (FP8 forward + FP8-weight
 *        backward dLHS)" -- Description, Data flow, Implementation, Tests.
 *   [DQ] "MoE fp8 backward: in-kernel drhs operand quantization + configurable
 *        gradient dtype" -- What.
 *   [SM] "Fix fp8 MoE on the sparse_matmul path" -- Fix (forward dtype is
 *        float8_e4m3fn).
 *
 * Common conventions
 *   - All array pointers are DEVICE pointers on the current CUDA device,
 *     row-major and contiguous, 16-byte aligned.  bf16 arrays are passed as
 *     void* (IEEE bfloat16 bit patterns).  FP8 codes are OCP float8_e4m3fn bit
 *     patterns in uint8_t.
 *   - The ragged buffer has a static number of rows M.  group_sizes (int32 [E],
 *     device memory) gives the rows of each expert, in order: expert e owns rows
 *     [off[e], off[e] + group_sizes[e]) with off the exclusive prefix sum.
 *     T = sum(group_sizes) may be smaller than M; rows >= T are never read and
 *     never written.  A negative size counts as 0 and ranges are clipped at M;
 *     both are recorded in the device status word (fp8moe_read_status).
 *   - Weights: codes[E, K, N] (N contiguous) with per-output-channel f32
 *     scale[E, N] (the pages' [g, 1, n] scale); weight w = code * scale.
 *   - K is whole in every call: the activation scale always spans all K.
 *   - Calls only enqueue work on `stream`; they never synchronize and never
 *     copy group_sizes to the host.  The caller owns every buffer, including the
 *     workspace (size from fp8moe_workspace_size); the library allocates no
 *     memory.
 *   - Shapes: 1 <= E <= 1024; K, N > 0 and multiples of 16 (TMA stride rule);
 *     0 <= M < 2^31 (M == 0 returns FP8MOE_OK without launching).
 *   - Return value: FP8MOE_OK (0) or a negative FP8MOE_E* code; nothing is
 *     launched when an argument check fails.  fp8moe_last_cuda_error() gives the
 *     CUDA error behind FP8MOE_ECUDA.
 */
#ifndef FP8MOE_H_
#define FP8MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp8moe_stream_t;

enum {
  FP8MOE_OK = 0,
  FP8MOE_EINVAL = -1,       /* null pointer, bad dimension, odd N for SwiGLU, E out of range */
  FP8MOE_EALIGN = -2,       /* pointer not 16-byte aligned, or K / N not a multiple of 16 */
  FP8MOE_EWORKSPACE = -3,   /* workspace missing or smaller than fp8moe_workspace_size() */
  FP8MOE_ECUDA = -4,        /* a CUDA call or launch failed; see fp8moe_last_cuda_error() */
  FP8MOE_EUNSUPPORTED = -5  /* the current device is not an sm_103 GPU */
};

/* Operation ids for fp8moe_workspace_size. */
enum {
  FP8MOE_OP_GMM_FP8_FWD = 1,
  FP8MOE_OP_GMM_SILU_FP8_FWD = 2,
  FP8MOE_OP_GMM_DLHS_FP8 = 3,
  FP8MOE_OP_TGMM_DRHS_QUANT = 4,
  FP8MOE_OP_GMM_BF16_FWD = 5,
  FP8MOE_OP_DEQUANTIZE = 6,
  FP8MOE_OP_GMM_FP8_FWD_BLOCK = 7
};

/* fp8 formats of the tgmm's dout (gradient) operand -- [DQ] What: the
 * gradient fp8 dtype is configurable, e5m2 (the recipe's default) or e4m3. */
enum {
  FP8MOE_FMT_E4M3 = 0,   /* OCP float8_e4m3fn, max 448 */
  FP8MOE_FMT_E5M2 = 1    /* OCP float8_e5m2, max 57344 */
};

/* Bits of the device status word. */
#define FP8MOE_STATUS_NEGATIVE_GROUP 0x1u    /* some group_sizes[e] < 0 (taken as 0) */
#define FP8MOE_STATUS_GROUPS_EXCEED_M 0x2u   /* sum(group_sizes) > M (clipped at M) */
#define FP8MOE_STATUS_WAIT_TIMEOUT 0x4u      /* a kernel pipeline wait gave up; bits 8..15 say where */
#define FP8MOE_STATUS_TOO_MANY_SEGMENTS 0x8u /* internal: segment bound exceeded */

/* Workspace bytes the operation needs for these sizes (0 if none); the
 * workspace pointer must be 256-byte aligned.  Depends on M, K, N, E only. */
size_t fp8moe_workspace_size(int op, int64_t M, int64_t K, int64_t N, int32_t E);

/* Forward FP8 GMM, no epilogue (wo forward; also the ring-of-experts down
 * projection forward) -- [NQ] Implementation (gmm_dswiglu_fp8 forward,
 * gmm_fp8_forward).  For row m of expert e:
 *   sx[m]  = max(max_k |lhs[m,k]|, 1e-12) / 448          (f32, full K)
 *   qx     = e4m3(lhs[m,k] / sx[m])                       (RNE, saturating)
 *   out[m,n] = bf16( sx[m] * scale[e,n] * sum_k qx[m,k] * codes[e,k,n] )  (f32 accumulation)
 * lhs: bf16 [M, K].  codes: u8 [E, K, N].  scale: f32 [E, N].
 * out: bf16 [M, N]; rows >= T untouched.  Workspace: FP8MOE_OP_GMM_FP8_FWD
 * (holds the activation codes and row scales). */
int fp8moe_gmm_fp8_fwd(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                       const float* scale, int32_t E, int64_t N, const int32_t* group_sizes,
                       void* out, void* workspace, size_t workspace_bytes,
                       fp8moe_stream_t stream);

/* Forward FP8 GMM with the fused SwiGLU epilogue (wi forward) -- [NQ]
 * Implementation (gmm_silu_fp8).  Same as fp8moe_gmm_fp8_fwd; the N columns
 * are gate | up halves (N a multiple of 32, else FP8MOE_EALIGN: the up half
 * must start on a 16-byte boundary) and, with y the scaled f32 accumulator,
 *   out[m, j] = bf16( silu(y[m, j]) * y[m, N/2 + j] ),  silu(z) = z / (1 + exp(-z)).
 * out: bf16 [M, N/2].  Workspace: FP8MOE_OP_GMM_SILU_FP8_FWD. */
int fp8moe_gmm_silu_fp8_fwd(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                            const float* scale, int32_t E, int64_t N,
                            const int32_t* group_sizes, void* out, void* workspace,
                            size_t workspace_bytes, fp8moe_stream_t stream);

/* Backward dLHS GMM from the FP8 weight -- [NQ] Description and Implementation
 * (rhs_contract_dequant): each weight tile is dequantized on chip,
 *   w[e,k,n] = bf16(f32(codes[e,k,n]) * scale[e,n]),
 *   dlhs[m,k] = bf16( sum_n dout[m,n] * w[e,k,n] )   (f32 accumulation),
 * bit-identical whichever internal path is taken (contraction N <= 256: the
 * dequantized weight block cached in shared memory; N > 256: CTA pairs with the
 * dequantized weight tile in tensor memory).
 * dout: bf16 [M, N] (the forward output's cotangent).  dlhs: bf16 [M, K];
 * rows >= T untouched.  No workspace (pass NULL, 0). */
int fp8moe_gmm_dlhs_fp8(const void* dout, int64_t M, int64_t N, const uint8_t* codes,
                        const float* scale, int32_t E, int64_t K, const int32_t* group_sizes,
                        void* dlhs, void* workspace, size_t workspace_bytes,
                        fp8moe_stream_t stream);

/* Same as fp8moe_gmm_dlhs_fp8 with the internal path forced: path 0 streams
 * and dequantizes every weight tile per output tile; path 1 keeps the
 * dequantized weight block of an (expert, k tile) on chip across the expert's
 * m tiles (needs N <= 256, else FP8MOE_EINVAL); path 2 computes the transposed
 * product on CTA pairs with the dequantized weight tile held in tensor memory
 * (the default for N > 256).  Any other path: FP8MOE_EINVAL.  All paths give
 * identical bits. */
int fp8moe_gmm_dlhs_fp8_path(const void* dout, int64_t M, int64_t N, const uint8_t* codes,
                             const float* scale, int32_t E, int64_t K,
                             const int32_t* group_sizes, void* dlhs, int32_t path,
                             fp8moe_stream_t stream);

/* wo dLHS with the SwiGLU backward fused into its epilogue -- [NQ]
 * Implementation (gmm_dswiglu_fp8, the wo op whose backward also undoes the wi
 * SwiGLU).  With codes/scale the wo weight [E, F, N] / [E, N]:
 *   dh[m,f]  = sum_n dout[m,n] * w[e,f,n]   (as fp8moe_gmm_dlhs_fp8, f32, not rounded)
 *   g = gu[m,f], u = gu[m,F+f], sig(z) = 1 / (1 + exp(-z))
 *   dgu[m,f]   = bf16( dh * u * sig(g) * (1 + g * (1 - sig(g))) )     (dg)
 *   dgu[m,F+f] = bf16( dh * g * sig(g) )                              (du)
 * gu: bf16 [M, 2F], the wi forward output before SwiGLU (gate | up halves).
 * dgu: bf16 [M, 2F]; rows >= T untouched; dh is never written to memory.
 * Pointers 16-byte aligned; F % 16 == 0 and N % 16 == 0 (FP8MOE_EALIGN);
 * gu NULL with M > 0: FP8MOE_EINVAL.  No workspace (pass NULL, 0). */
int fp8moe_gmm_dlhs_dswiglu_fp8(const void* dout, int64_t M, int64_t N, const uint8_t* codes,
                                const float* scale, int32_t E, int64_t F, const void* gu,
                                const int32_t* group_sizes, void* dgu, void* workspace,
                                size_t workspace_bytes, fp8moe_stream_t stream);

/* fp8moe_gmm_dlhs_dswiglu_fp8 with the internal path forced (0 streaming,
 * 1 on-chip weight cache, N <= 256, 2 CTA pairs with the weight in tensor
 * memory); all give identical bits. */
int fp8moe_gmm_dlhs_dswiglu_fp8_path(const void* dout, int64_t M, int64_t N, const uint8_t* codes,
                                     const float* scale, int32_t E, int64_t F, const void* gu,
                                     const int32_t* group_sizes, void* dgu, int32_t path,
                                     fp8moe_stream_t stream);

/* Weight-gradient tgmm with in-kernel per-tile operand quantization -- [DQ]
 * What.  Segments: the global 128-row tiles [128t, 128t+128) intersected with
 * each group.  Per segment q and channel:
 *   sx[q,k] = max(max_{m in q} |lhs[m,k]|, 1e-12) / 448,  qx = e4m3(lhs / sx)
 *   sd[q,n] = max(max_{m in q} |dout[m,n]|, 1e-12) / 448, qd = e4m3(dout / sd)
 *   dW[e,k,n] = sum_{q of e} sx[q,k] * sd[q,n] * sum_{m in q} qx[m,k] * qd[m,n]
 * lhs: bf16 [M, K]; dout: bf16 [M, N]; dW: f32 [E, K, N], fully written
 * (experts without rows get 0).  Rows >= T are never read, so garbage there
 * (NaN, Inf) cannot reach dW.  Workspace: FP8MOE_OP_TGMM_DRHS_QUANT. */
int fp8moe_tgmm_drhs_quant(const void* lhs, const void* dout, int64_t M, int64_t K, int64_t N,
                           int32_t E, const int32_t* group_sizes, float* dW, void* workspace,
                           size_t workspace_bytes, fp8moe_stream_t stream);

/* fp8moe_tgmm_drhs_quant with the dout operand's fp8 format chosen -- [DQ]
 * What (configurable gradient dtype).  FP8MOE_FMT_E5M2:
 *   sd[q,n] = max(max_{m in q} |dout[m,n]|, 1e-12) / 57344, qd = e5m2(dout / sd)
 * (round to nearest even, saturating at +-57344); lhs stays e4m3 and the MMA
 * multiplies e4m3 x e5m2.  FP8MOE_FMT_E4M3 is fp8moe_tgmm_drhs_quant.  Any
 * other dout_fmt: FP8MOE_EINVAL.  Same workspace. */
int fp8moe_tgmm_drhs_quant_fmt(const void* lhs, const void* dout, int64_t M, int64_t K, int64_t N,
                               int32_t E, const int32_t* group_sizes, float* dW, void* workspace,
                               size_t workspace_bytes, int32_t dout_fmt, fp8moe_stream_t stream);

/* dequantize_fp8_codes -- [NQ] Implementation: out[e,k,n] =
 * bf16(f32(codes[e,k,n]) * scale[e,n]) (one f32 multiply, round to nearest
 * even).  out: bf16 [E, K, N]. */
int fp8moe_dequantize_fp8_codes(const uint8_t* codes, const float* scale, int32_t E, int64_t K,
                                int64_t N, void* out, fp8moe_stream_t stream);

/* BF16 grouped matmul, the fake-QAT comparison arm ([NQ] Tests: the BF16 GMM
 * takes a weight dequantized beforehand): out = bf16(lhs x w[e]) with f32
 * accumulation, w: bf16 [E, K, N]; swiglu != 0 applies the same SwiGLU
 * epilogue as fp8moe_gmm_silu_fp8_fwd (out [M, N/2]). */
int fp8moe_gmm_bf16_fwd(const void* lhs, int64_t M, int64_t K, const void* w, int32_t E,
                        int64_t N, const int32_t* group_sizes, int32_t swiglu, void* out,
                        fp8moe_stream_t stream);

/* Forward GMM with per-block activation quantization -- [NQ] Implementation:
 * the ops-level lhs_quant_block_size = 512 option (the pages' earlier default;
 * the production forward is fp8moe_gmm_fp8_fwd's full-K f32 scale).  Per row m
 * and block b of 512 columns (the last one may be shorter):
 *   sb[m,b] = bf16( max(max_{k in b} |lhs[m,k]|, 1e-12) / 448 ),  q = e4m3(lhs / sb)
 *   acc = 0 (bf16); for each block b:  acc = bf16( acc + sb[m,b] * P_b[m,n] ),
 *     P_b = the f32 product of the block's codes,  sum_{k in b} q[m,k] * codes[e,k,n]
 *   out[m,n] = bf16( acc * scale[e,n] ), or with swiglu = 1 the SwiGLU of the
 *   gate | up halves as fp8moe_gmm_silu_fp8_fwd (out [M, N/2]).
 * block must be 512 (FP8MOE_EINVAL otherwise).  Workspace:
 * FP8MOE_OP_GMM_FP8_FWD_BLOCK (codes and block scales).  Rows >= T untouched. */
int fp8moe_gmm_fp8_fwd_block(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                             const float* scale, int32_t E, int64_t N,
                             const int32_t* group_sizes, void* out, void* workspace,
                             size_t workspace_bytes, int32_t block, int32_t swiglu,
                             fp8moe_stream_t stream);

/* Parity export of the block quantization above: q u8 [M, K] and the
 * bf16-valued f32 scales sb [M, ceil(K/512)] for rows < T. */
int fp8moe_quantize_rows_block(const void* lhs, int64_t M, int64_t K, const int32_t* group_sizes,
                               int32_t E, int32_t block, uint8_t* q, float* sb,
                               fp8moe_stream_t stream);

/* Parity export of the forward activation quantization: q u8 [M, K] and
 * sx f32 [M] for rows < T (rows >= T untouched). */
int fp8moe_quantize_rows(const void* lhs, int64_t M, int64_t K, const int32_t* group_sizes,
                         int32_t E, uint8_t* q, float* sx, fp8moe_stream_t stream);

/* Parity export of the tgmm operand quantization.  Segments are numbered
 * expert by expert, tiles ascending; S = the segment bound ceil(M/128) + E.
 * Segment q of tile t fills slot q: slot row r holds buffer row 128t + r if it
 * belongs to the segment, else zero codes.  qx u8 [S, 128, K], sx f32 [S, K],
 * qd u8 [S, 128, N], sd f32 [S, N]; slots past the last segment untouched. */
int fp8moe_tgmm_quantize_tiles(const void* lhs, const void* dout, int64_t M, int64_t K,
                               int64_t N, int32_t E, const int32_t* group_sizes, uint8_t* qx,
                               float* sx, uint8_t* qd, float* sd, fp8moe_stream_t stream);

/* fp8moe_tgmm_quantize_tiles with the dout format chosen (FP8MOE_FMT_*): qd
 * holds e5m2 codes and sd the e5m2 scales when dout_fmt = FP8MOE_FMT_E5M2. */
int fp8moe_tgmm_quantize_tiles_fmt(const void* lhs, const void* dout, int64_t M, int64_t K,
                                   int64_t N, int32_t E, const int32_t* group_sizes, uint8_t* qx,
                                   float* sx, uint8_t* qd, float* sd, int32_t dout_fmt,
                                   fp8moe_stream_t stream);

/* Exercises the failure path of the bounded pipeline waits: one thread waits on
 * an mbarrier that nothing ever completes, gives up after limit_us
 * microseconds (1 .. 2,000,000, else FP8MOE_EINVAL), records
 * FP8MOE_STATUS_WAIT_TIMEOUT with where = 6 (bits 8..15) in the status word and
 * exits; the context stays usable.  For tests of failure detection; the paper
 * has no counterpart. */
int fp8moe_selftest_wait_timeout(uint32_t limit_us, fp8moe_stream_t stream);

/* The f32 -> fp8 cast that every quantizer of the library ends in, on
 * arbitrary inputs: codes[i] = RN_sat(x[i]) in the format fmt (FP8MOE_FMT_E4M3:
 * round to nearest even, saturating at +-448, NaN -> NaN code; FP8MOE_FMT_E5M2:
 * the same at +-57344), converted two values at a time by the same
 * cvt.rn.satfinite helpers as the quantizers ("MoE: native FP8 QAT for
 * routed-expert GMMs", Implementation: the e4m3 activation codes; "MoE fp8
 * backward: in-kernel drhs operand quantization", What: the e5m2 gradient
 * codes).  x f32 [n] and codes u8 [n] are device pointers, x 4-byte aligned;
 * the caller owns both.  n = 0 does nothing.  FP8MOE_EINVAL: n < 0, an unknown
 * fmt, or a null pointer with n > 0.  For parity tests of the cast over whole
 * binades of bit patterns. */
int fp8moe_selftest_cast_f32(const float* x, int64_t n, int32_t fmt, uint8_t* codes,
                             fp8moe_stream_t stream);

/* Waits for `stream`, returns in *flags the OR of the FP8MOE_STATUS_* bits set
 * since the last call, and clears them. */
int fp8moe_read_status(fp8moe_stream_t stream, uint32_t* flags);

/* The wi forward of fp8moe_gmm_silu_fp8_fwd for callers that cannot allocate
 * device memory (a plugin inside a framework whose caching allocator holds
 * nearly all of it, or a runtime that forbids allocations after start-up).  The
 * pages have no counterpart: it is an interface variant, not a step of the
 * method.  Arguments and results are those of fp8moe_gmm_silu_fp8_fwd minus the
 * workspace, which comes from a fixed 32 MiB device array that the library holds
 * on every GPU it is loaded on until the process exits; sizes whose workspace
 * (fp8moe_workspace_size(FP8MOE_OP_GMM_SILU_FP8_FWD, ...)) exceeds it return
 * FP8MOE_EWORKSPACE and launch nothing.  Argument errors are checked first and
 * return what fp8moe_gmm_silu_fp8_fwd would (FP8MOE_EINVAL, FP8MOE_EALIGN),
 * whatever the size.  The first call on a device looks up the array's device
 * address and keeps it (make that call before any stream capture); after a
 * cudaDeviceReset the kept address is stale, so do not call this again in that
 * process.  All calls share the array, so calls that overlap on the GPU race;
 * each call rewrites everything it reads, so nothing needs clearing between
 * calls.  Allocates nothing. */
int fp8moe_gmm_silu_fp8_fwd_noalloc(const void* lhs, int64_t M, int64_t K, const uint8_t* codes,
                                    const float* scale, int32_t E, int64_t N,
                                    const int32_t* group_sizes, void* out,
                                    fp8moe_stream_t stream);

/* Text for a return code. */
const char* fp8moe_status_string(int code);

/* The cudaError_t value behind the last FP8MOE_ECUDA of this thread. */
int fp8moe_last_cuda_error(void);

/* Number of SMs the kernels size their grids for (0 if no device). */
int fp8moe_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8MOE_H_ */
