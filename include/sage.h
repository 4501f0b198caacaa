/*
 * sage.h -- C ABI of the GB300 (sm_103a) SageBwd attention library (libsage_gb300.so).
 *
 * SageBwd is the trainable INT8 attention of "SageBwd: A Trainable Low-bit Attention" and of the
 * SageBwd part of "SageAttention3: Microscaling FP4 Attention for Inference and An Exploration of
 * 8-Bit Training".  The library exposes the method's three steps:
 *
 *   sage_quantize_smooth  K-smoothing (and optional Q-smoothing) plus per-block INT8 quantisation
 *   sage_attn_fwd         tiled online-softmax forward with per-token P codes; writes O and L
 *   sage_attn_bwd         backward with 16-bit dP and per-tile INT8 P / dS codes; writes dQ, dK, dV
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous, row-major (B, H, N, d): token n of head (b, h) starts at element
 *     ((b * H + h) * N + n) * d.  Per-block scales are float32 (B, H, N / 64).
 *   - Every pointer is DEVICE memory allocated and owned by the caller, except `p` (host).  The
 *     library allocates nothing.  Scratch memory is the caller's `workspace` of at least the size
 *     the matching *_workspace_bytes() query returns, except for sage_quantize_smooth_noalloc,
 *     which keeps its scratch in a fixed array inside the library.  The other state kept between
 *     calls is the device error word that sage_device_status() reads and clears, and host-side
 *     caches (the SM count per device, the quantise kernels' occupancy, that array's address
 *     per device).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).  The
 *     return value reports argument and launch errors only; a device-side timeout of a bounded
 *     wait is reported by sage_device_status().
 *   - Supported: N a multiple of 64 (N >= 64), d in {64, 128}, dtype fp16 or bf16, self-attention
 *     (queries and keys share N).  Inputs must be finite.  All device pointers must be 16-byte
 *     aligned.
 *   - Causal masking is top-left aligned: query n attends to keys m <= n.
 */
#ifndef SAGE_GB300_H
#define SAGE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define SAGE_OK 0
#define SAGE_ERR_ARG 1          /* null pointer, non-positive size, bad flag value            */
#define SAGE_ERR_UNSUPPORTED 2  /* d not in {64,128}, N % 64 != 0, unknown dtype              */
#define SAGE_ERR_ALIGN 3        /* a device pointer is not 16-byte aligned                     */
#define SAGE_ERR_CUDA 4         /* a kernel launch or CUDA runtime call failed                 */
#define SAGE_ERR_TIMEOUT 5      /* a bounded device-side wait expired (see sage_device_status) */
#define SAGE_ERR_WORKSPACE 6    /* workspace missing or smaller than the query says            */

/* Element types of the 16-bit tensors (Q, K, V, dO, O). */
#define SAGE_FP16 0
#define SAGE_BF16 1

/* Flags. */
#define SAGE_FLAG_DUMP 1u       /* debug: write the integer block products and the in-kernel
                                   codes to `dump` (small problems only; see sage_dump_bytes) */
#define SAGE_FLAG_DP_INT8 2u    /* sage_attn_bwd only: form dP from the INT8 codes of dO and V,
                                   dP = fl32(MM(dO^, V^T) * fl32(s_dO s_V)), instead of the 16-bit
                                   product the method keeps -- the ablation of "SageAttention3 ..."
                                   (review), Table 1c.  V is quantised per 64-token block inside
                                   the call (same codes as sage_quantize_smooth); the workspace
                                   grows by 3 bytes per element plus the scales. */
#define SAGE_FLAG_FP8 4u        /* FP8 SageBwd ("SageAttention3 ..." (review), INT8 vs FP8
                                   training): every INT8 code becomes an FP8 E4M3 code (OCP
                                   format: bias 7, 3 mantissa bits, largest finite 448), with 448
                                   in place of 127 -- block scales fl32(max|x| / 448) and codes
                                   e4m3(fl32(x / delta)) (round to nearest even, saturating);
                                   forward P codes e4m3(fl32(448 ex2(x))); backward tile codes
                                   e4m3(fl32(x fl32(1 / s))), s = fl32(max|x| / 448), tiles with
                                   max|x| < 2^-110 zero.  The int8_t code buffers then hold E4M3
                                   bit patterns.  Pass it to all three calls of one pass; it
                                   cannot be combined with SAGE_FLAG_DUMP or SAGE_FLAG_DP_INT8
                                   (SAGE_ERR_UNSUPPORTED). */
#define SAGE_FLAG_OPS16 8u      /* operand copies in fp16: the tensor cores take the codes as their
                                   exact fp16 values, and without this flag the forward and backward
                                   calls widen the codes into their workspaces (5 passes a step).
                                   sage_quantize_smooth (and its QK-norm and no-allocation forms)
                                   then also writes those values to p->ops16: Q^, K^, V^ in that
                                   order, each (B,H,N,d) fp16, 16-byte aligned.  sage_attn_fwd and
                                   sage_attn_bwd read them from p->ops16 instead of widening (they
                                   must be the copies of the same codes) and their workspace
                                   queries drop the widened copies.  The tensor cores see the
                                   same operands as without the flag.  The FP4 and Attn-QAT entry
                                   points refuse it (SAGE_ERR_UNSUPPORTED). */

typedef struct CUstream_st *sage_stream_t;   /* identical to cudaStream_t */

#if defined(__GNUC__)
#define SAGE_API __attribute__((visibility("default")))
#else
#define SAGE_API
#endif

typedef struct sage_params {
    int B;           /* batch                                                                */
    int H;           /* heads                                                                */
    int N;           /* sequence length (queries = keys), multiple of 64                    */
    int d;           /* head dimension, 64 or 128                                            */
    int dtype;       /* SAGE_FP16 or SAGE_BF16: type of Q, K, V, dO and O                    */
    int causal;      /* 0 or 1                                                               */
    int smooth_k;    /* 1 (default): subtract the mean over tokens of K before quantising   */
    int smooth_q;    /* 0 (default): 1 subtracts each 64-row block mean of Q and adds the
                        bias mu_Q K_sm^T to the logits (and its gradient to dK)              */
    unsigned flags;  /* SAGE_FLAG_*                                                          */
    void *dump;      /* device buffer for SAGE_FLAG_DUMP, else NULL                          */
    size_t dump_bytes;
    void *ops16;     /* device buffer for SAGE_FLAG_OPS16, else NULL: (3,B,H,N,d) fp16       */
} sage_params;

/* ------------------------------------------------------------------------------------------ *
 * Step 1 -- smoothing and per-block INT8 quantisation.
 * "SageBwd: A Trainable Low-bit Attention" (structured summary): prerequisites, INT8
 * quantisation (X^ = round(X / delta), delta = max|X| / 127) and K-/Q-smoothing (mu_K = mean over
 * tokens of K, K_sm = K - mu_K; mu_Qi = mean over the rows of query block i); method steps,
 * forward (2).  "SageAttention3 ..." (review), eq. (7).
 *
 * In:  Q, K, V      (B,H,N,d) fp16/bf16.
 * Out: Qh, Kh, Vh   (B,H,N,d) int8 codes in [-127, 127] of Q (or Q - mu_Q), K - mu_K (or K), V.
 *      sQ, sK, sV   (B,H,N/64) float32 block scales delta = fl32(max|x| / 127); a block whose max
 *                   is zero gets delta = 0 and all-zero codes.
 *      muK          (B,H,d) float32: float64 sum over the N tokens / N, rounded once (zeros when
 *                   smooth_k = 0).
 *      muQ          (B,H,N/64,d) float32 block means (same rule), required iff smooth_q = 1.
 * Codes are round-half-even of fl32(x / delta) with IEEE float32 division, x = fl32(v - mu).
 * ------------------------------------------------------------------------------------------ */
SAGE_API size_t sage_quantize_workspace_bytes(const sage_params *p);
SAGE_API int sage_quantize_smooth(const sage_params *p, const void *Q, const void *K, const void *V,
                         int8_t *Qh, int8_t *Kh, int8_t *Vh, float *sQ, float *sK, float *sV,
                         float *muK, float *muQ, void *workspace, size_t workspace_bytes,
                         sage_stream_t stream);

/* ------------------------------------------------------------------------------------------ *
 * Step 1 with the QK-norm prologue fused in, and the QK-norm gradient.
 * "SageBwd: A Trainable Low-bit Attention" (structured summary), QK-norm: each token's query and
 * key vector is RMS-normalised, RMSNorm(x) = x / sqrt((1/d) sum_c x_c^2) * gamma, gamma a learnable
 * scale vector; the reproduction paragraph gives the norm epsilon 1e-6 (added to the mean square).
 *
 * sage_quantize_smooth_qknorm: as sage_quantize_smooth, on the normalised Q and K:
 *   r = the float32 nearest to 1 / sqrt(S / d + eps) per token, S = sum_c x_c^2 exactly
 *       (independent of any summation order; bf16 inputs need 2^-63 <= |x| < 2^63 or x = 0 for
 *       exact squares);
 *   y = rnd(fl32(fl32(x r) * gamma_c)) rounded to the input dtype, so the call equals a separate
 *       norm writing a 16-bit tensor followed by sage_quantize_smooth.  V is not normalised.
 *   Same workspace as sage_quantize_smooth.  With smooth_q = 1, Kn is required and is the K to
 *   pass to sage_attn_fwd / sage_attn_bwd (the Q-smoothing bias reads the normalised K).
 *   Errors: SAGE_ERR_ARG for a NULL qn, rQ or rK, a negative or non-finite eps, or smooth_q = 1
 *   without Kn; the rules of sage_quantize_smooth otherwise.
 * sage_qknorm_bwd: the gradient of y = gamma * x * r(x) for one of the two tensors (the rounding
 *   to 16 bits is taken as the identity), in float32:
 *   dX = r (gamma dY - xh * mean_c(gamma_c dY_c xh_c)), xh = x r;
 *   dg (nullable, (d) float32, overwritten) = sum over all B*H*N tokens of dY * xh, by float32
 *   reductions (not bit-reproducible).
 *   In: X (B,H,N,d) the raw Q or K (input dtype), g (nullable) its gamma, r the row factors the
 *   forward call wrote, dY (B,H,N,d) float32 (the gradient sage_attn_bwd wrote for the normalised
 *   tensor).  Out: dX (B,H,N,d) float32.  dX may not alias dY.
 * ------------------------------------------------------------------------------------------ */
typedef struct sage_qknorm {
    const float *gQ;   /* (d) float32 gamma of Q, or NULL for ones (device)                    */
    const float *gK;   /* (d) float32 gamma of K, or NULL for ones (device)                    */
    float eps;         /* added to the mean square; the pages' setup uses 1e-6                  */
    float *rQ;         /* out: (B,H,N) float32 row factors r of Q                               */
    float *rK;         /* out: (B,H,N) float32 row factors r of K                               */
    void *Qn;          /* out, nullable: (B,H,N,d) normalised Q in the input dtype              */
    void *Kn;          /* out, nullable (required when smooth_q = 1): normalised K              */
} sage_qknorm;

SAGE_API int sage_quantize_smooth_qknorm(const sage_params *p, const sage_qknorm *qn,
                         const void *Q, const void *K, const void *V, int8_t *Qh, int8_t *Kh,
                         int8_t *Vh, float *sQ, float *sK, float *sV, float *muK, float *muQ,
                         void *workspace, size_t workspace_bytes, sage_stream_t stream);
SAGE_API int sage_qknorm_bwd(const sage_params *p, const void *X, const float *g, const float *r,
                         const float *dY, float *dX, float *dg, sage_stream_t stream);

/* ------------------------------------------------------------------------------------------ *
 * FP4 inference forward (SageAttention3): sage_quantize_fp4 then sage_attn_fwd_fp4.
 * "SageAttention3: Microscaling FP4 Attention for Inference and An Exploration of 8-Bit
 * Training" (review): FP4 microscaling, eq. (2)-(3); the NVFP4 row of its format table (E2M1
 * values, 1 x 16 blocks, E4M3 scales); eq. (4)-(5) (S and O as FP4 products); two-level P
 * scaling, eq. (6); Q- and K-smoothing.
 *
 * sage_quantize_fp4: smoothing as sage_quantize_smooth (mu_K, and mu_Q when smooth_q), then per
 *   1 x 16 block s = e4m3(fl32(max|x| / 6)) (nearest E4M3, ties even) and codes
 *   e2m1(fl32(x / s)) (nearest E2M1: 0, 0.5, 1, 1.5, 2, 3, 4, 6; ties even; saturating; all zero
 *   where s = 0).
 *   Out: Qc, Kc, Vc (B,H,N,d/2) uint8, two codes a byte (the even element in the low nibble);
 *        sQ, sK (B,H,N,d/16) E4M3 bytes: Q and K blocked along d;
 *        sV (B,H,N/16,d) E4M3 bytes: V blocked along the tokens, 16 per channel;
 *        muK, muQ as sage_quantize_smooth.  Workspace: sage_quantize_workspace_bytes.
 * sage_attn_fwd_fp4: S = (s_Q Q^)(s_K K^)^T / sqrt(d) (+ the Q-smoothing bias, K required then),
 *   online softmax per 64-key tile; P~2 = fl32(2688 ex2(x)), x = logits - tile row max r, is
 *   quantised per 16 keys as above with codes e2m1(fl32(v fl32(1 / s))), and
 *   O += 2^(r - m) / 2688 * (s_P2 P^2)(s_V V^).  Writes O and L like sage_attn_fwd.  Workspace:
 *   sage_fwd_workspace_bytes.
 * Both calls refuse every flag (SAGE_ERR_UNSUPPORTED).  The tensor cores run the dequantised
 * values s * code, exact in fp16, through the same kind::f16 MMAs as the INT8 path.
 * ------------------------------------------------------------------------------------------ */
SAGE_API int sage_quantize_fp4(const sage_params *p, const void *Q, const void *K, const void *V,
                         uint8_t *Qc, uint8_t *Kc, uint8_t *Vc, uint8_t *sQ, uint8_t *sK,
                         uint8_t *sV, float *muK, float *muQ, void *workspace,
                         size_t workspace_bytes, sage_stream_t stream);
SAGE_API int sage_attn_fwd_fp4(const sage_params *p, const uint8_t *Qc, const uint8_t *Kc,
                         const uint8_t *Vc, const uint8_t *sQ, const uint8_t *sK,
                         const uint8_t *sV, const void *K, const float *muK, const float *muQ,
                         void *O, float *L, void *workspace, size_t workspace_bytes,
                         sage_stream_t stream);

/* ------------------------------------------------------------------------------------------ *
 * Step 2 -- forward.
 * "SageBwd: A Trainable Low-bit Attention" (structured summary), method steps, forward (3)-(5);
 * "SageAttention3 ..." (review) eq. (1) online softmax and eq. (8): S_ij = MM(Q^_i, K^_j) s_Q s_K,
 * s_P = exp(rowmax(S_ij) - m_ij) / 127 per token, P^_ij = P~_ij / s_P, O_ij accumulation; section
 * summary, A.1: the forward returns O and the log-sum-exp L.
 *
 * In:  Qh, Kh, Vh, sQ, sK, sV  as written by sage_quantize_smooth.
 *      K, muK, muQ             only when smooth_q = 1 (the bias mu_Qi . (K - mu_K)); else NULL.
 * Out: O  (B,H,N,d) fp16/bf16 (the dtype of p).
 *      L  (B,H,N) float32 natural-log log-sum-exp of the scaled logits S / sqrt(d) as formed
 *         (with K-smoothing these differ from the unsmoothed logits by a per-row constant).
 * Logits: S = fl32(acc * fl32(fl32(sQ sK) * fl32(log2(e) / sqrt(d)))) in log2 units; P codes are
 * round-half-even of fl32(127 * 2^fl32(S - r)) with r the row max of S over the 64-key tile; the
 * running sum l accumulates the unquantised probabilities.
 * ------------------------------------------------------------------------------------------ */
SAGE_API size_t sage_fwd_workspace_bytes(const sage_params *p);
SAGE_API int sage_attn_fwd(const sage_params *p, const int8_t *Qh, const int8_t *Kh, const int8_t *Vh,
                  const float *sQ, const float *sK, const float *sV, const void *K,
                  const float *muK, const float *muQ, void *O, float *L, void *workspace,
                  size_t workspace_bytes, sage_stream_t stream);

/* ------------------------------------------------------------------------------------------ *
 * Step 3 -- backward.
 * "SageBwd: A Trainable Low-bit Attention" (structured summary), method steps, backward (1)-(7):
 * D = rowsum(dO o O); recompute S_ij, P_ij; dV_j += MM(P^_ij^T, dO^_i) s_P s_dO; dP_ij = dO V_j^T in
 * 16 bits; dS_ij = P_ij o (dP_ij - D_i) quantised; dQ_i += MM(dS^_ij, K^_j) s_dS s_K;
 * dK_j += MM(dS^_ij^T, Q^_i) s_dS s_Q.  "SageAttention3 ..." (review), INT8 backward equations.
 *
 * In:  Qh, Kh, sQ, sK          the forward's codes and scales.
 *      K, muK, muQ             only when smooth_q = 1; else NULL.
 *      V, O, dO                (B,H,N,d) fp16/bf16: unquantised V, the stored forward output, dO.
 *      L                       (B,H,N) float32 from sage_attn_fwd.
 * Out: dQ, dK, dV              (B,H,N,d) float32, fully overwritten (the library zeroes them).
 * P and dS are quantised per 64x64 tile: s = fl32(max|x| / 127), code = the nearest integer
 * (ties to even) to the exact product x * fl32(1 / s) -- the nearest integer to
 * fl32(x * fl32(1 / s)) except within |x / s| 2^-24 of a half-integer; a tile whose max|x| is
 * below 2^-120 is a zero tile.  dO is quantised per 64-token block like Q.  dQ sums the tiles with
 * float32 reductions into global memory, so its last bits vary from run to run.
 * ------------------------------------------------------------------------------------------ */
SAGE_API size_t sage_bwd_workspace_bytes(const sage_params *p);
SAGE_API int sage_attn_bwd(const sage_params *p, const int8_t *Qh, const int8_t *Kh, const float *sQ,
                  const float *sK, const void *K, const float *muK, const float *muQ,
                  const void *V, const void *O, const float *L, const void *dO, float *dQ,
                  float *dK, float *dV, void *workspace, size_t workspace_bytes,
                  sage_stream_t stream);

/* ------------------------------------------------------------------------------------------ *
 * Step 1 without a workspace (the paper has no counterpart: this is a calling convenience).
 *
 * For callers that cannot allocate device memory while they run -- for example a plug-in whose
 * host framework owns all device memory and offers it no allocator, or a latency-critical loop
 * that must not pay for (or synchronise on) an allocation.  Same inputs, outputs, results and
 * parameter rules as sage_quantize_smooth, but the float64 K-mean partial sums live in a fixed
 * array inside the library (sage_quantize_noalloc_max_partials() entries, 1 MiB, held on every
 * device that loads the library until the process exits) instead of in a caller workspace.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - A call needs sage_quantize_noalloc_partials_needed(p) entries: (456 + B * H) * d + B * H
 *     with K-smoothing (a partial-sum slot of d entries for each of the pass's at most 456 CTAs
 *     and each head, and one entry of two 32-bit counters for each head), 0 without.  At
 *     d = 128 that admits B * H <= 563.  A call needing more than the capacity returns
 *     SAGE_ERR_WORKSPACE before any launch.  The query returns 0 for parameters the call would
 *     refuse.
 *   - The first call on a device looks up the array's device address on that device (the
 *     current device) and keeps it; make that first call before any stream capture.  The kept
 *     address is not refreshed after cudaDeviceReset: do not use this entry point on a device
 *     after resetting it in the same process.
 *   - Every call shares the one array, which keeps the last call's partial sums.  Nothing has to
 *     start at zero (each call writes every partial sum it reads first, and clears the counters
 *     on its stream before the launch), but calls that overlap on the GPU -- on different
 *     streams, or from different host threads -- race on it.
 *   - `flags` must be 0 or SAGE_FLAG_FP8 (no debug dump): SAGE_ERR_ARG otherwise.
 * ------------------------------------------------------------------------------------------ */
SAGE_API size_t sage_quantize_noalloc_max_partials(void);
SAGE_API size_t sage_quantize_noalloc_partials_needed(const sage_params *p);
SAGE_API int sage_quantize_smooth_noalloc(const sage_params *p, const void *Q, const void *K,
                                          const void *V, int8_t *Qh, int8_t *Kh, int8_t *Vh,
                                          float *sQ, float *sK, float *sV, float *muK, float *muQ,
                                          sage_stream_t stream);

/* ------------------------------------------------------------------------------------------ *
 * Attn-QAT: 4-bit attention trained with fake quantisation.
 * "Attn-QAT: 4-Bit Attention With Quantization-Aware Training" (technical summary), sections
 * 2.1-2.3: NVFP4 fake quantisation, no Q/K smoothing and no two-level P scaling; the backward
 * recomputes P with the forward's FP4 quantisation and forms D from a high-precision forward
 * output O'; the backward runs in 16 bits.
 * All three calls require flags = 0, smooth_k = 0 and smooth_q = 0 (SAGE_ERR_UNSUPPORTED
 * otherwise); pointers are device memory of the caller, 16-byte aligned (SAGE_ERR_ALIGN), and
 * asynchronous on `stream`.
 *
 * sage_qat_quantize -- Q' = s * code for Q, K (1 x 16 blocks along d) and V (16 tokens per
 *   channel), s = e4m3(fl32(max|x| / 6)), code = e2m1(fl32(x / s)) (nearest, ties to even,
 *   saturating at 6; a zero scale gives zero codes), written in the input type: the values have at
 *   most 6 significant bits and magnitudes in [2^-10, 2688], so they are exact.
 *   In: Q, K, V (B,H,N,d) fp16/bf16.  Out: Qf, Kf, Vf (B,H,N,d) same type.
 *
 * sage_qat_fwd -- per 64-key block, r = fl32(max acc * c) (c = fl32(log2(e) / sqrt(d)), acc the
 *   product Q' K'^T), e = ex2(fl32(fl32(acc c) - r)); P^ = phi(e), phi one-level NVFP4 over 16 keys
 *   (s = e4m3(fl32(max e / 6)), code = e2m1(fl32(e fl32(1/s)))); O = sum 2^(r - m) P^ V' / l,
 *   O' = sum 2^(r - m) rnd16(e) V' / l, l the running sum of e.
 *   In: Qf, Kf, Vf from sage_qat_quantize.
 *   Out: O (B,H,N,d) input type; Op = O' (B,H,N,d) float32; L (B,H,N) float32 natural-log LSE;
 *        R (B,H,N/64,N) float32: r of every (key block, query row) the forward visits (-inf when
 *        the row sees no key of the block); entries of pairs it never visits are left as they were.
 *
 * sage_qat_bwd -- P = ex2(fl32(acc c - L2)), L2 = fl32(L log2(e)); D = rowsum(dO o O');
 *   dP = dO V'^T; dS = fl32(P fl32(dP - D)) rounded to the input type; P^ = the forward's
 *   phi(ex2(fl32(fl32(acc c) - r))) times fl32(ex2(fl32(r - L2))), rounded to the input type;
 *   dV = P^^T dO; dQ = dS K' / sqrt(d); dK = dS^T Q' / sqrt(d) (fake quantisation passes the
 *   gradient straight through: these are the gradients of Q, K and V).
 *   In: Qf, Kf, Vf; Op, L, R from sage_qat_fwd; dO (B,H,N,d) input type.
 *   Out: dQ, dK, dV (B,H,N,d) float32, overwritten (dQ by float32 reductions: last bits vary).
 *   Workspace: sage_qat_bwd_workspace_bytes(p) bytes (D and L2), 256-byte aligned
 *   (SAGE_ERR_WORKSPACE when missing or short).
 * ------------------------------------------------------------------------------------------ */
SAGE_API int sage_qat_quantize(const sage_params *p, const void *Q, const void *K, const void *V,
                               void *Qf, void *Kf, void *Vf, sage_stream_t stream);
SAGE_API int sage_qat_fwd(const sage_params *p, const void *Qf, const void *Kf, const void *Vf,
                          void *O, float *Op, float *L, float *R, sage_stream_t stream);
SAGE_API size_t sage_qat_bwd_workspace_bytes(const sage_params *p);
SAGE_API int sage_qat_bwd(const sage_params *p, const void *Qf, const void *Kf, const void *Vf,
                          const float *Op, const float *L, const float *R, const void *dO,
                          float *dQ, float *dK, float *dV, void *workspace, size_t workspace_bytes,
                          sage_stream_t stream);

/* Bytes the SAGE_FLAG_DUMP buffer needs for a forward (which = 0) or backward (which = 1). */
SAGE_API size_t sage_dump_bytes(const sage_params *p, int which);

/* Waits for `stream`, then reads and clears the device-side error word of the current device:
 * SAGE_OK, or SAGE_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last call. */
SAGE_API int sage_device_status(sage_stream_t stream);

/* Human-readable name of a status code (static string). */
SAGE_API const char *sage_status_string(int status);

/* Library version string. */
SAGE_API const char *sage_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SAGE_GB300_H */
