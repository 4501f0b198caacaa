// sage_internal.h -- declarations shared by the translation units of libsage_gb300.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <type_traits>

#include "../../include/sage.h"

namespace sage {

constexpr float kLog2e = 1.4426950408889634f;   // log2(e) rounded to float32

// log2(e) / sqrt(d) rounded once to float32 (the double quotient is formed first)
inline float scale_log2(int d) {
    return static_cast<float>(1.4426950408889634 / __builtin_sqrt(static_cast<double>(d)));
}

struct QuantArgs {
    const void *Q, *K, *V;
    int8_t *Qh, *Kh, *Vh;
    float *sQ, *sK, *sV, *muK, *muQ;
    const double *kpartial;   // (B*H, ksplits, d) float64 partial sums of K (workspace)
    int ksplits;
    int N, d, smooth_k, smooth_q;
    int fp8;                  // 1: E4M3 codes, delta = max|x| / 448 (SAGE_FLAG_FP8)
    int qk_norm;              // 1: QK-norm prologue (arguments in QkNormArgs)
    __half *ops16;            // SAGE_FLAG_OPS16: (3,B,H,N,d) fp16 copies of the codes, else NULL
};

// QK-norm prologue: Q (index 0) and K (index 1) are RMS-normalised per token.  A kernel parameter
// of its own: folding these fields into QuantArgs raised the plain quantiser's register count.
struct QkNormArgs {
    float eps;
    const float *gamma[2];    // (d) scales or NULL (ones)
    float *rnorm[2];          // (B,H,N) row factors (written)
    void *xnorm[2];           // (B,H,N,d) normalised 16-bit tensors or NULL
};

// NVFP4 outputs of the FP4 quantiser: packed E2M1 codes (two per byte, the even element in the
// low nibble) and E4M3 block scales (one byte each)
struct Fp4Out {
    uint8_t *Qc, *Kc, *Vc;    // (B,H,N,d/2)
    uint8_t *sQ, *sK;         // (B,H,N,d/16): blocks of 16 channels
    uint8_t *sV;              // (B,H,N/16,d): blocks of 16 tokens per channel
};

struct BwdPrologueArgs {
    const void *dO, *O;
    const float *L;    // (B,H,N) log-sum-exp from the forward
    float *L2;         // (B,H,N) -fl32(L * log2 e) (negated), read by the backward kernel
    float *D;          // (B,H,N)
    __half *dO16;      // (B,H,N,d) integer-valued fp16 codes of dO
    int8_t *dOh;       // optional int8 codes of dO (debug dump), may be NULL
    float *sdO;        // (B,H,N/64)
    int N, d;
    int fp8;           // 1: the dO codes are E4M3 values (SAGE_FLAG_FP8)
};

// Forward kernel arguments (device pointers; tensor maps are separate __grid_constant__ params)
struct FwdArgs {
    const float *sQ, *sK, *sV;
    const float *qbias;   // (B,H,N/64,N) log2-unit Q-smoothing bias or NULL
    void *O;              // (B,H,N,d) 16-bit
    float *L;             // (B,H,N)
    int32_t *dump_s;      // debug: (B,H,N,N) integer S products, or NULL
    int16_t *dump_p;      // debug: (B,H,N,N) P codes, or NULL
    int32_t *dump_pv;     // debug: (B,H,N/64,N/64,64,d) integer P V products, or NULL
    int N, H, causal, dtype;
    float sl2;            // log2(e)/sqrt(d)
    int fp4;              // 1: FP4 inference forward (dequantised NVFP4 operands, two-level P)
    float *R;             // Attn-QAT: (B,H,N/64,N) row maxima r of each (key block, row), or NULL
};

struct BwdArgs {
    const float *sQ, *sK, *sdO, *D, *L2;   // D and -fl32(L log2 e) (negated): (B,H,N), from the prologue
    const float *sV;      // (B,H,N/64) V block scales (SAGE_FLAG_DP_INT8 only), else NULL
    const float *qbias;   // (B,H,N/64,N) or NULL
    const float *muQ;     // (B,H,N/64,d) or NULL (Q-smoothing dK bias term)
    float *dQ, *dK, *dV;  // (B,H,N,d) float32
    int32_t *dump_s;      // debug: (B,H,N,N) integer S products
    int16_t *dump_p;      // debug: (B,H,N,N) backward P codes
    int16_t *dump_ds;     // debug: (B,H,N,N) dS codes
    float *dump_sp;       // debug: (B,H,N/64,N/64) P tile scales
    float *dump_sds;      // debug: (B,H,N/64,N/64) dS tile scales
    float *dump_dp;       // debug: (B,H,N,N) dP as the score warpgroup uses it
    int32_t *dump_dv;     // debug: (B,H,N/64,N/64,64,d) integer P^T dO^ block products [i][j][key][c]
    int32_t *dump_dq;     // debug: (B,H,N/64,N/64,64,d) integer dS^ K^ block products [i][j][q][c]
    int32_t *dump_dk;     // debug: (B,H,N/64,N/64,64,d) integer dS^T Q^ block products [i][j][key][c]
    const float *R;       // Attn-QAT: the forward's row maxima (B,H,N/64,N), else NULL
    int N, H, causal, dtype;
    float sl2, inv_sqrt_d;
};

// sage_capi.cu: the parameter rules every entry point applies (SAGE_OK or a status code)
int check_params(const sage_params *p);

// sage_quant.cu
int kmean_splits(const sage_params &p);
cudaError_t launch_quantize(const sage_params &p, QuantArgs a, cudaStream_t st,
                            const QkNormArgs *qn = nullptr);
cudaError_t launch_quantize_v(const sage_params &p, QuantArgs a, cudaStream_t st);   // V only
unsigned int take_quant_error();
// float64 words of quantiser scratch the INT8 pass needs with K-smoothing (partial sums, barrier)
size_t quant_fused_doubles(const sage_params &p);
// NVFP4 quantisation of Q, K (along d) and V (along the tokens), smoothed as for INT8
cudaError_t launch_quantize_fp4(const sage_params &p, QuantArgs a, Fp4Out o, cudaStream_t st);
// NVFP4 codes and scales -> the exact fp16 values s * code (along_tokens: V's scale layout)
cudaError_t launch_widen_fp4(const uint8_t *codes, const uint8_t *scales, __half *dst,
                             const sage_params &p, bool along_tokens, cudaStream_t st);
// int8 codes (or E4M3 bit patterns when fp8) -> their exact fp16 values
cudaError_t launch_widen(const int8_t *src, __half *dst, size_t n, bool fp8, cudaStream_t st);
cudaError_t launch_bwd_prologue(const sage_params &p, BwdPrologueArgs a, cudaStream_t st);
// Attn-QAT: NVFP4 fake quantisation of Q, K, V into the input 16-bit type (no smoothing), and the
// backward prologue D = rowsum(dO o O') (O' float32), L2 = -fl32(L log2 e)
cudaError_t launch_qat_fake_quant(const sage_params &p, const void *Q, const void *K, const void *V,
                                  void *Qf, void *Kf, void *Vf, cudaStream_t st);
cudaError_t launch_qat_bwd_prologue(const sage_params &p, const void *dO, const float *Op, const float *L,
                                    float *L2, float *D, cudaStream_t st);
// gradient of the QK-norm: dX = r (g dY - xh mean(g dY xh)), xh = x r; dg (nullable, zeroed by
// the caller) += sum over rows of dY xh
cudaError_t launch_qknorm_bwd(const sage_params &p, const void *X, const float *g, const float *r,
                              const float *dY, float *dX, float *dg, cudaStream_t st);
cudaError_t launch_qbias(const sage_params &p, const void *K, const float *muK, const float *muQ,
                         float *bias, float sl2, cudaStream_t st);

// sage_fwd.cu
cudaError_t launch_fwd(const sage_params &p, const __half *Q16, const __half *K16,
                       const __half *V16, FwdArgs a, cudaStream_t st);
// Attn-QAT: the forward over fake-quantised Q', K', V' in the input type (a.O, a.L), then O' into Op
cudaError_t launch_fwd_qat(const sage_params &p, const void *Qf, const void *Kf, const void *Vf, FwdArgs a,
                           float *Op, cudaStream_t st);
unsigned int take_fwd_error();

// sage_bwd.cu
cudaError_t launch_bwd(const sage_params &p, const __half *Q16, const __half *K16,
                       const void *V, const void *dO, const __half *dO16, BwdArgs a,
                       cudaStream_t st);
// Attn-QAT backward: S^T, dP^T, dV, dK, dQ on the fake-quantised Q', K', V' and dO, all in the
// input 16-bit type (a.R, a.L2, a.D set; the scale pointers unused)
cudaError_t launch_bwd_qat(const sage_params &p, const void *Qf, const void *Kf, const void *Vf,
                           const void *dO, BwdArgs a, cudaStream_t st);
unsigned int take_bwd_error();

// tensor maps (sage_capi.cu)
// (d, N, B*H) 16-bit tensor maps with 64 x box_rows boxes and the 128-byte swizzle
bool make_tmap_3d(CUtensorMap *map, const void *ptr, int d, int N, uint64_t bh, uint32_t box_rows = 128);
bool make_tmap_3d_bf16(CUtensorMap *map, const void *ptr, int d, int N, uint64_t bh, uint32_t box_rows = 128);

}  // namespace sage
