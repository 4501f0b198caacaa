// sage_capi.cu -- the extern "C" boundary of libsage_gb300.so: argument checks, workspace
// layout, tensor-map construction and kernel launches.  No allocation happens here: every byte
// of device memory is the caller's.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <string.h>

#include "sage_internal.h"

namespace sage {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// (d, N, B*H) fp16 tensor, boxes of 64 x 128 x 1 with the 128-byte swizzle: rows past N of a
// head read as zeros.
bool make_tmap_3d(CUtensorMap *map, const void *ptr, int d, int N, uint64_t bh, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), bh};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_3d_bf16(CUtensorMap *map, const void *ptr, int d, int N, uint64_t bh, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), bh};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims,
                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------------------------
// workspace / dump layouts: consecutive 256-byte-aligned regions
// ------------------------------------------------------------------------------------------
struct Carve {
    uint8_t *base;
    size_t off = 0;
    explicit Carve(void *b) : base(static_cast<uint8_t *>(b)) {}
    template <typename T>
    T *take(size_t count) {
        off = (off + 255) & ~static_cast<size_t>(255);
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

static size_t elems(const sage_params &p) {
    return static_cast<size_t>(p.B) * p.H * p.N * p.d;
}
static size_t rows(const sage_params &p) { return static_cast<size_t>(p.B) * p.H * p.N; }
static size_t nblocks(const sage_params &p) { return static_cast<size_t>(p.B) * p.H * (p.N / 64); }

struct QuantWs {
    double *kpartial;
};
static QuantWs quant_ws(const sage_params &p, void *w, size_t *bytes) {
    Carve c(w);
    QuantWs r;
    // the FP4 quantiser's per-split partial sums, or the INT8 pass's per-CTA partials and barrier
    const size_t split = static_cast<size_t>(p.B) * p.H * kmean_splits(p) * p.d;
    const size_t fused = quant_fused_doubles(p);
    r.kpartial = c.take<double>(split > fused ? split : fused);
    if (bytes) *bytes = c.off;
    return r;
}

struct FwdWs {
    __half *q16, *k16, *v16;
    float *qbias;
};
static FwdWs fwd_ws(const sage_params &p, void *w, size_t *bytes) {
    Carve c(w);
    FwdWs r;
    // (with SAGE_FLAG_OPS16 the operand copies come from the caller's p->ops16)
    const bool own = !(p.flags & SAGE_FLAG_OPS16);
    r.q16 = own ? c.take<__half>(elems(p)) : nullptr;
    r.k16 = own ? c.take<__half>(elems(p)) : nullptr;
    r.v16 = own ? c.take<__half>(elems(p)) : nullptr;
    r.qbias = p.smooth_q ? c.take<float>(nblocks(p) * p.N) : nullptr;
    if (bytes) *bytes = c.off;
    return r;
}

struct BwdWs {
    __half *q16, *k16, *do16;
    float *D, *L2, *sdO, *qbias;
    int8_t *v8;      // SAGE_FLAG_DP_INT8: V codes, their fp16 copy and the block scales
    __half *v16;
    float *sV;
};
static BwdWs bwd_ws(const sage_params &p, void *w, size_t *bytes) {
    Carve c(w);
    BwdWs r;
    const bool own = !(p.flags & SAGE_FLAG_OPS16);
    r.q16 = own ? c.take<__half>(elems(p)) : nullptr;
    r.k16 = own ? c.take<__half>(elems(p)) : nullptr;
    r.do16 = c.take<__half>(elems(p));
    r.D = c.take<float>(rows(p));
    r.L2 = c.take<float>(rows(p));
    r.sdO = c.take<float>(nblocks(p));
    r.qbias = p.smooth_q ? c.take<float>(nblocks(p) * p.N) : nullptr;
    const bool dp8 = (p.flags & SAGE_FLAG_DP_INT8) != 0;
    r.v8 = dp8 ? c.take<int8_t>(elems(p)) : nullptr;
    r.v16 = dp8 ? c.take<__half>(elems(p)) : nullptr;
    r.sV = dp8 ? c.take<float>(nblocks(p)) : nullptr;
    if (bytes) *bytes = c.off;
    return r;
}

struct FwdDump {
    int32_t *s;
    int16_t *p;
    int32_t *pv;
};
static FwdDump fwd_dump(const sage_params &p, void *w, size_t *bytes) {
    Carve c(w);
    FwdDump r;
    const size_t nn = rows(p) * p.N;
    r.s = c.take<int32_t>(nn);
    r.p = c.take<int16_t>(nn);
    r.pv = c.take<int32_t>(nblocks(p) * (p.N / 64) * 64 * p.d);
    if (bytes) *bytes = c.off;
    return r;
}

struct BwdDump {
    int32_t *s;
    int16_t *p, *ds;
    float *sp, *sds;
    int8_t *doh;
    float *sdO, *D;
    float *dp;
    int32_t *dv, *dq, *dk;
};
static BwdDump bwd_dump(const sage_params &p, void *w, size_t *bytes) {
    Carve c(w);
    BwdDump r;
    const size_t nn = rows(p) * p.N;
    const size_t prod = nblocks(p) * (p.N / 64) * 64 * p.d;    // one 64 x d product per tile
    r.s = c.take<int32_t>(nn);
    r.p = c.take<int16_t>(nn);
    r.ds = c.take<int16_t>(nn);
    r.sp = c.take<float>(nblocks(p) * (p.N / 64));
    r.sds = c.take<float>(nblocks(p) * (p.N / 64));
    r.doh = c.take<int8_t>(elems(p));
    r.sdO = c.take<float>(nblocks(p));
    r.D = c.take<float>(rows(p));
    r.dp = c.take<float>(nn);
    r.dv = c.take<int32_t>(prod);
    r.dq = c.take<int32_t>(prod);
    r.dk = c.take<int32_t>(prod);
    if (bytes) *bytes = c.off;
    return r;
}

// ------------------------------------------------------------------------------------------
// argument checks
// ------------------------------------------------------------------------------------------
static bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// shared with sage_noalloc.cu (declared in sage_internal.h)
int check_params(const sage_params *p) {
    if (!p) return SAGE_ERR_ARG;
    if (p->B <= 0 || p->H <= 0 || p->N <= 0 || p->d <= 0) return SAGE_ERR_ARG;
    if (p->causal != 0 && p->causal != 1) return SAGE_ERR_ARG;
    if (p->smooth_k != 0 && p->smooth_k != 1) return SAGE_ERR_ARG;
    if (p->smooth_q != 0 && p->smooth_q != 1) return SAGE_ERR_ARG;
    if (p->flags & ~(SAGE_FLAG_DUMP | SAGE_FLAG_DP_INT8 | SAGE_FLAG_FP8 | SAGE_FLAG_OPS16)) return SAGE_ERR_ARG;
    if (p->flags & SAGE_FLAG_OPS16) {
        if (!p->ops16) return SAGE_ERR_ARG;
        if (reinterpret_cast<uintptr_t>(p->ops16) & 15u) return SAGE_ERR_ALIGN;
    }
    if ((p->flags & SAGE_FLAG_FP8) && (p->flags & (SAGE_FLAG_DUMP | SAGE_FLAG_DP_INT8))) return SAGE_ERR_UNSUPPORTED;
    if (p->dtype != SAGE_FP16 && p->dtype != SAGE_BF16) return SAGE_ERR_UNSUPPORTED;
    if (p->d != 64 && p->d != 128) return SAGE_ERR_UNSUPPORTED;
    if (p->N % 64 != 0) return SAGE_ERR_UNSUPPORTED;
    if (static_cast<long long>(p->B) * p->H > 65535) return SAGE_ERR_UNSUPPORTED;
    if (static_cast<long long>(p->N) > (1ll << 24)) return SAGE_ERR_UNSUPPORTED;
    return SAGE_OK;
}

static int check_ptrs(std::initializer_list<const void *> ptrs) {
    for (const void *q : ptrs) {
        if (!q) return SAGE_ERR_ARG;
        if (!aligned16(q)) return SAGE_ERR_ALIGN;
    }
    return SAGE_OK;
}

static int check_ws(void *ws, size_t have, size_t need) {
    if (need == 0) return SAGE_OK;
    if (!ws || have < need) return SAGE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SAGE_ERR_ALIGN;
    return SAGE_OK;
}

static int check_dump(const sage_params &p, int which) {
    if (!(p.flags & SAGE_FLAG_DUMP)) return SAGE_OK;
    size_t need = 0;
    if (which == 0) fwd_dump(p, nullptr, &need);
    else bwd_dump(p, nullptr, &need);
    if (!p.dump || p.dump_bytes < need) return SAGE_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(p.dump) & 255u) != 0) return SAGE_ERR_ALIGN;
    return SAGE_OK;
}

#define SAGE_TRY(x)                        \
    do {                                   \
        int _st = (x);                     \
        if (_st != SAGE_OK) return _st;    \
    } while (0)
#define SAGE_CUDA(x)                                  \
    do {                                              \
        if ((x) != cudaSuccess) return SAGE_ERR_CUDA; \
    } while (0)

}  // namespace sage

using namespace sage;

extern "C" {

size_t sage_quantize_workspace_bytes(const sage_params *p) {
    if (check_params(p) != SAGE_OK || !p->smooth_k) return 0;
    size_t b = 0;
    quant_ws(*p, nullptr, &b);
    return b;
}

}  // extern "C"

// sage_quantize_smooth and its QK-norm form (qn != NULL)
static int quantize_call(const sage_params *p, const sage_qknorm *qn, const void *Q, const void *K,
                         const void *V, int8_t *Qh, int8_t *Kh, int8_t *Vh, float *sQ, float *sK,
                         float *sV, float *muK, float *muQ, void *workspace, size_t workspace_bytes,
                         sage_stream_t stream) {
    SAGE_TRY(check_params(p));
    if (qn) {
        if (!(qn->eps >= 0.0f) || !(qn->eps <= 3.0e38f)) return SAGE_ERR_ARG;   // NaN, < 0 or inf
        SAGE_TRY(check_ptrs({qn->rQ, qn->rK}));
        const void *opt[] = {qn->gQ, qn->gK, qn->Qn, qn->Kn};
        for (const void *q : opt)
            if (q && !aligned16(q)) return SAGE_ERR_ALIGN;
        if (p->smooth_q && !qn->Kn) return SAGE_ERR_ARG;
    }
    SAGE_TRY(check_ptrs({Q, K, V, Qh, Kh, Vh, sQ, sK, sV, muK}));
    if (p->smooth_q) SAGE_TRY(check_ptrs({muQ}));
    SAGE_TRY(check_ws(workspace, workspace_bytes, sage_quantize_workspace_bytes(p)));
    QuantArgs a;
    memset(&a, 0, sizeof(a));
    a.Q = Q; a.K = K; a.V = V;
    a.Qh = Qh; a.Kh = Kh; a.Vh = Vh;
    a.sQ = sQ; a.sK = sK; a.sV = sV;
    a.muK = muK; a.muQ = p->smooth_q ? muQ : nullptr;
    a.ksplits = kmean_splits(*p);
    QuantWs w = quant_ws(*p, p->smooth_k ? workspace : nullptr, nullptr);
    a.kpartial = w.kpartial;
    a.N = p->N; a.d = p->d; a.smooth_k = p->smooth_k; a.smooth_q = p->smooth_q;
    a.fp8 = (p->flags & SAGE_FLAG_FP8) != 0;
    a.ops16 = (p->flags & SAGE_FLAG_OPS16) ? static_cast<__half *>(p->ops16) : nullptr;
    QkNormArgs na{};
    if (qn) {
        a.qk_norm = 1;
        na.eps = qn->eps;
        na.gamma[0] = qn->gQ; na.gamma[1] = qn->gK;
        na.rnorm[0] = qn->rQ; na.rnorm[1] = qn->rK;
        na.xnorm[0] = qn->Qn; na.xnorm[1] = qn->Kn;
    }
    SAGE_CUDA(launch_quantize(*p, a, reinterpret_cast<cudaStream_t>(stream), qn ? &na : nullptr));
    return SAGE_OK;
}

extern "C" {

int sage_quantize_smooth(const sage_params *p, const void *Q, const void *K, const void *V,
                         int8_t *Qh, int8_t *Kh, int8_t *Vh, float *sQ, float *sK, float *sV,
                         float *muK, float *muQ, void *workspace, size_t workspace_bytes,
                         sage_stream_t stream) {
    return quantize_call(p, nullptr, Q, K, V, Qh, Kh, Vh, sQ, sK, sV, muK, muQ, workspace,
                         workspace_bytes, stream);
}

int sage_quantize_smooth_qknorm(const sage_params *p, const sage_qknorm *qn, const void *Q,
                                const void *K, const void *V, int8_t *Qh, int8_t *Kh, int8_t *Vh,
                                float *sQ, float *sK, float *sV, float *muK, float *muQ,
                                void *workspace, size_t workspace_bytes, sage_stream_t stream) {
    if (!qn) return SAGE_ERR_ARG;
    return quantize_call(p, qn, Q, K, V, Qh, Kh, Vh, sQ, sK, sV, muK, muQ, workspace,
                         workspace_bytes, stream);
}

int sage_qknorm_bwd(const sage_params *p, const void *X, const float *g, const float *r,
                    const float *dY, float *dX, float *dg, sage_stream_t stream) {
    SAGE_TRY(check_params(p));
    SAGE_TRY(check_ptrs({X, r, dY, dX}));
    if ((g && !aligned16(g)) || (dg && !aligned16(dg))) return SAGE_ERR_ALIGN;
    if (static_cast<const void *>(dX) == static_cast<const void *>(dY)) return SAGE_ERR_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dg) SAGE_CUDA(cudaMemsetAsync(dg, 0, static_cast<size_t>(p->d) * sizeof(float), st));
    SAGE_CUDA(launch_qknorm_bwd(*p, X, g, r, dY, dX, dg, st));
    return SAGE_OK;
}

size_t sage_fwd_workspace_bytes(const sage_params *p) {
    if (check_params(p) != SAGE_OK) return 0;
    size_t b = 0;
    fwd_ws(*p, nullptr, &b);
    return b;
}

int sage_attn_fwd(const sage_params *p, const int8_t *Qh, const int8_t *Kh, const int8_t *Vh,
                  const float *sQ, const float *sK, const float *sV, const void *K,
                  const float *muK, const float *muQ, void *O, float *L, void *workspace,
                  size_t workspace_bytes, sage_stream_t stream) {
    SAGE_TRY(check_params(p));
    SAGE_TRY(check_ptrs({Qh, Kh, Vh, sQ, sK, sV, O, L}));
    if (p->smooth_q) SAGE_TRY(check_ptrs({K, muK, muQ}));
    SAGE_TRY(check_ws(workspace, workspace_bytes, sage_fwd_workspace_bytes(p)));
    SAGE_TRY(check_dump(*p, 0));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    FwdWs w = fwd_ws(*p, workspace, nullptr);
    const size_t n = elems(*p);
    const bool fp8 = (p->flags & SAGE_FLAG_FP8) != 0;
    if (p->flags & SAGE_FLAG_OPS16) {
        // the quantiser wrote the operand copies (Q^, K^, V^ in that order)
        const __half *o16 = static_cast<const __half *>(p->ops16);
        w.q16 = const_cast<__half *>(o16);
        w.k16 = const_cast<__half *>(o16 + n);
        w.v16 = const_cast<__half *>(o16 + 2 * n);
    } else {
        SAGE_CUDA(launch_widen(Qh, w.q16, n, fp8, st));
        SAGE_CUDA(launch_widen(Kh, w.k16, n, fp8, st));
        SAGE_CUDA(launch_widen(Vh, w.v16, n, fp8, st));
    }
    const float sl2 = scale_log2(p->d);
    if (p->smooth_q) SAGE_CUDA(launch_qbias(*p, K, muK, muQ, w.qbias, sl2, st));
    FwdArgs a;
    memset(&a, 0, sizeof(a));
    a.sQ = sQ; a.sK = sK; a.sV = sV;
    a.qbias = w.qbias;
    a.O = O; a.L = L;
    if (p->flags & SAGE_FLAG_DUMP) {
        FwdDump dd = fwd_dump(*p, p->dump, nullptr);
        a.dump_s = dd.s; a.dump_p = dd.p; a.dump_pv = dd.pv;
    }
    a.N = p->N; a.H = p->H; a.causal = p->causal; a.dtype = p->dtype;
    a.sl2 = sl2;
    SAGE_CUDA(launch_fwd(*p, w.q16, w.k16, w.v16, a, st));
    return SAGE_OK;
}

int sage_quantize_fp4(const sage_params *p, const void *Q, const void *K, const void *V,
                      uint8_t *Qc, uint8_t *Kc, uint8_t *Vc, uint8_t *sQ, uint8_t *sK, uint8_t *sV,
                      float *muK, float *muQ, void *workspace, size_t workspace_bytes,
                      sage_stream_t stream) {
    SAGE_TRY(check_params(p));
    if (p->flags) return SAGE_ERR_UNSUPPORTED;
    SAGE_TRY(check_ptrs({Q, K, V, Qc, Kc, Vc, sQ, sK, sV, muK}));
    if (p->smooth_q) SAGE_TRY(check_ptrs({muQ}));
    SAGE_TRY(check_ws(workspace, workspace_bytes, sage_quantize_workspace_bytes(p)));
    QuantArgs a;
    memset(&a, 0, sizeof(a));
    a.Q = Q; a.K = K; a.V = V;
    a.muK = muK; a.muQ = p->smooth_q ? muQ : nullptr;
    a.ksplits = kmean_splits(*p);
    a.kpartial = quant_ws(*p, p->smooth_k ? workspace : nullptr, nullptr).kpartial;
    a.N = p->N; a.d = p->d; a.smooth_k = p->smooth_k; a.smooth_q = p->smooth_q;
    Fp4Out o{Qc, Kc, Vc, sQ, sK, sV};
    SAGE_CUDA(launch_quantize_fp4(*p, a, o, reinterpret_cast<cudaStream_t>(stream)));
    return SAGE_OK;
}

int sage_attn_fwd_fp4(const sage_params *p, const uint8_t *Qc, const uint8_t *Kc, const uint8_t *Vc,
                      const uint8_t *sQ, const uint8_t *sK, const uint8_t *sV, const void *K,
                      const float *muK, const float *muQ, void *O, float *L, void *workspace,
                      size_t workspace_bytes, sage_stream_t stream) {
    SAGE_TRY(check_params(p));
    if (p->flags) return SAGE_ERR_UNSUPPORTED;
    SAGE_TRY(check_ptrs({Qc, Kc, Vc, sQ, sK, sV, O, L}));
    if (p->smooth_q) SAGE_TRY(check_ptrs({K, muK, muQ}));
    SAGE_TRY(check_ws(workspace, workspace_bytes, sage_fwd_workspace_bytes(p)));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    FwdWs w = fwd_ws(*p, workspace, nullptr);
    SAGE_CUDA(launch_widen_fp4(Qc, sQ, w.q16, *p, false, st));
    SAGE_CUDA(launch_widen_fp4(Kc, sK, w.k16, *p, false, st));
    SAGE_CUDA(launch_widen_fp4(Vc, sV, w.v16, *p, true, st));
    const float sl2 = scale_log2(p->d);
    if (p->smooth_q) SAGE_CUDA(launch_qbias(*p, K, muK, muQ, w.qbias, sl2, st));
    FwdArgs a;
    memset(&a, 0, sizeof(a));
    a.qbias = w.qbias;
    a.O = O; a.L = L;
    a.N = p->N; a.H = p->H; a.causal = p->causal; a.dtype = p->dtype;
    a.sl2 = sl2;
    a.fp4 = 1;
    SAGE_CUDA(launch_fwd(*p, w.q16, w.k16, w.v16, a, st));
    return SAGE_OK;
}

size_t sage_bwd_workspace_bytes(const sage_params *p) {
    if (check_params(p) != SAGE_OK) return 0;
    size_t b = 0;
    bwd_ws(*p, nullptr, &b);
    return b;
}

int sage_attn_bwd(const sage_params *p, const int8_t *Qh, const int8_t *Kh, const float *sQ,
                  const float *sK, const void *K, const float *muK, const float *muQ,
                  const void *V, const void *O, const float *L, const void *dO, float *dQ,
                  float *dK, float *dV, void *workspace, size_t workspace_bytes,
                  sage_stream_t stream) {
    SAGE_TRY(check_params(p));
    SAGE_TRY(check_ptrs({Qh, Kh, sQ, sK, V, O, L, dO, dQ, dK, dV}));
    if (p->smooth_q) SAGE_TRY(check_ptrs({K, muK, muQ}));
    SAGE_TRY(check_ws(workspace, workspace_bytes, sage_bwd_workspace_bytes(p)));
    SAGE_TRY(check_dump(*p, 1));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    BwdWs w = bwd_ws(*p, workspace, nullptr);
    const size_t n = elems(*p);
    BwdDump dd;
    memset(&dd, 0, sizeof(dd));
    if (p->flags & SAGE_FLAG_DUMP) dd = bwd_dump(*p, p->dump, nullptr);
    const bool fp8 = (p->flags & SAGE_FLAG_FP8) != 0;
    if (p->flags & SAGE_FLAG_OPS16) {
        const __half *o16 = static_cast<const __half *>(p->ops16);
        w.q16 = const_cast<__half *>(o16);
        w.k16 = const_cast<__half *>(o16 + n);
    } else {
        SAGE_CUDA(launch_widen(Qh, w.q16, n, fp8, st));
        SAGE_CUDA(launch_widen(Kh, w.k16, n, fp8, st));
    }
    const bool dp8 = (p->flags & SAGE_FLAG_DP_INT8) != 0;
    if (dp8) {
        // V codes for dP (the ablation): the same per-block quantiser as sage_quantize_smooth
        QuantArgs qa;
        memset(&qa, 0, sizeof(qa));
        qa.V = V; qa.Vh = w.v8; qa.sV = w.sV;
        qa.N = p->N; qa.d = p->d;
        SAGE_CUDA(launch_quantize_v(*p, qa, st));
        SAGE_CUDA(launch_widen(w.v8, w.v16, n, false, st));
    }
    BwdPrologueArgs pa;
    pa.dO = dO; pa.O = O; pa.L = L; pa.L2 = w.L2; pa.D = w.D; pa.dO16 = w.do16; pa.dOh = dd.doh; pa.sdO = w.sdO;
    pa.N = p->N; pa.d = p->d; pa.fp8 = fp8;
    SAGE_CUDA(launch_bwd_prologue(*p, pa, st));
    const float sl2 = scale_log2(p->d);
    if (p->smooth_q) SAGE_CUDA(launch_qbias(*p, K, muK, muQ, w.qbias, sl2, st));
    SAGE_CUDA(cudaMemsetAsync(dQ, 0, n * sizeof(float), st));
    BwdArgs a;
    memset(&a, 0, sizeof(a));
    a.sQ = sQ; a.sK = sK; a.sdO = w.sdO; a.D = w.D; a.L2 = w.L2; a.sV = w.sV;
    a.qbias = w.qbias; a.muQ = p->smooth_q ? muQ : nullptr;
    a.dQ = dQ; a.dK = dK; a.dV = dV;
    if (p->flags & SAGE_FLAG_DUMP) {
        a.dump_s = dd.s; a.dump_p = dd.p; a.dump_ds = dd.ds; a.dump_sp = dd.sp; a.dump_sds = dd.sds;
        a.dump_dp = dd.dp; a.dump_dv = dd.dv; a.dump_dq = dd.dq; a.dump_dk = dd.dk;
        SAGE_CUDA(cudaMemcpyAsync(dd.sdO, w.sdO, nblocks(*p) * sizeof(float), cudaMemcpyDeviceToDevice, st));
        SAGE_CUDA(cudaMemcpyAsync(dd.D, w.D, rows(*p) * sizeof(float), cudaMemcpyDeviceToDevice, st));
    }
    a.N = p->N; a.H = p->H; a.causal = p->causal; a.dtype = p->dtype;
    a.sl2 = sl2;
    a.inv_sqrt_d = static_cast<float>(1.0 / __builtin_sqrt(static_cast<double>(p->d)));
    // the ablation feeds dP from the codes: V^ instead of V, dO^ instead of dO
    SAGE_CUDA(launch_bwd(*p, w.q16, w.k16, dp8 ? static_cast<const void *>(w.v16) : V,
                         dp8 ? static_cast<const void *>(w.do16) : dO, w.do16, a, st));
    return SAGE_OK;
}

// Attn-QAT entries: no flags, no smoothing
static int check_qat(const sage_params *p) {
    SAGE_TRY(check_params(p));
    if (p->flags || p->smooth_k || p->smooth_q) return SAGE_ERR_UNSUPPORTED;
    return SAGE_OK;
}

int sage_qat_quantize(const sage_params *p, const void *Q, const void *K, const void *V,
                      void *Qf, void *Kf, void *Vf, sage_stream_t stream) {
    SAGE_TRY(check_qat(p));
    SAGE_TRY(check_ptrs({Q, K, V, Qf, Kf, Vf}));
    SAGE_CUDA(launch_qat_fake_quant(*p, Q, K, V, Qf, Kf, Vf, reinterpret_cast<cudaStream_t>(stream)));
    return SAGE_OK;
}

int sage_qat_fwd(const sage_params *p, const void *Qf, const void *Kf, const void *Vf, void *O,
                 float *Op, float *L, float *R, sage_stream_t stream) {
    SAGE_TRY(check_qat(p));
    SAGE_TRY(check_ptrs({Qf, Kf, Vf, O, Op, L, R}));
    FwdArgs a;
    memset(&a, 0, sizeof(a));
    a.O = O; a.L = L; a.R = R;
    a.N = p->N; a.H = p->H; a.causal = p->causal; a.dtype = p->dtype;
    a.sl2 = scale_log2(p->d);
    SAGE_CUDA(launch_fwd_qat(*p, Qf, Kf, Vf, a, Op, reinterpret_cast<cudaStream_t>(stream)));
    return SAGE_OK;
}

size_t sage_qat_bwd_workspace_bytes(const sage_params *p) {
    if (check_qat(p) != SAGE_OK) return 0;
    return 2 * ((rows(*p) * sizeof(float) + 255) & ~static_cast<size_t>(255));
}

int sage_qat_bwd(const sage_params *p, const void *Qf, const void *Kf, const void *Vf, const float *Op,
                 const float *L, const float *R, const void *dO, float *dQ, float *dK, float *dV,
                 void *workspace, size_t workspace_bytes, sage_stream_t stream) {
    SAGE_TRY(check_qat(p));
    SAGE_TRY(check_ptrs({Qf, Kf, Vf, Op, L, R, dO, dQ, dK, dV}));
    SAGE_TRY(check_ws(workspace, workspace_bytes, sage_qat_bwd_workspace_bytes(p)));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Carve c(workspace);
    float *D = c.take<float>(rows(*p));
    float *L2 = c.take<float>(rows(*p));
    SAGE_CUDA(launch_qat_bwd_prologue(*p, dO, Op, L, L2, D, st));
    SAGE_CUDA(cudaMemsetAsync(dQ, 0, elems(*p) * sizeof(float), st));
    BwdArgs a;
    memset(&a, 0, sizeof(a));
    a.D = D; a.L2 = L2; a.R = R;
    a.dQ = dQ; a.dK = dK; a.dV = dV;
    a.N = p->N; a.H = p->H; a.causal = p->causal; a.dtype = p->dtype;
    a.sl2 = scale_log2(p->d);
    a.inv_sqrt_d = static_cast<float>(1.0 / __builtin_sqrt(static_cast<double>(p->d)));
    SAGE_CUDA(launch_bwd_qat(*p, Qf, Kf, Vf, dO, a, st));
    return SAGE_OK;
}

size_t sage_dump_bytes(const sage_params *p, int which) {
    if (check_params(p) != SAGE_OK) return 0;
    size_t b = 0;
    if (which == 0) fwd_dump(*p, nullptr, &b);
    else bwd_dump(*p, nullptr, &b);
    return b;
}

int sage_device_status(sage_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SAGE_ERR_CUDA;
    const unsigned int e = take_fwd_error() | take_bwd_error() | take_quant_error();
    if (cudaGetLastError() != cudaSuccess) return SAGE_ERR_CUDA;
    return e ? SAGE_ERR_TIMEOUT : SAGE_OK;
}

const char *sage_status_string(int status) {
    switch (status) {
        case SAGE_OK: return "ok";
        case SAGE_ERR_ARG: return "invalid argument";
        case SAGE_ERR_UNSUPPORTED: return "unsupported problem (d, N or dtype)";
        case SAGE_ERR_ALIGN: return "device pointer not 16-byte aligned";
        case SAGE_ERR_CUDA: return "CUDA launch or runtime error";
        case SAGE_ERR_TIMEOUT: return "device-side bounded wait expired";
        case SAGE_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

const char *sage_version(void) { return "sage-gb300 0.1 (sm_103a, tcgen05 kind::f16 integer-valued)"; }

}  // extern "C"
