// sage_noalloc.cu -- sage_quantize_smooth_noalloc: the quantise step without caller scratch.
//
// sage_quantize_smooth needs a small scratch buffer for the float64 partial sums of K (the
// K-mean).  Some callers have no way to provide one: code that must not call cudaMalloc or an
// allocator at all once it is running, such as a plug-in whose host framework owns every byte of
// device memory and exposes no allocator to it, or a latency-critical loop where an allocation
// (which may synchronise the device) is not acceptable.  This entry point serves them: it keeps
// the partial sums in a fixed array inside the library itself and otherwise runs exactly the same
// kernels as sage_quantize_smooth.
#include <mutex>

#include "sage_internal.h"

namespace sage {

// Capacity of the library-resident scratch, in float64 partial sums (1 MiB).  Every GPU that
// loads the library holds this array until the process exits.
constexpr size_t kNoallocPartials = 131072;

static __device__ __align__(256) double g_noalloc_kpartial[kNoallocPartials];

// Device address of the array on each device, looked up once per device (the host-side name of
// the array is not a device address and must never be handed to a kernel).
static constexpr int kMaxDevices = 64;
static double *g_noalloc_ptr[kMaxDevices];
static std::once_flag g_noalloc_once[kMaxDevices];
static cudaError_t g_noalloc_status[kMaxDevices];

static double *noalloc_scratch(int device) {
    std::call_once(g_noalloc_once[device], [device]() {
        void *ptr = nullptr;
        g_noalloc_status[device] = cudaGetSymbolAddress(&ptr, g_noalloc_kpartial);
        g_noalloc_ptr[device] = g_noalloc_status[device] == cudaSuccess ? static_cast<double *>(ptr) : nullptr;
    });
    return g_noalloc_ptr[device];
}

}  // namespace sage

using namespace sage;

extern "C" size_t sage_quantize_noalloc_max_partials(void) { return kNoallocPartials; }

extern "C" int sage_quantize_smooth_noalloc(const sage_params *p, const void *Q, const void *K,
                                            const void *V, int8_t *Qh, int8_t *Kh, int8_t *Vh,
                                            float *sQ, float *sK, float *sV, float *muK,
                                            float *muQ, sage_stream_t stream) {
    // same argument rules as sage_quantize_smooth; the caller passes no workspace
    if (!p) return SAGE_ERR_ARG;
    if (p->B <= 0 || p->H <= 0 || p->N <= 0 || p->d <= 0) return SAGE_ERR_ARG;
    if ((p->causal | p->smooth_k | p->smooth_q) & ~1) return SAGE_ERR_ARG;
    if (p->flags & ~SAGE_FLAG_FP8) return SAGE_ERR_ARG;
    if (p->dtype != SAGE_FP16 && p->dtype != SAGE_BF16) return SAGE_ERR_UNSUPPORTED;
    if ((p->d != 64 && p->d != 128) || p->N % 64 != 0) return SAGE_ERR_UNSUPPORTED;
    if (static_cast<long long>(p->B) * p->H > 65535) return SAGE_ERR_UNSUPPORTED;
    const void *ptrs[] = {Q, K, V, Qh, Kh, Vh, sQ, sK, sV, muK};
    for (const void *q : ptrs) {
        if (!q) return SAGE_ERR_ARG;
        if (reinterpret_cast<uintptr_t>(q) & 15u) return SAGE_ERR_ALIGN;
    }
    if (p->smooth_q) {
        if (!muQ) return SAGE_ERR_ARG;
        if (reinterpret_cast<uintptr_t>(muQ) & 15u) return SAGE_ERR_ALIGN;
    }
    const int splits = kmean_splits(*p);
    const size_t need = static_cast<size_t>(p->B) * p->H * splits * p->d;
    if (p->smooth_k && need > kNoallocPartials) return SAGE_ERR_WORKSPACE;   // beyond the static scratch

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) return SAGE_ERR_CUDA;
    double *scratch = noalloc_scratch(device);
    if (!scratch) return SAGE_ERR_CUDA;

    QuantArgs a{};
    a.Q = Q; a.K = K; a.V = V;
    a.Qh = Qh; a.Kh = Kh; a.Vh = Vh;
    a.sQ = sQ; a.sK = sK; a.sV = sV;
    a.muK = muK; a.muQ = p->smooth_q ? muQ : nullptr;
    a.ksplits = splits;
    // every partial sum the quantiser reads is written by the K-mean pass of the same call, so the
    // array needs no clearing; calls that overlap on the GPU share it and race
    a.kpartial = p->smooth_k ? scratch : nullptr;
    a.N = p->N; a.d = p->d; a.smooth_k = p->smooth_k; a.smooth_q = p->smooth_q;
    a.fp8 = (p->flags & SAGE_FLAG_FP8) != 0;
    if (launch_quantize(*p, a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return SAGE_ERR_CUDA;
    return SAGE_OK;
}
