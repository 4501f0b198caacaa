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

// Device address of the array on each device.  The host-side name of the array is not a device
// address and must never be handed to a kernel, so the address is looked up with
// cudaGetSymbolAddress, once per device with that device current, and kept.  A failed lookup is
// not kept: the next call on that device tries again.
static constexpr int kMaxDevices = 64;
static double *g_noalloc_ptr[kMaxDevices];
static std::mutex g_noalloc_mutex;

static double *noalloc_scratch(int device) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[device]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_kpartial) == cudaSuccess)
            g_noalloc_ptr[device] = static_cast<double *>(ptr);
        else
            (void)cudaGetLastError();    // clear the error so that the next call starts clean
    }
    return g_noalloc_ptr[device];
}

// Partial sums a call with these parameters keeps in the array (0 without K-smoothing).
static size_t partials_needed(const sage_params &p) {
    if (!p.smooth_k) return 0;
    return quant_fused_doubles(p);
}

}  // namespace sage

using namespace sage;

extern "C" size_t sage_quantize_noalloc_max_partials(void) { return kNoallocPartials; }

extern "C" size_t sage_quantize_noalloc_partials_needed(const sage_params *p) {
    if (check_params(p) != SAGE_OK) return 0;
    return partials_needed(*p);
}

extern "C" int sage_quantize_smooth_noalloc(const sage_params *p, const void *Q, const void *K,
                                            const void *V, int8_t *Qh, int8_t *Kh, int8_t *Vh,
                                            float *sQ, float *sK, float *sV, float *muK,
                                            float *muQ, sage_stream_t stream) {
    // the rules of sage_quantize_smooth, less its workspace; no debug dump, no INT8-dP flag
    const int st = check_params(p);
    if (st != SAGE_OK) return st;
    if (p->flags & ~(SAGE_FLAG_FP8 | SAGE_FLAG_OPS16)) return SAGE_ERR_ARG;
    const void *ptrs[] = {Q, K, V, Qh, Kh, Vh, sQ, sK, sV, muK};
    for (const void *q : ptrs) {
        if (!q) return SAGE_ERR_ARG;
        if (reinterpret_cast<uintptr_t>(q) & 15u) return SAGE_ERR_ALIGN;
    }
    if (p->smooth_q) {
        if (!muQ) return SAGE_ERR_ARG;
        if (reinterpret_cast<uintptr_t>(muQ) & 15u) return SAGE_ERR_ALIGN;
    }
    if (partials_needed(*p) > kNoallocPartials) return SAGE_ERR_WORKSPACE;   // beyond the array

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) return SAGE_ERR_CUDA;
    double *scratch = noalloc_scratch(device);
    if (!scratch) return SAGE_ERR_CUDA;

    QuantArgs a{};
    a.Q = Q; a.K = K; a.V = V;
    a.Qh = Qh; a.Kh = Kh; a.Vh = Vh;
    a.sQ = sQ; a.sK = sK; a.sV = sV;
    a.muK = muK; a.muQ = p->smooth_q ? muQ : nullptr;
    a.ksplits = kmean_splits(*p);
    // every partial sum the quantiser reads is written by the K-mean phase of the same call, and
    // the two barrier words at the end are cleared on the stream before the launch, so the array
    // needs no other clearing; calls that overlap on the GPU share it and race
    a.kpartial = p->smooth_k ? scratch : nullptr;
    a.N = p->N; a.d = p->d; a.smooth_k = p->smooth_k; a.smooth_q = p->smooth_q;
    a.fp8 = (p->flags & SAGE_FLAG_FP8) != 0;
    a.ops16 = (p->flags & SAGE_FLAG_OPS16) ? static_cast<__half *>(p->ops16) : nullptr;
    if (launch_quantize(*p, a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return SAGE_ERR_CUDA;
    return SAGE_OK;
}
