// sage_bwd.cu -- SageBwd backward (placeholder until the tcgen05 kernel lands).
#include "sage_device.cuh"
#include "sage_internal.h"

namespace sage {

__device__ unsigned int g_bwd_err;

cudaError_t launch_bwd(const sage_params &, const __half *, const __half *, const void *,
                       const void *, const __half *, BwdArgs, cudaStream_t) {
    return cudaErrorNotSupported;
}

unsigned int take_bwd_error() {
    unsigned int v = 0, zero = 0;
    cudaMemcpyFromSymbol(&v, g_bwd_err, sizeof(v));
    cudaMemcpyToSymbol(g_bwd_err, &zero, sizeof(zero));
    return v;
}

}  // namespace sage
