// wgrad_gemm.cu -- INT4-dequant-fused weight-gradient GEMM (placeholder launcher).
#include "agoq_device.cuh"
#include "agoq_launch.h"

namespace agoq {

// Device-side status word: a GEMM pipeline wait that exceeds its iteration
// limit records a non-zero code here instead of spinning forever.
__device__ unsigned g_device_status;

cudaError_t launch_wgrad_gemm(const void *, const void *, const float *, int, int, int, void *, bool,
                              cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t read_and_clear_device_status(cudaStream_t st, unsigned *status) {
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
        if (e != cudaSuccess) return e;
    }
    *status = v;
    return cudaSuccess;
}

}  // namespace agoq
