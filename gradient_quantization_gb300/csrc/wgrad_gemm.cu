// wgrad_gemm.cu -- the weight-gradient GEMM with 128-deep k-blocks (K a
// multiple of 128), and the entry points that pick an instance by K (the
// kernel itself is in wgrad_gemm_impl.cuh).
// Ring depths (k-blocks): A 2, B 2, X 3 -- what the shared memory holds at
// this depth.
#define AGOQ_GEMM_BK 128
#define AGOQ_GEMM_NA 2
#define AGOQ_GEMM_NB 2
#define AGOQ_GEMM_NX 3
#define AGOQ_WGRAD_NS wg128
#include "wgrad_gemm_impl.cuh"

namespace agoq {

// The 64-deep instance (wgrad_gemm_k64.cu).
namespace wg64 {
cudaError_t launch_gemm(const void *dY, const void *xc, const float *xs, int M, int N, int K,
                        void *dW, bool f32_out, cudaStream_t st);
cudaError_t launch_accum_fp8(const void *dY, const void *xc, const float *xs, int M, int N, int K,
                             void *master, float *master_scales, cudaStream_t st);
cudaError_t read_and_clear_status(unsigned *status);
}  // namespace wg64

cudaError_t launch_wgrad_gemm(const void *dY, const void *xc, const float *xs, int M, int N, int K,
                              void *dW, bool f32_out, cudaStream_t st) {
    return K % AGOQ_GEMM_BK == 0 ? wg128::launch_gemm(dY, xc, xs, M, N, K, dW, f32_out, st)
                                 : wg64::launch_gemm(dY, xc, xs, M, N, K, dW, f32_out, st);
}

cudaError_t launch_wgrad_accum_fp8(const void *dY, const void *xc, const float *xs, int M, int N,
                                   int K, void *master, float *master_scales, cudaStream_t st) {
    return K % AGOQ_GEMM_BK == 0
               ? wg128::launch_accum_fp8(dY, xc, xs, M, N, K, master, master_scales, st)
               : wg64::launch_accum_fp8(dY, xc, xs, M, N, K, master, master_scales, st);
}

cudaError_t launch_wait_timeout_probe(long long limit_cycles, cudaStream_t st) {
    return wg128::launch_wait_timeout_probe(limit_cycles, st);
}

cudaError_t read_and_clear_device_status(cudaStream_t st, unsigned *status) {
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    unsigned a = 0, b = 0;
    e = wg128::read_and_clear_status(&a);
    if (e != cudaSuccess) return e;
    e = wg64::read_and_clear_status(&b);
    if (e != cudaSuccess) return e;
    *status = a ? a : b;
    return cudaSuccess;
}

}  // namespace agoq
