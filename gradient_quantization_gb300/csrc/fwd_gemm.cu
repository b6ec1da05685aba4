// fwd_gemm.cu -- the forward GEMM with fused LAAQ quantization, 128-deep
// k-blocks (K a multiple of 128), and the entry points that pick an instance
// by K (the kernel itself is in fwd_gemm_impl.cuh).
#define AGOQ_FWD_BK 128
#define AGOQ_FWD_STAGES 3
#define AGOQ_FWD_INSTANCE fwd128
#include "fwd_gemm_impl.cuh"

namespace agoq {

// The 64-deep instance (fwd_gemm_k64.cu).
namespace fwd64 {
cudaError_t launch(const void *x, const void *w, int T, int N, int K, int bits, void *y,
                   void *codes, float *scales, cudaStream_t st);
cudaError_t read_and_clear_status(unsigned *status);
}  // namespace fwd64

cudaError_t launch_fwd_gemm_quant(const void *x, const void *w, int T, int N, int K, int bits,
                                  void *y, void *codes, float *scales, cudaStream_t st) {
    return K % AGOQ_FWD_BK == 0 ? fwd128::launch(x, w, T, N, K, bits, y, codes, scales, st)
                                : fwd64::launch(x, w, T, N, K, bits, y, codes, scales, st);
}

cudaError_t read_and_clear_fwd_status(unsigned *status) {
    unsigned a = 0, b = 0;
    cudaError_t e = fwd128::read_and_clear_status(&a);
    if (e != cudaSuccess) return e;
    e = fwd64::read_and_clear_status(&b);
    if (e != cudaSuccess) return e;
    *status = a ? a : b;
    return cudaSuccess;
}

}  // namespace agoq
