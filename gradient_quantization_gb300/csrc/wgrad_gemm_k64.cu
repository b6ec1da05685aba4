// wgrad_gemm_k64.cu -- the weight-gradient GEMM with 64-deep k-blocks, used
// when K is a multiple of 64 but not of 128 (kernel: wgrad_gemm_impl.cuh).
#undef AGOQ_GEMM_BK
#undef AGOQ_GEMM_NA
#undef AGOQ_GEMM_NB
#undef AGOQ_GEMM_NX
#define AGOQ_GEMM_BK 64
#define AGOQ_GEMM_NA 3
#define AGOQ_GEMM_NB 3
#define AGOQ_GEMM_NX 3
#define AGOQ_WGRAD_NS wg64
#include "wgrad_gemm_impl.cuh"
