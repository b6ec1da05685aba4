// fwd_gemm_k64.cu -- the forward GEMM with 64-deep k-blocks, used when K is
// a multiple of 64 but not of 128 (kernel: fwd_gemm_impl.cuh).
#undef AGOQ_FWD_BK
#undef AGOQ_FWD_STAGES
#define AGOQ_FWD_BK 64
#define AGOQ_FWD_STAGES 6
#define AGOQ_FWD_INSTANCE fwd64
#include "fwd_gemm_impl.cuh"
