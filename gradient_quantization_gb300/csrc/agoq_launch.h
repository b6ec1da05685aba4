// agoq_launch.h -- internal launchers behind the C ABI (not installed).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace agoq {

constexpr int kMaxDevices = 64;
constexpr int64_t kBlockElems = 128;   // elements per quantization block

// Multiprocessor count of the current device (cached per device).
int sm_count();

// Resident CTAs per SM for `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory; cached in `cache` (one slot per device, 0 = unknown).
template <typename K>
int resident_per_sm(K kernel, int threads, size_t smem, int *cache) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    if (cache[dev] == 0) {
        int per_sm = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
        cache[dev] = per_sm > 0 ? per_sm : 1;
    }
    return cache[dev];
}

// Launch `kernel` with programmatic stream serialization: it may be scheduled
// while the previous kernel on the stream is finishing.  Every kernel launched
// this way begins with pdl_wait_and_release() (griddepcontrol.wait) before
// touching global memory, so it still observes all effects of the work before
// it in the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem,
                       cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_laaq_quant(const void *x, int64_t n, int bits, void *codes, float *scales,
                              cudaStream_t st);
cudaError_t launch_laaq_dequant(const void *codes, const float *scales, int64_t n, int bits,
                                void *y, cudaStream_t st);
cudaError_t launch_silu_backward(const void *codes, const float *scales, const void *dy, int64_t n,
                                 int bits, void *dx, void *y, cudaStream_t st);
// RMSNorm backward from LAAQ codes of x [T][H]; dw may be NULL (then not computed).
cudaError_t launch_rmsnorm_backward(const void *codes, const float *scales, const void *dy,
                                    const void *w, int64_t T, int64_t H, int bits, float eps,
                                    void *dx, float *rstd, float *dw, cudaStream_t st);
// The same in one read of the input (H <= rmsnorm_fused_max_h()): dx, rstd and
// per-CTA dw partial sums in `partials` (rmsnorm_fused_partials() x H floats),
// then dw from them in a fixed order.
cudaError_t launch_rmsnorm_backward_fused(const void *codes, const float *scales, const void *dy,
                                          const void *w, int64_t T, int64_t H, int bits, float eps,
                                          void *dx, float *rstd, float *dw, float *partials,
                                          cudaStream_t st);
int rmsnorm_fused_partials();
int rmsnorm_fused_max_h();
// The single-read form with the library's own static scratch (H <= rmsnorm_fused_max_h()).
cudaError_t launch_rmsnorm_backward_noalloc(const void *codes, const float *scales, const void *dy,
                                            const void *w, int64_t T, int64_t H, int bits,
                                            float eps, void *dx, float *rstd, float *dw,
                                            cudaStream_t st);
// mid: intermediate format of the sum (0 binary32, 1 BF16, 2 FP16).
cudaError_t launch_grad_accum(void *master, float *master_scales, const void *grad, int64_t n,
                              int mid, cudaStream_t st);
cudaError_t launch_reduce_shards(const void *shards, const float *shard_scales, int W, int64_t n,
                                 void *out, float *out_scales, unsigned long long *naive_count,
                                 cudaStream_t st);
cudaError_t launch_wgrad_gemm(const void *dY, const void *xc, const float *xs, int M, int N, int K,
                              void *dW, bool f32_out, cudaStream_t st);
cudaError_t launch_wgrad_accum_fp8(const void *dY, const void *xc, const float *xs, int M, int N,
                                   int K, void *master, float *master_scales, cudaStream_t st);
cudaError_t launch_fwd_gemm_quant(const void *x, const void *w, int T, int N, int K, int bits,
                                  void *y, void *codes, float *scales, cudaStream_t st);
// A kernel whose one pipeline wait runs out after `limit_cycles` (failure-path test).
cudaError_t launch_wait_timeout_probe(long long limit_cycles, cudaStream_t st);
// Read and clear the forward GEMM's status word (call after synchronising).
cudaError_t read_and_clear_fwd_status(unsigned *status);
// The same for the staged FP8 shard reduce.
cudaError_t read_and_clear_reduce_status(unsigned *status);
// The same for the TMA-staged RMSNorm weight-gradient kernel.
cudaError_t read_and_clear_rmsnorm_status(unsigned *status);
// Synchronise `st`, read and clear the device status word (0 = no timeout).
cudaError_t read_and_clear_device_status(cudaStream_t st, unsigned *status);

}  // namespace agoq
