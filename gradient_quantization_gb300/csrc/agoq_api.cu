// agoq_api.cu -- the extern "C" entry points declared in include/agoq.h.
//
// Each entry point validates its arguments on the host (null pointers, sizes,
// widths, alignment, overlap of outputs with inputs) before launching
// anything, then launches on the caller's stream and maps a launch failure to
// AGOQ_ERR_CUDA.  No entry point allocates or synchronises (except
// agoq_device_status, whose purpose is to synchronise).
#include "../../include/agoq.h"
#include "agoq_launch.h"

#include <cstdint>

namespace agoq {

int sm_count() {
    static int cache[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    if (cache[dev] == 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = sms > 0 ? sms : 1;
    }
    return cache[dev];
}

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Half-open byte ranges [a, a+na) and [b, b+nb) overlap.
bool overlap(const void *a, uint64_t na, const void *b, uint64_t nb) {
    if (na == 0 || nb == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

bool bits_ok(int bits) { return bits == 4 || bits == 5 || bits == 6 || bits == 8; }

agoq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? AGOQ_OK : AGOQ_ERR_CUDA; }

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

}  // namespace
}  // namespace agoq

extern "C" {

const char *agoq_status_string(agoq_status s) {
    switch (s) {
        case AGOQ_OK: return "AGOQ_OK";
        case AGOQ_ERR_NULL: return "AGOQ_ERR_NULL: a required pointer is NULL";
        case AGOQ_ERR_SHAPE: return "AGOQ_ERR_SHAPE: size not supported (n % 128, GEMM tiles)";
        case AGOQ_ERR_BITS: return "AGOQ_ERR_BITS: bits must be 4, 5, 6 or 8";
        case AGOQ_ERR_ALIGN: return "AGOQ_ERR_ALIGN: pointer not aligned as required";
        case AGOQ_ERR_ALIAS: return "AGOQ_ERR_ALIAS: an output overlaps an input";
        case AGOQ_ERR_CUDA: return "AGOQ_ERR_CUDA: CUDA runtime error";
        case AGOQ_ERR_TIMEOUT: return "AGOQ_ERR_TIMEOUT: a pipeline wait gave up";
        case AGOQ_ERR_FORMAT: return "AGOQ_ERR_FORMAT: unsupported intermediate format";
    }
    return "AGOQ_ERR_UNKNOWN";
}

int agoq_version(void) { return 100; }

agoq_status agoq_quant_act(const void *x_bf16, int64_t n, int bits, void *codes, float *scales,
                           void *stream) {
    using namespace agoq;
    if (!bits_ok(bits)) return AGOQ_ERR_BITS;
    if (n < 0 || n % kBlockElems) return AGOQ_ERR_SHAPE;
    if (n == 0) return AGOQ_OK;
    if (!x_bf16 || !codes || !scales) return AGOQ_ERR_NULL;
    if (!aligned(x_bf16, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return AGOQ_ERR_ALIGN;
    const uint64_t nb = (uint64_t)n / kBlockElems;
    const uint64_t xb = 2ull * n, cb = nb * 16 * bits, sb = nb * 4;
    if (overlap(codes, cb, x_bf16, xb) || overlap(scales, sb, x_bf16, xb) ||
        overlap(codes, cb, scales, sb))
        return AGOQ_ERR_ALIAS;
    return from_cuda(launch_laaq_quant(x_bf16, n, bits, codes, scales, as_stream(stream)));
}

agoq_status agoq_dequant_act(const void *codes, const float *scales, int64_t n, int bits,
                             void *y_bf16, void *stream) {
    using namespace agoq;
    if (!bits_ok(bits)) return AGOQ_ERR_BITS;
    if (n < 0 || n % kBlockElems) return AGOQ_ERR_SHAPE;
    if (n == 0) return AGOQ_OK;
    if (!codes || !scales || !y_bf16) return AGOQ_ERR_NULL;
    if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(y_bf16, 16)) return AGOQ_ERR_ALIGN;
    const uint64_t nb = (uint64_t)n / kBlockElems;
    const uint64_t yb = 2ull * n, cb = nb * 16 * bits, sb = nb * 4;
    if (overlap(y_bf16, yb, codes, cb) || overlap(y_bf16, yb, scales, sb)) return AGOQ_ERR_ALIAS;
    return from_cuda(launch_laaq_dequant(codes, scales, n, bits, y_bf16, as_stream(stream)));
}

agoq_status agoq_silu_backward(const void *codes, const float *scales, const void *dy_bf16,
                               int64_t n, int bits, void *dx_bf16, void *y_bf16, void *stream) {
    using namespace agoq;
    if (!bits_ok(bits)) return AGOQ_ERR_BITS;
    if (n < 0 || n % kBlockElems) return AGOQ_ERR_SHAPE;
    if (n == 0) return AGOQ_OK;
    if (!codes || !scales || !dy_bf16 || !dx_bf16) return AGOQ_ERR_NULL;
    if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(dy_bf16, 16) ||
        !aligned(dx_bf16, 16) || (y_bf16 && !aligned(y_bf16, 16)))
        return AGOQ_ERR_ALIGN;
    const uint64_t nb = (uint64_t)n / kBlockElems;
    const uint64_t cb = nb * 16 * bits, sb = nb * 4, vb = 2ull * n, yb = y_bf16 ? vb : 0;
    if (overlap(dx_bf16, vb, codes, cb) || overlap(dx_bf16, vb, scales, sb) ||
        overlap(dx_bf16, vb, dy_bf16, vb) || overlap(y_bf16, yb, codes, cb) ||
        overlap(y_bf16, yb, scales, sb) || overlap(y_bf16, yb, dy_bf16, vb) ||
        overlap(y_bf16, yb, dx_bf16, vb))
        return AGOQ_ERR_ALIAS;
    return from_cuda(
        launch_silu_backward(codes, scales, dy_bf16, n, bits, dx_bf16, y_bf16, as_stream(stream)));
}

agoq_status agoq_rmsnorm_backward(const void *codes, const float *scales, const void *dy_bf16,
                                  const void *w_bf16, int64_t T, int64_t H, int bits, float eps,
                                  void *dx_bf16, float *rstd, float *dw, void *stream) {
    using namespace agoq;
    if (!bits_ok(bits)) return AGOQ_ERR_BITS;
    if (T < 0 || H <= 0 || H % 256 || H > 8192 || !(eps >= 0.0f) || eps > 3.0e38f)
        return AGOQ_ERR_SHAPE;
    if (T == 0 && !dw) return AGOQ_OK;
    if (!codes || !scales || !dy_bf16 || !w_bf16 || !dx_bf16 || !rstd) return AGOQ_ERR_NULL;
    if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(dy_bf16, 16) ||
        !aligned(w_bf16, 16) || !aligned(dx_bf16, 16) || !aligned(rstd, 4) ||
        (dw && !aligned(dw, 4)))
        return AGOQ_ERR_ALIGN;
    const uint64_t n = (uint64_t)T * H, nb = n / kBlockElems;
    const uint64_t cb = nb * 16 * bits, sb = nb * 4, vb = 2 * n, wb = 2ull * H;
    const uint64_t rb = 4ull * T, db = dw ? 4ull * H : 0;
    const void *in[4] = {codes, scales, dy_bf16, w_bf16};
    const uint64_t inb[4] = {cb, sb, vb, wb};
    for (int i = 0; i < 4; ++i)
        if (overlap(dx_bf16, vb, in[i], inb[i]) || overlap(rstd, rb, in[i], inb[i]) ||
            overlap(dw, db, in[i], inb[i]))
            return AGOQ_ERR_ALIAS;
    if (overlap(dx_bf16, vb, rstd, rb) || overlap(dx_bf16, vb, dw, db) || overlap(rstd, rb, dw, db))
        return AGOQ_ERR_ALIAS;
    if (T == 0) return from_cuda(cudaMemsetAsync(dw, 0, 4ull * H, as_stream(stream)));
    return from_cuda(launch_rmsnorm_backward(codes, scales, dy_bf16, w_bf16, T, H, bits, eps,
                                             dx_bf16, rstd, dw, as_stream(stream)));
}

int64_t agoq_rmsnorm_backward_workspace_bytes(int64_t H) {
    using namespace agoq;
    if (H <= 0 || H % 256 || H > 8192) return -1;
    return H <= rmsnorm_fused_max_h() ? (int64_t)rmsnorm_fused_partials() * H * 4 : 0;
}

agoq_status agoq_rmsnorm_backward_ws(const void *codes, const float *scales, const void *dy_bf16,
                                     const void *w_bf16, int64_t T, int64_t H, int bits, float eps,
                                     void *dx_bf16, float *rstd, float *dw, void *workspace,
                                     int64_t workspace_bytes, void *stream) {
    using namespace agoq;
    if (!bits_ok(bits)) return AGOQ_ERR_BITS;
    if (T < 0 || H <= 0 || H % 256 || H > 8192 || !(eps >= 0.0f) || eps > 3.0e38f)
        return AGOQ_ERR_SHAPE;
    const int64_t need = agoq_rmsnorm_backward_workspace_bytes(H);
    if (workspace_bytes < need) return AGOQ_ERR_SHAPE;
    if (!dw || (need > 0 && !workspace)) return AGOQ_ERR_NULL;
    if (need == 0 || T == 0)
        return agoq_rmsnorm_backward(codes, scales, dy_bf16, w_bf16, T, H, bits, eps, dx_bf16,
                                     rstd, dw, stream);
    if (!codes || !scales || !dy_bf16 || !w_bf16 || !dx_bf16 || !rstd) return AGOQ_ERR_NULL;
    if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(dy_bf16, 16) ||
        !aligned(w_bf16, 16) || !aligned(dx_bf16, 16) || !aligned(rstd, 4) || !aligned(dw, 4) ||
        !aligned(workspace, 16))
        return AGOQ_ERR_ALIGN;
    const uint64_t n = (uint64_t)T * H, nb = n / kBlockElems;
    const uint64_t cb = nb * 16 * bits, sb = nb * 4, vb = 2 * n, wb = 2ull * H;
    const uint64_t rb = 4ull * T, db = 4ull * H, kb = (uint64_t)need;
    const void *in[4] = {codes, scales, dy_bf16, w_bf16};
    const uint64_t inb[4] = {cb, sb, vb, wb};
    for (int i = 0; i < 4; ++i)
        if (overlap(dx_bf16, vb, in[i], inb[i]) || overlap(rstd, rb, in[i], inb[i]) ||
            overlap(dw, db, in[i], inb[i]) || overlap(workspace, kb, in[i], inb[i]))
            return AGOQ_ERR_ALIAS;
    if (overlap(dx_bf16, vb, rstd, rb) || overlap(dx_bf16, vb, dw, db) || overlap(rstd, rb, dw, db) ||
        overlap(workspace, kb, dx_bf16, vb) || overlap(workspace, kb, rstd, rb) ||
        overlap(workspace, kb, dw, db))
        return AGOQ_ERR_ALIAS;
    return from_cuda(launch_rmsnorm_backward_fused(codes, scales, dy_bf16, w_bf16, T, H, bits, eps,
                                                   dx_bf16, rstd, dw,
                                                   static_cast<float *>(workspace),
                                                   as_stream(stream)));
}

agoq_status agoq_rmsnorm_backward_noalloc(const void *codes, const float *scales,
                                          const void *dy_bf16, const void *w_bf16, int64_t T,
                                          int64_t H, int bits, float eps, void *dx_bf16,
                                          float *rstd, float *dw, void *stream) {
    using namespace agoq;
    if (!bits_ok(bits)) return AGOQ_ERR_BITS;
    if (T < 0 || H <= 0 || H % 256 || H > rmsnorm_fused_max_h() || !(eps >= 0.0f) ||
        eps > 3.0e38f)
        return AGOQ_ERR_SHAPE;
    if (!dw) return AGOQ_ERR_NULL;
    if (T == 0) {
        if (!aligned(dw, 4)) return AGOQ_ERR_ALIGN;
        return from_cuda(cudaMemsetAsync(dw, 0, 4ull * H, as_stream(stream)));
    }
    if (!codes || !scales || !dy_bf16 || !w_bf16 || !dx_bf16 || !rstd) return AGOQ_ERR_NULL;
    if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(dy_bf16, 16) ||
        !aligned(w_bf16, 16) || !aligned(dx_bf16, 16) || !aligned(rstd, 4) || !aligned(dw, 4))
        return AGOQ_ERR_ALIGN;
    const uint64_t n = (uint64_t)T * H, nb = n / kBlockElems;
    const uint64_t cb = nb * 16 * bits, sb = nb * 4, vb = 2 * n, wb = 2ull * H;
    const uint64_t rb = 4ull * T, db = 4ull * H;
    const void *in[4] = {codes, scales, dy_bf16, w_bf16};
    const uint64_t inb[4] = {cb, sb, vb, wb};
    for (int i = 0; i < 4; ++i)
        if (overlap(dx_bf16, vb, in[i], inb[i]) || overlap(rstd, rb, in[i], inb[i]) ||
            overlap(dw, db, in[i], inb[i]))
            return AGOQ_ERR_ALIAS;
    if (overlap(dx_bf16, vb, rstd, rb) || overlap(dx_bf16, vb, dw, db) || overlap(rstd, rb, dw, db))
        return AGOQ_ERR_ALIAS;
    return from_cuda(launch_rmsnorm_backward_noalloc(codes, scales, dy_bf16, w_bf16, T, H, bits,
                                                     eps, dx_bf16, rstd, dw, as_stream(stream)));
}

agoq_status agoq_grad_accum_fp8(void *master_e4m3, float *master_scales, const void *grad_bf16,
                                int64_t n, void *stream) {
    return agoq_grad_accum_fp8_mid(master_e4m3, master_scales, grad_bf16, n, AGOQ_MID_FP32, stream);
}

agoq_status agoq_grad_accum_fp8_mid(void *master_e4m3, float *master_scales,
                                    const void *grad_bf16, int64_t n, int mid_format,
                                    void *stream) {
    using namespace agoq;
    if (mid_format != AGOQ_MID_FP32 && mid_format != AGOQ_MID_BF16 && mid_format != AGOQ_MID_FP16)
        return AGOQ_ERR_FORMAT;
    if (n < 0 || n % kBlockElems) return AGOQ_ERR_SHAPE;
    if (n == 0) return AGOQ_OK;
    if (!master_e4m3 || !master_scales || !grad_bf16) return AGOQ_ERR_NULL;
    if (!aligned(master_e4m3, 16) || !aligned(master_scales, 4) || !aligned(grad_bf16, 16))
        return AGOQ_ERR_ALIGN;
    const uint64_t nb = (uint64_t)n / kBlockElems;
    const uint64_t mb = (uint64_t)n, sb = nb * 4, gb = 2ull * n;
    if (overlap(master_e4m3, mb, grad_bf16, gb) || overlap(master_scales, sb, grad_bf16, gb) ||
        overlap(master_e4m3, mb, master_scales, sb))
        return AGOQ_ERR_ALIAS;
    return from_cuda(
        launch_grad_accum(master_e4m3, master_scales, grad_bf16, n, mid_format, as_stream(stream)));
}

agoq_status agoq_reduce_fp8_shards(const void *shards_e4m3, const float *shard_scales, int W,
                                   int64_t n, void *out_e4m3, float *out_scales,
                                   unsigned long long *naive_overflow_count, void *stream) {
    using namespace agoq;
    if (W < 1 || n < 0 || n % kBlockElems) return AGOQ_ERR_SHAPE;
    if (n == 0) {
        if (naive_overflow_count)
            return from_cuda(cudaMemsetAsync(naive_overflow_count, 0, sizeof(unsigned long long),
                                             as_stream(stream)));
        return AGOQ_OK;
    }
    if (!shards_e4m3 || !shard_scales || !out_e4m3 || !out_scales) return AGOQ_ERR_NULL;
    if (!aligned(shards_e4m3, 16) || !aligned(shard_scales, 4) || !aligned(out_e4m3, 16) ||
        !aligned(out_scales, 4) || (naive_overflow_count && !aligned(naive_overflow_count, 8)))
        return AGOQ_ERR_ALIGN;
    const uint64_t nb = (uint64_t)n / kBlockElems;
    const uint64_t shb = (uint64_t)W * n, ssb = (uint64_t)W * nb * 4, ob = (uint64_t)n, osb = nb * 4;
    const uint64_t cntb = naive_overflow_count ? 8 : 0;
    if (overlap(out_e4m3, ob, shards_e4m3, shb) || overlap(out_e4m3, ob, shard_scales, ssb) ||
        overlap(out_scales, osb, shards_e4m3, shb) || overlap(out_scales, osb, shard_scales, ssb) ||
        overlap(out_e4m3, ob, out_scales, osb) ||
        overlap(naive_overflow_count, cntb, shards_e4m3, shb) ||
        overlap(naive_overflow_count, cntb, shard_scales, ssb) ||
        overlap(naive_overflow_count, cntb, out_e4m3, ob) ||
        overlap(naive_overflow_count, cntb, out_scales, osb))
        return AGOQ_ERR_ALIAS;
    return from_cuda(launch_reduce_shards(shards_e4m3, shard_scales, W, n, out_e4m3, out_scales,
                                          naive_overflow_count, as_stream(stream)));
}

static agoq_status wgrad_common(const void *dY, const void *xc, const float *xs, int M, int N,
                                int K, void *dW, bool f32_out, void *stream) {
    using namespace agoq;
    if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 64) return AGOQ_ERR_SHAPE;
    if (!dY || !xc || !xs || !dW) return AGOQ_ERR_NULL;
    if (!aligned(dY, 16) || !aligned(xc, 16) || !aligned(xs, 4) || !aligned(dW, 16))
        return AGOQ_ERR_ALIGN;
    const uint64_t dyb = 2ull * K * M, xcb = (uint64_t)K * N / 2, xsb = (uint64_t)K * (N / 128) * 4;
    const uint64_t dwb = (uint64_t)M * N * (f32_out ? 4 : 2);
    if (overlap(dW, dwb, dY, dyb) || overlap(dW, dwb, xc, xcb) || overlap(dW, dwb, xs, xsb))
        return AGOQ_ERR_ALIAS;
    return from_cuda(launch_wgrad_gemm(dY, xc, xs, M, N, K, dW, f32_out, as_stream(stream)));
}

agoq_status agoq_wgrad_gemm_int4(const void *dY_bf16, const void *x_codes, const float *x_scales,
                                 int M, int N, int K, void *dW_bf16, void *stream) {
    return wgrad_common(dY_bf16, x_codes, x_scales, M, N, K, dW_bf16, false, stream);
}

agoq_status agoq_wgrad_gemm_int4_f32out(const void *dY_bf16, const void *x_codes,
                                        const float *x_scales, int M, int N, int K, float *dW_f32,
                                        void *stream) {
    return wgrad_common(dY_bf16, x_codes, x_scales, M, N, K, dW_f32, true, stream);
}

agoq_status agoq_wgrad_gemm_int4_accum_fp8(const void *dY_bf16, const void *x_codes,
                                           const float *x_scales, int M, int N, int K,
                                           void *master_e4m3, float *master_scales,
                                           void *stream) {
    using namespace agoq;
    if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 64) return AGOQ_ERR_SHAPE;
    if (!dY_bf16 || !x_codes || !x_scales || !master_e4m3 || !master_scales) return AGOQ_ERR_NULL;
    if (!aligned(dY_bf16, 16) || !aligned(x_codes, 16) || !aligned(x_scales, 4) ||
        !aligned(master_e4m3, 16) || !aligned(master_scales, 4))
        return AGOQ_ERR_ALIGN;
    const uint64_t dyb = 2ull * K * M, xcb = (uint64_t)K * N / 2, xsb = (uint64_t)K * (N / 128) * 4;
    const uint64_t mb = (uint64_t)M * N, msb = (uint64_t)M * (N / 128) * 4;
    if (overlap(master_e4m3, mb, dY_bf16, dyb) || overlap(master_e4m3, mb, x_codes, xcb) ||
        overlap(master_e4m3, mb, x_scales, xsb) || overlap(master_scales, msb, dY_bf16, dyb) ||
        overlap(master_scales, msb, x_codes, xcb) || overlap(master_scales, msb, x_scales, xsb) ||
        overlap(master_e4m3, mb, master_scales, msb))
        return AGOQ_ERR_ALIAS;
    return from_cuda(launch_wgrad_accum_fp8(dY_bf16, x_codes, x_scales, M, N, K, master_e4m3,
                                            master_scales, as_stream(stream)));
}

agoq_status agoq_dbca_pp_bits(int stages, int microbatches, int base_bits, int *bits) {
    if (stages < 1 || microbatches < 1) return AGOQ_ERR_SHAPE;
    if (base_bits != 4 && base_bits != 5 && base_bits != 6 && base_bits != 8) return AGOQ_ERR_BITS;
    if (!bits) return AGOQ_ERR_NULL;
    static const int kWidths[4] = {4, 5, 6, 8};
    const long long first = stages < microbatches ? stages : microbatches;   // stage 0's batches
    const long long cap = first * base_bits;
    for (int s = 0; s < stages; ++s) {
        const long long live = (stages - s) < microbatches ? (stages - s) : microbatches;
        int b = base_bits;
        for (int i = 0; i < 4; ++i)
            if (kWidths[i] >= base_bits && live * kWidths[i] <= cap) b = kWidths[i];
        bits[s] = b;
    }
    return AGOQ_OK;
}

agoq_status agoq_fwd_gemm_quant(const void *x_bf16, const void *w_bf16, int T, int N, int K,
                                int bits, void *y_bf16, void *codes, float *scales, void *stream) {
    using namespace agoq;
    if (!bits_ok(bits)) return AGOQ_ERR_BITS;
    if (T <= 0 || N <= 0 || K <= 0 || T % 128 || N % 256 || K % 64) return AGOQ_ERR_SHAPE;
    if (!x_bf16 || !w_bf16 || !y_bf16 || !codes || !scales) return AGOQ_ERR_NULL;
    if (!aligned(x_bf16, 16) || !aligned(w_bf16, 16) || !aligned(y_bf16, 16) ||
        !aligned(codes, 16) || !aligned(scales, 4))
        return AGOQ_ERR_ALIGN;
    const uint64_t n = (uint64_t)T * N, nb = n / kBlockElems;
    const uint64_t xb = 2ull * T * K, wb = 2ull * N * K, yb = 2 * n, cb = nb * 16 * bits,
                   sb = nb * 4;
    const void *in[2] = {x_bf16, w_bf16};
    const uint64_t inb[2] = {xb, wb};
    for (int i = 0; i < 2; ++i)
        if (overlap(y_bf16, yb, in[i], inb[i]) || overlap(codes, cb, in[i], inb[i]) ||
            overlap(scales, sb, in[i], inb[i]))
            return AGOQ_ERR_ALIAS;
    if (overlap(y_bf16, yb, codes, cb) || overlap(y_bf16, yb, scales, sb) ||
        overlap(codes, cb, scales, sb))
        return AGOQ_ERR_ALIAS;
    return from_cuda(launch_fwd_gemm_quant(x_bf16, w_bf16, T, N, K, bits, y_bf16, codes, scales,
                                           as_stream(stream)));
}

agoq_status agoq_test_wait_timeout(int64_t limit_cycles, void *stream) {
    if (limit_cycles <= 0 || limit_cycles > 4000000000ll) return AGOQ_ERR_SHAPE;
    return agoq::from_cuda(agoq::launch_wait_timeout_probe(limit_cycles, agoq::as_stream(stream)));
}

agoq_status agoq_device_status(void *stream) {
    unsigned status = 0, fwd = 0, red = 0, rms = 0;
    if (agoq::read_and_clear_device_status(agoq::as_stream(stream), &status) != cudaSuccess ||
        agoq::read_and_clear_fwd_status(&fwd) != cudaSuccess ||
        agoq::read_and_clear_reduce_status(&red) != cudaSuccess ||
        agoq::read_and_clear_rmsnorm_status(&rms) != cudaSuccess)
        return AGOQ_ERR_CUDA;
    return (status || fwd || red || rms) ? AGOQ_ERR_TIMEOUT : AGOQ_OK;
}

}  // extern "C"
