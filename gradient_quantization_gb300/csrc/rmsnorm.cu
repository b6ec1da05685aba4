// rmsnorm.cu -- RMSNorm backward recomputed from the stored low-bit input
// ("AGoQ: Activation and Gradient Quantization for Memory-Efficient
// Distributed Training of LLMs", section 2.A "Herberekening versus Caching":
// only the quantized RMSNorm input is kept; the backward pass dequantizes it
// and recomputes the row statistics).
//
// Forward: y[t][i] = x[t][i] * r_t * w[i], r_t = 1 / sqrt(mean_i x[t][i]^2 + eps).
// Backward, with xh the LAAQ dequantization of the stored codes and
// g[i] = dy[t][i] * w[i]:
//   rstd[t]  = r_t
//   dx[t][i] = r_t * g[i] - xh[t][i] * (r_t^3 * sum_j g[j] xh[t][j] / H)
//   dw[i]    = sum_t dy[t][i] * xh[t][i] * r_t
//
// Row kernel: one CTA of 256 threads per row (an octet of lanes per 128-element
// block, lane j holding chunks j and j+8, at most kRowBlocks blocks per octet
// held in registers): the codes, scales, dy and w of the row are read once,
// the two row sums are reduced over the CTA in a fixed order, and dx and rstd
// are written.
// Weight-gradient kernel: a cluster of 8 CTAs per 256-column slice; each of the
// 64 warps of the cluster sums every 64th row for its 256 columns (one chunk
// of 8 columns per lane), the warps' sums are added in a fixed order in shared
// memory, and rank 0 adds the 8 CTAs' sums in rank order through distributed
// shared memory.  No global scratch, no atomics: dw is deterministic.
#include <cooperative_groups.h>

#include "agoq_device.cuh"
#include "agoq_launch.h"

namespace agoq {
namespace {

namespace cg = cooperative_groups;

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kRowThreads = 256;                 // 32 octets: one row per CTA iteration
constexpr int kRowOctets = kRowThreads / 8;
constexpr int kRowBlocks = 2;                    // 128-element blocks per octet (H <= 8192)
constexpr int kDwThreads = 256;                  // 8 warps
constexpr int kDwCluster = 8;                    // CTAs per cluster (ranks along y)
constexpr int kDwCols = 256;                     // columns per slice (32 lanes x 8)
constexpr int kDwUnroll = 4;                     // rows in flight per warp

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Element k (0..7) of a chunk of 8 BF16 values.
__device__ __forceinline__ float elem(const uint4 &v, int k) {
    const uint32_t w = (k >> 1) == 0 ? v.x : (k >> 1) == 1 ? v.y : (k >> 1) == 2 ? v.z : v.w;
    return (k & 1) ? bf16_hi(w) : bf16_lo(w);
}

template <int BITS>
__global__ void __launch_bounds__(kRowThreads) rmsnorm_backward_rows_kernel(
    const uint32_t *__restrict__ codes, const float *__restrict__ scales,
    const uint4 *__restrict__ dy, const uint4 *__restrict__ w, int64_t T, int H, float eps,
    uint4 *__restrict__ dx, float *__restrict__ rstd) {
    pdl_wait_and_release();
    constexpr int kWords = 4 * BITS;
    __shared__ float red[2][kRowThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int oct = threadIdx.x >> 3, j = lane & 7;
    const int nb = H / kBlock;                   // blocks per row
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        // xh: dequantized input, dv: upstream gradient, wv: weight (8 BF16 per chunk)
        uint4 xh[kRowBlocks][2], dv[kRowBlocks][2], wv[kRowBlocks][2];
        float sxx = 0.0f, sgx = 0.0f;
#pragma unroll
        for (int q = 0; q < kRowBlocks; ++q) {
            const int b = oct + kRowOctets * q;  // block of the row
            if (b < nb) {
                const int64_t blk = t * nb + b;
                uint32_t lo, hi;
                const float s = __ldg(scales + blk);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    load_chunk<BITS>(codes + blk * kWords, j + 8 * h, lo, hi);
                    xh[q][h] = dequantize_chunk<BITS>(lo, hi, s);
                    dv[q][h] = ld_stream(dy + blk * 16 + j + 8 * h);
                    wv[q][h] = __ldg(w + (int64_t)b * 16 + j + 8 * h);
                }
            }
        }
        // row sums
#pragma unroll
        for (int q = 0; q < kRowBlocks; ++q) {
            const int b = oct + kRowOctets * q;
            if (b < nb) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float x = elem(xh[q][h], k);
                        const float gg = __fmul_rn(elem(dv[q][h], k), elem(wv[q][h], k));
                        sxx = __fadd_rn(sxx, __fmul_rn(x, x));
                        sgx = __fadd_rn(sgx, __fmul_rn(gg, x));
                    }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sxx = __fadd_rn(sxx, __shfl_xor_sync(kFull, sxx, o));
            sgx = __fadd_rn(sgx, __shfl_xor_sync(kFull, sgx, o));
        }
        if (lane == 0) {
            red[0][warp] = sxx;
            red[1][warp] = sgx;
        }
        __syncthreads();
        float txx = 0.0f, tgx = 0.0f;
#pragma unroll
        for (int i = 0; i < kRowThreads / 32; ++i) {
            txx = __fadd_rn(txx, red[0][i]);
            tgx = __fadd_rn(tgx, red[1][i]);
        }
        __syncthreads();   // red is rewritten for the next row
        const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(txx, (float)H), eps)));
        const float kk = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), __fdiv_rn(tgx, (float)H));
        if (threadIdx.x == 0) rstd[t] = r;
#pragma unroll
        for (int q = 0; q < kRowBlocks; ++q) {
            const int b = oct + kRowOctets * q;
            if (b < nb) {
                const int64_t blk = t * nb + b;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t o[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        float d[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int k = 2 * p + e;
                            const float gg = __fmul_rn(elem(dv[q][h], k), elem(wv[q][h], k));
                            d[e] = __fsub_rn(__fmul_rn(r, gg), __fmul_rn(elem(xh[q][h], k), kk));
                        }
                        o[p] = pack_bf16x2(d[0], d[1]);
                    }
                    dx[blk * 16 + j + 8 * h] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(kDwThreads) rmsnorm_dw_kernel(
    const uint32_t *__restrict__ codes, const float *__restrict__ scales,
    const uint4 *__restrict__ dy, const float *__restrict__ rstd, int64_t T, int H,
    float *__restrict__ dw) {
    pdl_wait_and_release();
    constexpr int kWords = 4 * BITS;
    __shared__ float part[kDwThreads / 32][kDwCols];
    __shared__ float csum[kDwCols];
    cg::cluster_group cluster = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = (int)cluster.block_rank();                  // 0 .. kDwCluster-1
    const int group = rank * (kDwThreads / 32) + warp;            // 0 .. 63
    constexpr int kGroups = kDwCluster * (kDwThreads / 32);
    const int nb = H / kBlock;
    const int col0 = blockIdx.x * kDwCols + 8 * lane;             // this lane's 8 columns
    const int b = col0 / kBlock, chunk = (col0 % kBlock) / 8;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
    for (int64_t t0 = group; t0 < T; t0 += (int64_t)kGroups * kDwUnroll) {
        uint32_t lo[kDwUnroll], hi[kDwUnroll];
        float s[kDwUnroll], r[kDwUnroll];
        uint4 d[kDwUnroll];
#pragma unroll
        for (int u = 0; u < kDwUnroll; ++u) {
            const int64_t t = t0 + (int64_t)kGroups * u;
            if (t < T) {
                const int64_t blk = t * nb + b;
                load_chunk<BITS>(codes + blk * kWords, chunk, lo[u], hi[u]);
                s[u] = __ldg(scales + blk);
                r[u] = __ldg(rstd + t);
                d[u] = ld_stream(dy + (t * H + col0) / 8);
            } else {
                lo[u] = hi[u] = 0u;
                s[u] = r[u] = 0.0f;
                d[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < kDwUnroll; ++u) {
            const uint4 xh = dequantize_chunk<BITS>(lo[u], hi[u], s[u]);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                acc[k] = __fadd_rn(acc[k], __fmul_rn(__fmul_rn(elem(d[u], k), elem(xh, k)), r[u]));
        }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) part[warp][8 * lane + k] = acc[k];
    __syncthreads();
    {
        float v = 0.0f;
#pragma unroll
        for (int i = 0; i < kDwThreads / 32; ++i) v = __fadd_rn(v, part[i][threadIdx.x]);
        csum[threadIdx.x] = v;
    }
    cluster.sync();
    if (rank == 0) {
        float v = 0.0f;
        for (int q = 0; q < kDwCluster; ++q)
            v = __fadd_rn(v, cluster.map_shared_rank(csum, q)[threadIdx.x]);
        dw[blockIdx.x * kDwCols + threadIdx.x] = v;
    }
    cluster.sync();   // the other CTAs' csum stays alive until rank 0 has read it
}

template <typename K>
int rows_grid(K kernel, int64_t T) {
    static int per_sm[kMaxDevices];
    int64_t g = (int64_t)sm_count() * resident_per_sm(kernel, kRowThreads, 0, per_sm);
    if (T < g) g = T;
    return (int)(g > 0 ? g : 1);
}

template <int BITS>
cudaError_t rmsnorm_bits(const void *codes, const float *scales, const void *dy, const void *w,
                         int64_t T, int H, float eps, void *dx, float *rstd, float *dw,
                         cudaStream_t st) {
    auto kr = rmsnorm_backward_rows_kernel<BITS>;
    cudaError_t e = launch_pdl(kr, rows_grid(kr, T), kRowThreads, 0, st,
                               static_cast<const uint32_t *>(codes), scales,
                               static_cast<const uint4 *>(dy), static_cast<const uint4 *>(w), T, H,
                               eps, static_cast<uint4 *>(dx), rstd);
    if (e != cudaSuccess || !dw) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(H / kDwCols, kDwCluster, 1);
    cfg.blockDim = dim3(kDwThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = kDwCluster;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, rmsnorm_dw_kernel<BITS>, static_cast<const uint32_t *>(codes),
                              scales, static_cast<const uint4 *>(dy),
                              static_cast<const float *>(rstd), T, H, dw);
}

}  // namespace

cudaError_t launch_rmsnorm_backward(const void *codes, const float *scales, const void *dy,
                                    const void *w, int64_t T, int64_t H, int bits, float eps,
                                    void *dx, float *rstd, float *dw, cudaStream_t st) {
    switch (bits) {
        case 4: return rmsnorm_bits<4>(codes, scales, dy, w, T, (int)H, eps, dx, rstd, dw, st);
        case 5: return rmsnorm_bits<5>(codes, scales, dy, w, T, (int)H, eps, dx, rstd, dw, st);
        case 6: return rmsnorm_bits<6>(codes, scales, dy, w, T, (int)H, eps, dx, rstd, dw, st);
        case 8: return rmsnorm_bits<8>(codes, scales, dy, w, T, (int)H, eps, dx, rstd, dw, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace agoq
