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
// Row kernels: the codes, scales, dy and w of each row are read once, the two
// row sums are reduced in a fixed order, and dx and rstd are written.  For
// H = 4096 one warp owns a row (shuffle reductions only, w staged in shared
// memory); other H (multiples of 256 up to 8192) use one CTA of 256 threads per
// row with an octet of lanes per 128-element block.
// Weight-gradient kernel: a cluster of 8 CTAs per 128-column slice; each of the
// 128 half warps of the cluster sums every 128th row for its 128 columns (one
// chunk of 8 columns per lane, 8 rows in flight), the half warps' sums are
// added in a fixed order in shared memory, and rank 0 adds the 8 CTAs' sums in
// rank order through distributed shared memory.  No global scratch, no
// atomics: dw is deterministic.
#include <cooperative_groups.h>
#include <mutex>

#include "agoq_device.cuh"
#include "agoq_launch.h"
#include "gemm_common.cuh"

namespace agoq {
namespace {

namespace cg = cooperative_groups;

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kRowThreads = 256;                 // 32 octets: one row per CTA iteration
constexpr int kRowOctets = kRowThreads / 8;
constexpr int kRowBlocks = 2;                    // 128-element blocks per octet (H <= 8192)
constexpr int kDwThreads = 256;                  // 8 warps
constexpr int kDwCluster = 8;                    // CTAs per cluster (ranks along y)
constexpr int kDwCols = 128;                     // columns per slice (16 lanes x 8)
constexpr int kDwUnroll = 4;                     // rows in flight per half warp
// dw through TMA-staged row tiles (when T, H and the alignments allow it):
// kDwTileRows rows of a 128-column slice per stage, kDwStagesTma stages,
// kDwTmaCluster CTAs per slice (4, 6, 9 and 12 stages and clusters of 4, 12 or
// 16 CTAs measured slower than 8 and 8).
constexpr int kDwTileRows = 32;
constexpr int kDwTmaCluster = 8;                 // CTAs per slice (cluster along y)
constexpr int kDwStagesTma = 8;
constexpr int kDwTmaMinCtas = 2;
constexpr int kDwTmaThreads = kDwThreads + 32;   // 8 consumer warps + 1 producer warp

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

// General row kernel (any H that is a multiple of 256, up to 8192): a CTA of
// 256 threads per row, an octet of lanes per 128-element block (lane j holding
// chunks j and j+8, at most kRowBlocks blocks per octet in registers).
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
        // fixed-order reduction: lanes (xor tree), then the 8 warps in order
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

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Chunk c (8 codes) of a row's concatenated block records in shared memory:
// the row's records are contiguous, so chunk c starts at byte BITS * c.
template <int BITS>
__device__ __forceinline__ void chunk_from_smem(const uint32_t *rowcodes, int c, uint32_t &lo,
                                                uint32_t &hi) {
    if constexpr (BITS == 4) {
        lo = rowcodes[c];
        hi = 0u;
    } else if constexpr (BITS == 8) {
        const uint2 v = reinterpret_cast<const uint2 *>(rowcodes)[c];
        lo = v.x;
        hi = v.y;
    } else {
        const int byte = BITS * c;
        const uint32_t a = rowcodes[byte >> 2], b = rowcodes[(byte >> 2) + 1];
        const int sh = 8 * (byte & 3);
        lo = __funnelshift_r(a, b, sh);
        hi = b >> sh;
    }
}

constexpr int kWarpRowThreads = 128;             // 4 warps per CTA, one row per warp at a time

// The row kernels form the BF16 x BF16 products (xh^2, xh w, dy w) with the
// mixed-precision fma.rn.f32.bf16 on the BF16 halves directly instead of
// widening both operands first.  Each such product is exact in binary32, so
// the sums and dx are the same bits either way (measured faster).

// d_k = fl(a_k * b_k + c_k) for the BF16 halves k = 0 (bits 0-15), 1 of a and b.
__device__ __forceinline__ void fma_bf16x2_f32(uint32_t a, uint32_t b, float c0, float c1,
                                               float &d0, float &d1) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %4;\n\tfma.rn.f32.bf16 %1, ah, bh, %5;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(a), "r"(b), "f"(c0), "f"(c1));
}

// dw terms of one chunk: acc[k] += fl(fl(dy_k * xh_k) * r) for the 8 BF16
// values of d (dy) and xh (the BF16 x BF16 product is exact in binary32).
__device__ __forceinline__ void dw_accum8(float acc[8], const uint4 &d, const uint4 &xh, float r) {
    const uint32_t dw4[4] = {d.x, d.y, d.z, d.w}, xw[4] = {xh.x, xh.y, xh.z, xh.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float q0, q1;
        fma_bf16x2_f32(dw4[p], xw[p], -0.0f, -0.0f, q0, q1);
        acc[2 * p] = __fadd_rn(acc[2 * p], __fmul_rn(q0, r));
        acc[2 * p + 1] = __fadd_rn(acc[2 * p + 1], __fmul_rn(q1, r));
    }
}

// Shared-memory words of one warp's row stage: dy (H/8 x 16 B), the row's
// codes (H*BITS/8 B, padded by 16 B so a 5/6-bit chunk read may touch the
// next word) and its H/128 scales.
template <int BITS, int H>
struct RowStage {
    static constexpr int kDy = H / 8;                        // uint4
    static constexpr int kCodes = H * BITS / 128 + 1;        // uint4
    static constexpr int kScales = (H / kBlock + 3) / 4;     // uint4
    static constexpr int kU4 = kDy + kCodes + kScales;
};

// Row kernel for H = 256 * C (C chunks of 8 elements per lane): one warp per
// row, lane l handling chunks l, l + 32, ...  The warp stages its row's dy,
// codes and scales in shared memory with cp.async (the next row's copies in
// flight while the current row is computed), forms the row sums from shared
// memory, reduces them with shuffles alone, then forms dx.  w is staged once
// per CTA.  The cp.async waits are hardware group completions.
template <int BITS, int C>
__global__ void __launch_bounds__(kWarpRowThreads) rmsnorm_backward_warp_rows_kernel(
    const uint32_t *__restrict__ codes, const float *__restrict__ scales,
    const uint4 *__restrict__ dy, const uint4 *__restrict__ w, int64_t T, float eps,
    uint4 *__restrict__ dx, float *__restrict__ rstd) {
    pdl_wait_and_release();
    constexpr int H = 256 * C, nb = H / kBlock;
    using St = RowStage<BITS, H>;
    extern __shared__ uint4 smem4[];
    uint4 *ws = smem4;                                       // H/8
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint4 *stage0 = smem4 + H / 8 + (size_t)wid * 2 * St::kU4;
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) ws[i] = __ldg(w + i);
    __syncthreads();
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    auto issue = [&](int64_t t, int buf) {
        uint4 *st = stage0 + buf * St::kU4;
        const uint4 *dyr = dy + t * (H / 8);
#pragma unroll
        for (int k = 0; k < C; ++k) cp_async16(st + lane + 32 * k, dyr + lane + 32 * k);
        const uint4 *cr = reinterpret_cast<const uint4 *>(codes + (size_t)t * nb * 4 * BITS);
        for (int i = lane; i < St::kCodes - 1; i += 32) cp_async16(st + St::kDy + i, cr + i);
        float *sc = reinterpret_cast<float *>(st + St::kDy + St::kCodes);
        for (int i = lane; i < nb; i += 32) cp_async4(sc + i, scales + t * nb + i);
        cp_async_commit();
    };
    int64_t t = gw;
    int buf = 0;
    if (t < T) issue(t, 0);
    for (; t < T; t += nw, buf ^= 1) {
        if (t + nw < T) {
            issue(t + nw, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncwarp();
        const uint4 *dyS = stage0 + buf * St::kU4;
        const uint32_t *cS = reinterpret_cast<const uint32_t *>(dyS + St::kDy);
        const float *sS = reinterpret_cast<const float *>(dyS + St::kDy + St::kCodes);
        auto xh_of = [&](int k) {
            const int c = lane + 32 * k;
            uint32_t lo, hi;
            chunk_from_smem<BITS>(cS, c, lo, hi);
            return dequantize_chunk<BITS>(lo, hi, sS[c / 16]);
        };
        // Row sums in packed pairs with fused multiply-adds (a tolerance-
        // bounded result: fusing only removes roundings).
        uint64_t sxx2 = 0ull, sgx2 = 0ull;
        float sxx0 = 0.0f, sxx1 = 0.0f;
#pragma unroll 4
        for (int k = 0; k < C; ++k) {
            const uint4 xh = xh_of(k);
            const uint4 dv = dyS[lane + 32 * k];
            const uint4 wv = ws[lane + 32 * k];
            const uint32_t xw[4] = {xh.x, xh.y, xh.z, xh.w}, dw4[4] = {dv.x, dv.y, dv.z, dv.w},
                           ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                // sxx += xh^2;  sgx += dy * (xh w): the same exact products as (dy w) xh
                float v0, v1;
                fma_bf16x2_f32(xw[p], xw[p], sxx0, sxx1, sxx0, sxx1);
                fma_bf16x2_f32(xw[p], ww[p], -0.0f, -0.0f, v0, v1);
                sgx2 = fma_f32x2(u32x2(dw4[p] << 16, dw4[p] & 0xFFFF0000u), f32x2(v0, v1), sgx2);
            }
        }
        sxx2 = f32x2(sxx0, sxx1);
        float sxx = __fadd_rn(lo_f32(sxx2), hi_f32(sxx2));
        float sgx = __fadd_rn(lo_f32(sgx2), hi_f32(sgx2));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sxx = __fadd_rn(sxx, __shfl_xor_sync(kFull, sxx, o));
            sgx = __fadd_rn(sgx, __shfl_xor_sync(kFull, sgx, o));
        }
        const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(sxx, (float)H), eps)));
        const float kk = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), __fdiv_rn(sgx, (float)H));
        if (lane == 0) rstd[t] = r;
        const uint64_t r2 = f32x2(r, r), nkk2 = f32x2(-kk, -kk);
#pragma unroll 4
        for (int k = 0; k < C; ++k) {
            const uint4 xh = xh_of(k);
            const uint4 dv = dyS[lane + 32 * k];
            const uint4 wv = ws[lane + 32 * k];
            const uint32_t xw[4] = {xh.x, xh.y, xh.z, xh.w}, dw4[4] = {dv.x, dv.y, dv.z, dv.w},
                           ww[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t o[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint64_t x2 = u32x2(xw[p] << 16, xw[p] & 0xFFFF0000u);
                float g0, g1;
                fma_bf16x2_f32(dw4[p], ww[p], -0.0f, -0.0f, g0, g1);
                const uint64_t g2 = f32x2(g0, g1);
                // dx = r * g - xh * kk
                const uint64_t d2 = fma_f32x2(r2, g2, mul_f32x2(x2, nkk2));
                o[p] = pack_bf16x2(lo_f32(d2), hi_f32(d2));
            }
            dx[t * (H / 8) + lane + 32 * k] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncwarp();   // every lane is done with this stage before it is refilled
    }
}

template <int BITS, int C>
constexpr size_t warp_rows_smem() {
    return sizeof(uint4) * (256 * C / 8 + (kWarpRowThreads / 32) * 2 * RowStage<BITS, 256 * C>::kU4);
}

template <int BITS>
__global__ void __launch_bounds__(kDwThreads, 2) rmsnorm_dw_kernel(
    const uint32_t *__restrict__ codes, const float *__restrict__ scales,
    const uint4 *__restrict__ dy, const float *__restrict__ rstd, int64_t T, int H,
    float *__restrict__ dw) {
    pdl_wait_and_release();
    constexpr int kWords = 4 * BITS;
    constexpr int kHalves = 2 * (kDwThreads / 32);                 // row groups per CTA
    __shared__ float part[kHalves][kDwCols];
    __shared__ float csum[kDwCols];
    cg::cluster_group cluster = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int half = lane >> 4, l16 = lane & 15;
    const int rank = (int)cluster.block_rank();                    // 0 .. kDwCluster-1
    const int hw = 2 * warp + half;                                // 0 .. kHalves-1
    const int group = rank * kHalves + hw;                          // 0 .. 127
    constexpr int kGroups = kDwCluster * kHalves;
    const int nb = H / kBlock;
    const int col0 = blockIdx.x * kDwCols + 8 * l16;                // this lane's 8 columns
    const int b = col0 / kBlock, chunk = (col0 % kBlock) / 8;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
    // kDwUnroll rows per batch; the next batch's loads are issued before the
    // current batch is accumulated (register double buffering)
    struct Batch {
        uint32_t lo[kDwUnroll], hi[kDwUnroll];
        float s[kDwUnroll], r[kDwUnroll];
        uint4 d[kDwUnroll];
    };
    auto load = [&](int64_t t0, Batch &bt) {
#pragma unroll
        for (int u = 0; u < kDwUnroll; ++u) {
            const int64_t t = t0 + (int64_t)kGroups * u;
            if (t < T) {
                const int64_t blk = t * nb + b;
                load_chunk<BITS>(codes + blk * kWords, chunk, bt.lo[u], bt.hi[u]);
                bt.s[u] = __ldg(scales + blk);
                bt.r[u] = __ldg(rstd + t);
                bt.d[u] = ld_stream(dy + (t * H + col0) / 8);
            } else {
                bt.lo[u] = bt.hi[u] = 0u;
                bt.s[u] = bt.r[u] = 0.0f;
                bt.d[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    };
    constexpr int64_t kStep = (int64_t)kGroups * kDwUnroll;
    Batch cur, nxt;
    int64_t t0 = group;
    if (t0 < T) load(t0, cur);
    for (; t0 < T; t0 += kStep) {
        const bool more = t0 + kStep < T;
        if (more) load(t0 + kStep, nxt);
#pragma unroll
        for (int u = 0; u < kDwUnroll; ++u) {
            const uint4 xh = dequantize_chunk<BITS>(cur.lo[u], cur.hi[u], cur.s[u]);
            dw_accum8(acc, cur.d[u], xh, cur.r[u]);
        }
        if (more) cur = nxt;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) part[hw][8 * l16 + k] = acc[k];
    __syncthreads();
    if (threadIdx.x < kDwCols) {
        float v = 0.0f;
#pragma unroll
        for (int i = 0; i < kHalves; ++i) v = __fadd_rn(v, part[i][threadIdx.x]);
        csum[threadIdx.x] = v;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x < kDwCols) {
        float v = 0.0f;
        for (int q = 0; q < kDwCluster; ++q)
            v = __fadd_rn(v, cluster.map_shared_rank(csum, q)[threadIdx.x]);
        dw[blockIdx.x * kDwCols + threadIdx.x] = v;
    }
    cluster.sync();   // the other CTAs' csum stays alive until rank 0 has read it
}

__device__ unsigned g_rms_status;

// Shared-memory layout of one stage of the TMA dw kernel (offsets 128-byte
// aligned): dy [32][128] BF16, the slice's block records [32][16 BITS] bytes,
// the scales of the 4-block group holding the slice [32][4], rstd [32].
template <int BITS>
struct DwTmaStage {
    static constexpr int kDy = 0;
    static constexpr int kCodes = kDwTileRows * 256;
    static constexpr int kScales = kCodes + kDwTileRows * 16 * BITS;
    static constexpr int kRstd = kScales + kDwTileRows * 16;
    static constexpr int kBytes = kRstd + kDwTileRows * 4;
    static constexpr uint32_t kTx = kBytes;
    static_assert(kBytes % 128 == 0, "stages stay 128-byte aligned");
};

// dw[i] = sum_t dy[t][i] * xh[t][i] * r_t with the rows streamed by TMA: a
// cluster of 8 CTAs per 128-column slice; CTA rank q takes the contiguous
// 32-row tiles [q S/8, (q+1) S/8) of the S = T/32 tiles.  One producer lane
// loads each tile (dy, codes and scales as 2-D tensor boxes, rstd as one bulk
// copy) into a kDwStagesTma-deep ring; half warp h of the CTA sums rows h and
// h + 16 of every tile, in row order, for its 8 columns (so each column's sum
// is a chain of T/128 rows per half warp, then the 16 half warps and the 8
// CTAs in fixed order, as in rmsnorm_dw_kernel).  Waits are time-limited: on
// expiry g_rms_status records a timeout, the CTA stops (still joining the
// cluster barriers) and the producer waits for its copies in flight.
template <int BITS>
__global__ void __launch_bounds__(kDwTmaThreads, kDwTmaMinCtas) rmsnorm_dw_tma_kernel(
    const __grid_constant__ CUtensorMap map_dy, const __grid_constant__ CUtensorMap map_codes,
    const __grid_constant__ CUtensorMap map_scales, const float *__restrict__ rstd, int64_t T,
    float *__restrict__ dw) {
    using namespace gemm;
    using St = DwTmaStage<BITS>;
    constexpr int kHalves = 2 * (kDwThreads / 32);                 // 16 consumer half warps
    extern __shared__ __align__(128) uint8_t dwt_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(dwt_raw) + 127) & ~static_cast<uintptr_t>(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)kDwStagesTma * St::kBytes);
    uint64_t *empty = full + kDwStagesTma;
    __shared__ float part[kHalves][kDwCols];
    __shared__ float csum[kDwCols];
    __shared__ int abort_flag;
    cg::cluster_group cluster = cg::this_cluster();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x;                                       // slice = block b of each row
    const int64_t tiles = T / kDwTileRows;
    const int64_t tile0 = tiles * rank / kDwTmaCluster, tile1 = tiles * (rank + 1) / kDwTmaCluster;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDwStagesTma; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kDwThreads / 32);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_wait_and_release();
    volatile int *abort = &abort_flag;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
    const int half = lane >> 4, l16 = lane & 15, hw = 2 * warp + half;

    if (warp == kDwThreads / 32) {
        if (lane == 0) {
            uint32_t it = 0;
            for (int64_t tl = tile0; tl < tile1; ++tl, ++it) {
                const int s = it % kDwStagesTma;
                const uint32_t ph = (it / kDwStagesTma) & 1u;
                if (it >= (uint32_t)kDwStagesTma &&
                    !wait_bar(&empty[s], ph ^ 1u, abort, &g_rms_status))
                    break;
                uint8_t *st = smem + (size_t)s * St::kBytes;
                const int y = (int)(tl * kDwTileRows);
                mbar_expect_tx(&full[s], St::kTx);
                tma_load_2d(st + St::kDy, &map_dy, &full[s], b * kDwCols, y);
                tma_load_2d(st + St::kCodes, &map_codes, &full[s], b * 16 * BITS, y);
                tma_load_2d(st + St::kScales, &map_scales, &full[s], b & ~3, y);
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], "
                    "%2, [%3];" ::"r"(smem_u32(st + St::kRstd)),
                    "l"(rstd + (int64_t)y), "r"(kDwTileRows * 4), "r"(smem_u32(&full[s]))
                    : "memory");
            }
            // copies still in flight land before the CTA may exit
            const uint32_t first = it > (uint32_t)kDwStagesTma ? it - kDwStagesTma : 0u;
            for (uint32_t j = first; j < it; ++j)
                wait_bar(&full[j % kDwStagesTma], (j / kDwStagesTma) & 1u, abort, &g_rms_status,
                         true);
        }
    } else {
        uint32_t it = 0;
        for (int64_t tl = tile0; tl < tile1; ++tl, ++it) {
            const int s = it % kDwStagesTma;
            if (!warp_wait(&full[s], (it / kDwStagesTma) & 1u, abort, &g_rms_status)) break;
            mbar_try_wait(&full[s], (it / kDwStagesTma) & 1u, 0);   // each lane's own acquire
            const uint8_t *st = smem + (size_t)s * St::kBytes;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int row = hw + kHalves * rr;                   // 0 .. 31
                const float sc = reinterpret_cast<const float *>(st + St::kScales)[4 * row + (b & 3)];
                const float r = reinterpret_cast<const float *>(st + St::kRstd)[row];
                uint32_t lo, hi;
                chunk_from_smem<BITS>(
                    reinterpret_cast<const uint32_t *>(st + St::kCodes + row * 16 * BITS), l16, lo, hi);
                const uint4 xh = dequantize_chunk<BITS>(lo, hi, sc);
                const uint4 d = reinterpret_cast<const uint4 *>(st + St::kDy + row * 256)[l16];
                dw_accum8(acc, d, xh, r);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    if (warp < kDwThreads / 32) {
#pragma unroll
        for (int k = 0; k < 8; ++k) part[hw][8 * l16 + k] = acc[k];
    }
    __syncthreads();
    if (threadIdx.x < kDwCols) {
        float v = 0.0f;
#pragma unroll
        for (int i = 0; i < kHalves; ++i) v = __fadd_rn(v, part[i][threadIdx.x]);
        csum[threadIdx.x] = v;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x < kDwCols) {
        float v = 0.0f;
        for (int q = 0; q < kDwTmaCluster; ++q)
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

// dw through rmsnorm_dw_tma_kernel: T a multiple of 32, H of 512, scales and
// rstd 16-byte aligned (the caller has checked).
template <int BITS>
cudaError_t launch_dw_tma(const void *codes, const float *scales, const void *dy, const float *rstd,
                          int64_t T, int H, float *dw, cudaStream_t st) {
    using namespace gemm;
    using Stg = DwTmaStage<BITS>;
    const int nb = H / kBlock;
    CUtensorMap m_dy, m_codes, m_scales;
    if (!encode_2d(&m_dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dy, (uint64_t)H, (uint64_t)T,
                   (uint64_t)H * 2, kDwCols, kDwTileRows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&m_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, (uint64_t)nb * 16 * BITS,
                   (uint64_t)T, (uint64_t)nb * 16 * BITS, 16 * BITS, kDwTileRows,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&m_scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, scales, (uint64_t)nb, (uint64_t)T,
                   (uint64_t)nb * 4, 4, kDwTileRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    constexpr size_t smem = (size_t)kDwStagesTma * (Stg::kBytes + 16) + 128;
    static bool attr_set[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevices && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(rmsnorm_dw_tma_kernel<BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (kDwTmaCluster > 8) {
            e = cudaFuncSetAttribute(rmsnorm_dw_tma_kernel<BITS>,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(H / kDwCols, kDwTmaCluster, 1);
    cfg.blockDim = dim3(kDwTmaThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = kDwTmaCluster;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, rmsnorm_dw_tma_kernel<BITS>, m_dy, m_codes, m_scales, rstd, T,
                              dw);
}

template <int BITS>
cudaError_t rmsnorm_bits(const void *codes, const float *scales, const void *dy, const void *w,
                         int64_t T, int H, float eps, void *dx, float *rstd, float *dw,
                         cudaStream_t st) {
    cudaError_t e;
    if (H == 4096) {
        auto kr = rmsnorm_backward_warp_rows_kernel<BITS, 16>;
        constexpr size_t smem = warp_rows_smem<BITS, 16>();
        static int per_sm[kMaxDevices];
        static bool attr_set[kMaxDevices];
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev >= 0 && dev < kMaxDevices && !attr_set[dev]) {
            e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
        int64_t g = (int64_t)sm_count() * resident_per_sm(kr, kWarpRowThreads, smem, per_sm);
        const int64_t need = (T + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32);
        if (need < g) g = need;
        e = launch_pdl(kr, (int)(g > 0 ? g : 1), kWarpRowThreads, smem, st,
                       static_cast<const uint32_t *>(codes), scales,
                       static_cast<const uint4 *>(dy), static_cast<const uint4 *>(w), T, eps,
                       static_cast<uint4 *>(dx), rstd);
    } else {
        auto kr = rmsnorm_backward_rows_kernel<BITS>;
        e = launch_pdl(kr, rows_grid(kr, T), kRowThreads, 0, st,
                       static_cast<const uint32_t *>(codes), scales,
                       static_cast<const uint4 *>(dy), static_cast<const uint4 *>(w), T, H, eps,
                       static_cast<uint4 *>(dx), rstd);
    }
    if (e != cudaSuccess || !dw) return e;
    if (T % kDwTileRows == 0 && T / kDwTileRows <= INT32_MAX / kDwTileRows &&
        H % 512 == 0 && reinterpret_cast<uintptr_t>(scales) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(rstd) % 16 == 0)
        return launch_dw_tma<BITS>(codes, scales, dy, rstd, T, H, dw, st);
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

// ---- single-pass backward: dx, rstd and the dw partial sums in one read ----
// A row group of 128 threads (4 warps) takes one row at a time; thread i of the
// group holds chunks i, i + 128, ... (CPT of them, 8 columns each) of the row,
// so its dequantized input, dy and w stay in registers from the row sums to dx
// and the dw terms (the input is dequantized once).  A CTA is two row groups:
// CTA p of G takes rows 2p + g, 2p + g + 2G, ... in group g, the next row's
// loads in flight while the current one is computed.  The two row sums are
// reduced with shuffles, then over the group's 4 warps in shared memory in
// warp order (one CTA barrier per row; the buffers alternate by row).  Each
// thread adds its columns' dw terms fma(dy * xh, r, sum) (the BF16 x BF16
// product is exact; one rounding per term) in row order; at the
// end group 1's sums are added to group 0's and written as the CTA's row of
// `partials` [G][H].  rmsnorm_dw_partials_kernel then adds the G rows in a
// fixed order: eight contiguous ranges of ceil(G/8) rows, each summed in row
// order, then the eight range sums in order.  Every dw sum is therefore a chain
// of at most ceil(T/2G) + 1 + ceil(G/8) + 8 additions, and the result does not
// depend on the schedule.
constexpr int kFusedThreads = 256, kFusedGroup = 128, kFusedMaxH = 4096;
constexpr int kFusedPartials = 304;              // G at most: the workspace is G x H floats
constexpr int kFusedL2Ahead = 3;                 // rows asked of the L2 ahead of the loads

template <int BITS, int CPT>
__global__ void __launch_bounds__(kFusedThreads, 2) rmsnorm_backward_fused_kernel(
    const uint32_t *__restrict__ codes, const float *__restrict__ scales,
    const uint4 *__restrict__ dy, const uint4 *__restrict__ w, int64_t T, int H, float eps,
    uint4 *__restrict__ dx, float *__restrict__ rstd, float *__restrict__ partials) {
    pdl_wait_and_release();
    constexpr int kWords = 4 * BITS;
    __shared__ float red[2][2][2][kFusedGroup / 32];   // [group][row parity][sum][warp]
    __shared__ __align__(16) float comb[kFusedMaxH];   // group 1's dw sums at the end
    const int g = threadIdx.x / kFusedGroup, i = threadIdx.x % kFusedGroup;
    const int lane = threadIdx.x & 31, wg = i >> 5;
    const int nch = H / 8, nb = H / kBlock;
    const bool full = nch == kFusedGroup * CPT;        // every thread has CPT chunks
    // 1/H when H is a power of two (then x * (1/H) is x / H exactly), else 0
    const float inv_h = (H & (H - 1)) == 0 ? 1.0f / (float)H : 0.0f;
    uint4 wv[CPT];
    uint64_t acc[CPT][4];                               // dw sums, column pairs
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        const int c = i + kFusedGroup * k;
        wv[k] = full || c < nch ? __ldg(w + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[k][p] = 0ull;
    }
    struct RowIn {
        uint4 d[CPT];
        uint32_t lo[CPT], hi[CPT];
        float s[CPT];
    };
    // Row t's inputs (zeros for chunks past H or a row past T).
    auto load = [&](int64_t t, RowIn &in) {
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = i + kFusedGroup * k;
            if (t < T && (full || c < nch)) {
                const int64_t blk = t * nb + c / 16;
                load_chunk<BITS>(codes + blk * kWords, c % 16, in.lo[k], in.hi[k]);
                in.s[k] = __ldg(scales + blk);
                in.d[k] = ld_stream(dy + t * nch + c);
            } else {
                in.lo[k] = in.hi[k] = 0u;
                in.s[k] = 0.0f;
                in.d[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    };
    const int64_t stride = 2 * (int64_t)gridDim.x;
    // One thread of each group asks the L2 for a row's dy and codes
    // kFusedL2Ahead rows before its loads are issued (a hint: no effect on results).
    auto l2_ahead = [&](int64_t t) {
        if (i == 0 && t < T) {
            prefetch_l2(dy + t * nch, (uint32_t)H * 2u);
            prefetch_l2(codes + t * nb * kWords, (uint32_t)(H / 8) * BITS);
        }
    };
    // Row t of this group from `in`; every thread of the CTA calls it for every
    // row pair (its barrier), with t past T for a group without a row.
    auto process = [&](const RowIn &in, int64_t t, int par) {
        uint4 xh[CPT];
        float sxx0 = 0.0f, sxx1 = 0.0f;
        uint64_t sgx2 = 0ull;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            xh[k] = dequantize_chunk<BITS>(in.lo[k], in.hi[k], in.s[k]);
            const uint32_t xw[4] = {xh[k].x, xh[k].y, xh[k].z, xh[k].w};
            const uint32_t dw4[4] = {in.d[k].x, in.d[k].y, in.d[k].z, in.d[k].w};
            const uint32_t ww[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                // sxx += xh^2;  sgx += dy * (xh w) (exact BF16 x BF16 products)
                float v0, v1;
                fma_bf16x2_f32(xw[p], xw[p], sxx0, sxx1, sxx0, sxx1);
                fma_bf16x2_f32(xw[p], ww[p], -0.0f, -0.0f, v0, v1);
                sgx2 = fma_f32x2(u32x2(dw4[p] << 16, dw4[p] & 0xFFFF0000u), f32x2(v0, v1), sgx2);
            }
        }
        float sxx = __fadd_rn(sxx0, sxx1);
        float sgx = __fadd_rn(lo_f32(sgx2), hi_f32(sgx2));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sxx = __fadd_rn(sxx, __shfl_xor_sync(kFull, sxx, o));
            sgx = __fadd_rn(sgx, __shfl_xor_sync(kFull, sgx, o));
        }
        if (lane == 0) {
            red[g][par][0][wg] = sxx;
            red[g][par][1][wg] = sgx;
        }
        __syncthreads();
        sxx = red[g][par][0][0];
        sgx = red[g][par][1][0];
#pragma unroll
        for (int q = 1; q < kFusedGroup / 32; ++q) {
            sxx = __fadd_rn(sxx, red[g][par][0][q]);
            sgx = __fadd_rn(sgx, red[g][par][1][q]);
        }
        const float mxx = inv_h != 0.0f ? __fmul_rn(sxx, inv_h) : __fdiv_rn(sxx, (float)H);
        const float mgx = inv_h != 0.0f ? __fmul_rn(sgx, inv_h) : __fdiv_rn(sgx, (float)H);
        const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(mxx, eps)));
        const float kk = __fmul_rn(__fmul_rn(__fmul_rn(r, r), r), mgx);
        if (t < T) {
            if (i == 0) rstd[t] = r;
            const uint64_t r2 = f32x2(r, r), nkk2 = f32x2(-kk, -kk);
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int c = i + kFusedGroup * k;
                if (!full && c >= nch) continue;
                const uint32_t xw[4] = {xh[k].x, xh[k].y, xh[k].z, xh[k].w};
                const uint32_t dw4[4] = {in.d[k].x, in.d[k].y, in.d[k].z, in.d[k].w};
                const uint32_t ww[4] = {wv[k].x, wv[k].y, wv[k].z, wv[k].w};
                uint32_t o[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    // dx = r * g - xh * kk, g = dy * w
                    float g0, g1, q0, q1;
                    fma_bf16x2_f32(dw4[p], ww[p], -0.0f, -0.0f, g0, g1);
                    const uint64_t x2 = u32x2(xw[p] << 16, xw[p] & 0xFFFF0000u);
                    const uint64_t d2 = fma_f32x2(r2, f32x2(g0, g1), mul_f32x2(x2, nkk2));
                    o[p] = pack_bf16x2(lo_f32(d2), hi_f32(d2));
                    // dw += (dy xh) r, the exact product scaled and added in one rounding
                    fma_bf16x2_f32(dw4[p], xw[p], -0.0f, -0.0f, q0, q1);
                    acc[k][p] = fma_f32x2(f32x2(q0, q1), r2, acc[k][p]);
                }
                dx[t * nch + c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    };
    RowIn ra, rb;
    const int64_t first = 2 * (int64_t)blockIdx.x + g;
#pragma unroll
    for (int a = 0; a <= kFusedL2Ahead; ++a) l2_ahead(first + a * stride);
    load(first, ra);
    // Rows alternate between the two input buffers (no copies); both groups
    // run the same row pairs.
    int par = 0;
    for (int64_t b0 = 2 * (int64_t)blockIdx.x; b0 < T; b0 += 2 * stride) {
        l2_ahead(b0 + g + (kFusedL2Ahead + 1) * stride);
        load(b0 + g + stride, rb);
        process(ra, b0 + g, par);
        par ^= 1;
        if (b0 + stride >= T) break;
        l2_ahead(b0 + g + (kFusedL2Ahead + 2) * stride);
        load(b0 + g + 2 * stride, ra);
        process(rb, b0 + g + stride, par);
        par ^= 1;
    }
    // group 0's sums + group 1's sums -> this CTA's partial row
    __syncthreads();
    if (g == 1) {
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = i + kFusedGroup * k;
            if (full || c < nch) {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    comb[8 * c + 2 * p] = lo_f32(acc[k][p]);
                    comb[8 * c + 2 * p + 1] = hi_f32(acc[k][p]);
                }
            }
        }
    }
    __syncthreads();
    if (g == 0) {
        float4 *prow = reinterpret_cast<float4 *>(partials + (size_t)blockIdx.x * H);
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = i + kFusedGroup * k;
            if (full || c < nch) {
                float v[8];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    v[2 * p] = __fadd_rn(lo_f32(acc[k][p]), comb[8 * c + 2 * p]);
                    v[2 * p + 1] = __fadd_rn(hi_f32(acc[k][p]), comb[8 * c + 2 * p + 1]);
                }
                prow[2 * c] = make_float4(v[0], v[1], v[2], v[3]);
                prow[2 * c + 1] = make_float4(v[4], v[5], v[6], v[7]);
            }
        }
    }
}

// dw[col] from the G partial rows in a fixed order: a CTA takes 32 columns;
// warp q sums rows q*R .. q*R + R - 1 (R = ceil(G/8)) in row order, then the
// eight warp sums are added in warp order.
constexpr int kPartialsWarps = 8;
__global__ void __launch_bounds__(32 * kPartialsWarps) rmsnorm_dw_partials_kernel(
    const float *__restrict__ partials, int G, int H, float *__restrict__ dw) {
    pdl_wait_and_release();
    __shared__ float wsum[kPartialsWarps][32];
    const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + lane;       // H is a multiple of 256
    const int R = (G + kPartialsWarps - 1) / kPartialsWarps;
    const int p0 = q * R, p1 = p0 + R < G ? p0 + R : G;
    float s = 0.0f;
    int p = p0;
    for (; p + 8 <= p1; p += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __ldg(partials + (size_t)(p + j) * H + col);
#pragma unroll
        for (int j = 0; j < 8; ++j) s = __fadd_rn(s, v[j]);
    }
    for (; p < p1; ++p) s = __fadd_rn(s, __ldg(partials + (size_t)p * H + col));
    wsum[q][lane] = s;
    __syncthreads();
    if (q == 0) {
        float tot = wsum[0][lane];
#pragma unroll
        for (int k = 1; k < kPartialsWarps; ++k) tot = __fadd_rn(tot, wsum[k][lane]);
        dw[col] = tot;
    }
}

// G: as many CTAs as are resident at once (at most kFusedPartials), so that
// every CTA runs in one wave; G depends on the GPU, so dw's order of additions
// (and last bits) is fixed per GPU model.
template <int BITS>
cudaError_t rmsnorm_fused_bits(const void *codes, const float *scales, const void *dy,
                               const void *w, int64_t T, int H, float eps, void *dx, float *rstd,
                               float *dw, float *partials, cudaStream_t st) {
    const int cpt = (H / 8 + kFusedGroup - 1) / kFusedGroup;   // chunks per thread
    static int cache[4][kMaxDevices];
    int per_sm = 1;
    switch (cpt) {
        case 1: per_sm = resident_per_sm(rmsnorm_backward_fused_kernel<BITS, 1>, kFusedThreads, 0, cache[0]); break;
        case 2: per_sm = resident_per_sm(rmsnorm_backward_fused_kernel<BITS, 2>, kFusedThreads, 0, cache[1]); break;
        case 3: per_sm = resident_per_sm(rmsnorm_backward_fused_kernel<BITS, 3>, kFusedThreads, 0, cache[2]); break;
        default: per_sm = resident_per_sm(rmsnorm_backward_fused_kernel<BITS, 4>, kFusedThreads, 0, cache[3]); break;
    }
    int64_t G = (T + 1) / 2;
    const int64_t resident = (int64_t)sm_count() * per_sm;
    if (G > resident) G = resident;
    if (G > kFusedPartials) G = kFusedPartials;
    cudaError_t e = cudaSuccess;
    if (G > 0) {
        auto args = [&](auto kernel) {
            return launch_pdl(kernel, (int)G, kFusedThreads, 0, st,
                              static_cast<const uint32_t *>(codes), scales,
                              static_cast<const uint4 *>(dy), static_cast<const uint4 *>(w), T, H,
                              eps, static_cast<uint4 *>(dx), rstd, partials);
        };
        switch (cpt) {
            case 1: e = args(rmsnorm_backward_fused_kernel<BITS, 1>); break;
            case 2: e = args(rmsnorm_backward_fused_kernel<BITS, 2>); break;
            case 3: e = args(rmsnorm_backward_fused_kernel<BITS, 3>); break;
            default: e = args(rmsnorm_backward_fused_kernel<BITS, 4>); break;
        }
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(rmsnorm_dw_partials_kernel, H / 32, 32 * kPartialsWarps, 0, st,
                      static_cast<const float *>(partials), (int)G, H, dw);
}

}  // namespace

cudaError_t read_and_clear_rmsnorm_status(unsigned *status) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_rms_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_rms_status, &zero, sizeof zero);
        if (e != cudaSuccess) return e;
    }
    *status = v;
    return cudaSuccess;
}

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

// Single-pass form (H <= 4096): `partials` holds rmsnorm_fused_partials() x H
// floats of scratch.
cudaError_t launch_rmsnorm_backward_fused(const void *codes, const float *scales, const void *dy,
                                          const void *w, int64_t T, int64_t H, int bits, float eps,
                                          void *dx, float *rstd, float *dw, float *partials,
                                          cudaStream_t st) {
    switch (bits) {
        case 4: return rmsnorm_fused_bits<4>(codes, scales, dy, w, T, (int)H, eps, dx, rstd, dw, partials, st);
        case 5: return rmsnorm_fused_bits<5>(codes, scales, dy, w, T, (int)H, eps, dx, rstd, dw, partials, st);
        case 6: return rmsnorm_fused_bits<6>(codes, scales, dy, w, T, (int)H, eps, dx, rstd, dw, partials, st);
        case 8: return rmsnorm_fused_bits<8>(codes, scales, dy, w, T, (int)H, eps, dx, rstd, dw, partials, st);
        default: return cudaErrorInvalidValue;
    }
}

int rmsnorm_fused_partials() { return kFusedPartials; }
int rmsnorm_fused_max_h() { return kFusedMaxH; }

// ---- the same single-read backward without a caller-provided workspace ----
// For callers that cannot allocate device memory at the point of the call (a
// framework's custom-operator hook that must not touch the allocator, code
// running while device memory is locked down or accounted by someone else, a
// plain C caller without an allocator of its own), the partial-sum scratch is
// this file-scope array instead of a workspace argument.  It holds the partial
// rows of the largest case the entry point accepts (rows of up to kFusedMaxH =
// 4096 elements: kFusedPartials x 4096 floats, about 5 MB), and every GPU that
// loads the library keeps it until the process exits.
static __device__ __align__(256) float g_rms_noalloc_scratch[kFusedPartials * kFusedMaxH];

// The array's device address, looked up once per device (with that device
// current) on the first call; the name of the array in host code is only a
// stand-in for the symbol and must not be handed to a kernel.
static cudaError_t noalloc_scratch(float **out) {
    static std::mutex lock;
    static float *addr[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> hold(lock);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_rms_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<float *>(p);
    }
    *out = addr[dev];
    return cudaSuccess;
}

// The caller has checked H <= kFusedMaxH.  Every CTA writes its whole partial
// row before the second kernel reads it, so nothing in the array needs to
// start at zero; the array is shared by all calls on a device.
cudaError_t launch_rmsnorm_backward_noalloc(const void *codes, const float *scales, const void *dy,
                                            const void *w, int64_t T, int64_t H, int bits,
                                            float eps, void *dx, float *rstd, float *dw,
                                            cudaStream_t st) {
    float *scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return e;
    return launch_rmsnorm_backward_fused(codes, scales, dy, w, T, H, bits, eps, dx, rstd, dw,
                                         scratch, st);
}

}  // namespace agoq
