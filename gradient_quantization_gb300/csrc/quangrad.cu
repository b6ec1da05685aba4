// quangrad.cu -- QuanGrad FP8 gradient kernels ("AGoQ: Activation and Gradient
// Quantization for Memory-Efficient Distributed Training of LLMs", section 2.B):
//   * local accumulation ("Lokale accumulatie"): dequantize the FP8 master,
//     add the micro-batch gradient in FP32, requantize with a fresh block scale;
//   * the local reduce of the precision-preserved all-reduce (step 2, "Lokale
//     reduce"): dequantize W received FP8 shards, sum them in FP32 in rank
//     order, requantize; optionally count where a naive FP8 sum overflows.
//
// Accumulation: a half warp owns a 128-element block, lane j holds elements
// 8j..8j+7 (8 bytes of master codes, 16 bytes of BF16 gradient); the master is
// rewritten in place by the same lane that read it.
// Reduce: 8 lanes own a block, each lane 16 elements (one 16-byte load of
// codes per shard), so a warp reads 4 adjacent blocks (512 contiguous bytes)
// of every shard per load instruction; RUNROLL shards are loaded ahead.
#include "agoq_device.cuh"
#include "agoq_launch.h"

namespace agoq {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kThreads = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Requantize 8 binary32 values held by one lane, given the block's absmax `am`
// (already reduced over the block): codes = e4m3_rne_satfinite(fl(t / s')),
// s' = fl(am / 448); an all-zero block gives s' = +0 and zero codes.
__device__ __forceinline__ uint2 requant8(const float t[8], float am, float &s_out) {
    const float s = __fdiv_rn(am, kE4M3Max);
    s_out = s;
    if (am == 0.0f) return make_uint2(0u, 0u);
    uint32_t c[4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
        c[p] = e4m3x2_from_f32(__fdiv_rn(t[2 * p], s), __fdiv_rn(t[2 * p + 1], s));
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

template <int UNROLL>
__global__ void __launch_bounds__(kThreads) grad_accum_kernel(uint2 *__restrict__ master,
                                                              float *__restrict__ scales,
                                                              const uint4 *__restrict__ grad,
                                                              int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, j = lane & 15;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = warp * (2 * UNROLL); base < nblocks; base += nwarps * (2 * UNROLL)) {
        uint2 mc[UNROLL];
        uint4 g[UNROLL];
        float s[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            if (blk < nblocks) {
                mc[u] = master[blk * 16 + j];
                s[u] = scales[blk];
                g[u] = ld_stream(grad + blk * 16 + j);
            } else {
                mc[u] = make_uint2(0u, 0u);
                s[u] = 0.0f;
                g[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            float e[8], t[8];
            e4m3x2_to_f32(mc[u].x & 0xFFFFu, e[0], e[1]);
            e4m3x2_to_f32(mc[u].x >> 16, e[2], e[3]);
            e4m3x2_to_f32(mc[u].y & 0xFFFFu, e[4], e[5]);
            e4m3x2_to_f32(mc[u].y >> 16, e[6], e[7]);
            const float gv[8] = {bf16_lo(g[u].x), bf16_hi(g[u].x), bf16_lo(g[u].y), bf16_hi(g[u].y),
                                 bf16_lo(g[u].z), bf16_hi(g[u].z), bf16_lo(g[u].w), bf16_hi(g[u].w)};
            float am = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                t[i] = __fadd_rn(__fmul_rn(e[i], s[u]), gv[i]);
                am = fmaxf(am, fabsf(t[i]));
            }
            am = halfwarp_max(am);
            float snew;
            const uint2 out = requant8(t, am, snew);
            if (blk < nblocks) {
                master[blk * 16 + j] = out;
                if (j == 0) scales[blk] = snew;
            }
        }
    }
}

// One E4M3 value rounded again from an exact binary32 sum (|t| <= 448).
__device__ __forceinline__ void e4m3_round_pair(float &a, float &b) {
    e4m3x2_to_f32(e4m3x2_from_f32(a, b), a, b);
}

template <bool NAIVE, int RUNROLL>
__global__ void __launch_bounds__(kThreads) reduce_shards_kernel(
    const uint4 *__restrict__ shards, const float *__restrict__ shard_scales, int W, int64_t n,
    int64_t nblocks, uint4 *__restrict__ out, float *__restrict__ out_scales,
    unsigned long long *__restrict__ naive_count) {
    const int lane = threadIdx.x & 31;
    const int oct = lane >> 3, t8 = lane & 7;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t shard_vec = n / 16;   // uint4 per shard
    unsigned long long overflowed = 0;
    for (int64_t base = warp * 4; base < nblocks; base += nwarps * 4) {
        const int64_t blk = base + oct;
        const bool valid = blk < nblocks;
        const int64_t blk_c = valid ? blk : nblocks - 1;   // in-range address for idle lanes
        float acc[16];
        float nv[16];
        uint32_t alive = 0xFFFFu;
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        for (int r0 = 0; r0 < W; r0 += RUNROLL) {
            uint4 c[RUNROLL];
            float s[RUNROLL];
#pragma unroll
            for (int u = 0; u < RUNROLL; ++u) {
                const int r = r0 + u < W ? r0 + u : W - 1;
                c[u] = ld_stream(shards + (int64_t)r * shard_vec + blk_c * 8 + t8);
                s[u] = __ldg(shard_scales + (int64_t)r * nblocks + blk_c);
            }
#pragma unroll
            for (int u = 0; u < RUNROLL; ++u) {
                const int r = r0 + u;
                if (r >= W) break;
                const uint32_t w4[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
                float e[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    e4m3x2_to_f32(w4[q] & 0xFFFFu, e[4 * q], e[4 * q + 1]);
                    e4m3x2_to_f32(w4[q] >> 16, e[4 * q + 2], e[4 * q + 3]);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(e[i], s[u]));
                if constexpr (NAIVE) {
                    if (r == 0) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) nv[i] = e[i];
                    } else if (alive) {
                        float tt[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            tt[i] = __fadd_rn(nv[i], e[i]);   // exact: both are E4M3 values
                            if (fabsf(tt[i]) > kE4M3Max) alive &= ~(1u << i);
                        }
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            e4m3_round_pair(tt[i], tt[i + 1]);
                            nv[i] = tt[i];
                            nv[i + 1] = tt[i + 1];
                        }
                    }
                }
            }
        }
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(acc[i]));
        am = octet_max(am);
        float s0, s1;
        const uint2 lo = requant8(acc, am, s0);
        const uint2 hi = requant8(acc + 8, am, s1);
        if (valid) {
            out[blk * 8 + t8] = make_uint4(lo.x, lo.y, hi.x, hi.y);
            if (t8 == 0) out_scales[blk] = s0;
            if constexpr (NAIVE) overflowed += (unsigned long long)__popc(~alive & 0xFFFFu);
        }
    }
    if constexpr (NAIVE) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) overflowed += __shfl_xor_sync(kFull, overflowed, o);
        if (lane == 0 && overflowed) atomicAdd(naive_count, overflowed);
    }
}

template <typename K>
int resident_grid(K kernel, int *cache, int64_t work_ctas) {
    int64_t g = (int64_t)sm_count() * resident_per_sm(kernel, kThreads, 0, cache);
    if (work_ctas < g) g = work_ctas;
    return (int)(g > 0 ? g : 1);
}

}  // namespace

cudaError_t launch_grad_accum(void *master, float *master_scales, const void *grad, int64_t n,
                              cudaStream_t st) {
    constexpr int kUnroll = 2;
    static int cache[kMaxDevices];
    const int64_t nb = n / kBlock;
    auto k = grad_accum_kernel<kUnroll>;
    const int64_t per_cta = 2 * kUnroll * (kThreads / 32);
    k<<<resident_grid(k, cache, (nb + per_cta - 1) / per_cta), kThreads, 0, st>>>(
        static_cast<uint2 *>(master), master_scales, static_cast<const uint4 *>(grad), nb);
    return cudaGetLastError();
}

cudaError_t launch_reduce_shards(const void *shards, const float *shard_scales, int W, int64_t n,
                                 void *out, float *out_scales, unsigned long long *naive_count,
                                 cudaStream_t st) {
    constexpr int kRUnroll = 4;
    const int64_t nb = n / kBlock;
    const int64_t per_cta = 4 * (kThreads / 32);
    const int64_t ctas = (nb + per_cta - 1) / per_cta;
    if (naive_count) {
        cudaError_t e = cudaMemsetAsync(naive_count, 0, sizeof(unsigned long long), st);
        if (e != cudaSuccess) return e;
        static int cache[kMaxDevices];
        auto k = reduce_shards_kernel<true, kRUnroll>;
        k<<<resident_grid(k, cache, ctas), kThreads, 0, st>>>(
            static_cast<const uint4 *>(shards), shard_scales, W, n, nb, static_cast<uint4 *>(out),
            out_scales, naive_count);
    } else {
        static int cache[kMaxDevices];
        auto k = reduce_shards_kernel<false, kRUnroll>;
        k<<<resident_grid(k, cache, ctas), kThreads, 0, st>>>(
            static_cast<const uint4 *>(shards), shard_scales, W, n, nb, static_cast<uint4 *>(out),
            out_scales, nullptr);
    }
    return cudaGetLastError();
}

}  // namespace agoq
