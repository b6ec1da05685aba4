// laaq.cu -- LAAQ block-wise activation quantize / dequantize at 4, 5, 6 and 8
// bits ("AGoQ: Activation and Gradient Quantization for Memory-Efficient
// Distributed Training of LLMs", section 2.A: "Strategie" for 4 bits,
// "Dynamic Bit-width Compensation (DBCA-PP)" for 5, 6 and 8 bits;
// "Herberekening versus Caching" for reading the stored input back).
//
// Work decomposition: a half warp owns one 128-element block; lane j of the
// half holds elements 8j..8j+7 (one 16-byte BF16 load or store), so a warp
// moves two adjacent blocks (512 contiguous bytes of BF16) per memory
// instruction, and UNROLL block pairs are in flight per warp.  The block
// absmax is a 4-step shuffle reduction inside the half warp.  Lane j's eight
// codes form a chunk of 8*bits bits at bit 8*bits*j of the block record:
//   bits 4, 8 : the chunk is one aligned 4- or 8-byte word;
//   bits 5    : 4 lanes (160 bits) fill 5 aligned words; lane q of the group
//               writes word q from its own chunk and lane q-1's, and lane 3
//               also writes word 4;
//   bits 6    : 2 lanes (96 bits) fill 3 words the same way.
// The grid is one resident wave striding over the blocks.
#include "agoq_device.cuh"
#include "agoq_launch.h"

#ifndef AGOQ_QUANT_UNROLL
#define AGOQ_QUANT_UNROLL 2
#endif
#ifndef AGOQ_DEQUANT_UNROLL
#define AGOQ_DEQUANT_UNROLL 4
#endif

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

__device__ __forceinline__ void st_stream(uint4 *p, uint4 v) {
    asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Quantize the lane's 8 BF16 values (block scale reduced over the half warp).
template <int BITS>
__device__ __forceinline__ void quantize_lane(const uint4 v, float &scale, uint32_t &lo,
                                              uint32_t &hi) {
    constexpr int kQmax = (1 << (BITS - 1)) - 1;
    float f[8];
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    float am = fabsf(f[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
    am = halfwarp_max(am);
    const float s = __fdiv_rn(am, (float)kQmax);   // +0 for an all-zero block
    scale = s;
    uint32_t cb[8];
    integer_codes8<kQmax>(f, s, cb);
    pack_fields8<BITS>(cb, lo, hi);
}

// Write the lane's chunk (lo, hi) into the block record `rec` (4*BITS words).
// Every lane of the warp must call this (5 and 6 bits shuffle); `valid` gates
// the stores.
template <int BITS>
__device__ __forceinline__ void store_chunk(uint32_t *rec, int lane, uint32_t lo, uint32_t hi,
                                            bool valid) {
    const int j = lane & 15;
    if constexpr (BITS == 4) {
        if (valid) rec[j] = lo;
    } else if constexpr (BITS == 8) {
        if (valid) reinterpret_cast<uint2 *>(rec)[j] = make_uint2(lo, hi);
    } else if constexpr (BITS == 5) {
        // group of 4 lanes g = j/4, q = j%4; chunk q starts at bit 40q of the group's 160 bits
        const uint32_t plo = __shfl_up_sync(kFull, lo, 1);
        const uint32_t phi = __shfl_up_sync(kFull, hi, 1);
        const int q = j & 3;
        uint32_t *w = rec + 5 * (j >> 2);
        const uint32_t word = q == 0 ? lo : (__funnelshift_rc(plo, phi, 40 - 8 * q) | (lo << (8 * q)));
        if (valid) {
            w[q] = word;
            if (q == 3) w[4] = __funnelshift_r(lo, hi, 8);
        }
    } else {  // BITS == 6: group of 2 lanes, chunk q starts at bit 48q of 96 bits
        const uint32_t phi = __shfl_up_sync(kFull, hi, 1);
        const int q = j & 1;
        uint32_t *w = rec + 3 * (j >> 1);
        if (valid) {
            if (q == 0) {
                w[0] = lo;
            } else {
                w[1] = phi | (lo << 16);
                w[2] = __funnelshift_r(lo, hi, 16);
            }
        }
    }
}

template <int BITS, int UNROLL>
__global__ void __launch_bounds__(kThreads) laaq_quant_kernel(const uint4 *__restrict__ x,
                                                              uint32_t *__restrict__ codes,
                                                              float *__restrict__ scales,
                                                              int64_t nblocks) {
    constexpr int kWords = 4 * BITS;
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, j = lane & 15;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = warp * (2 * UNROLL); base < nblocks; base += nwarps * (2 * UNROLL)) {
        uint4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            v[u] = blk < nblocks ? ld_stream(x + blk * 16 + j) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            const bool valid = blk < nblocks;
            float s;
            uint32_t lo, hi;
            quantize_lane<BITS>(v[u], s, lo, hi);
            store_chunk<BITS>(codes + blk * kWords, lane, lo, hi, valid);
            if (valid && j == 0) scales[blk] = s;
        }
    }
}

// The lane's 8*BITS-bit chunk of a block record, as (lo, hi).
template <int BITS>
__device__ __forceinline__ void load_chunk(const uint32_t *rec, int j, uint32_t &lo, uint32_t &hi) {
    if constexpr (BITS == 4) {
        lo = __ldg(rec + j);
        hi = 0u;
    } else if constexpr (BITS == 8) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(rec) + j);
        lo = w.x;
        hi = w.y;
    } else {
        const int byte = BITS * j;                          // chunk starts at this byte
        const uint32_t a = __ldg(rec + (byte >> 2));
        const uint32_t b = __ldg(rec + (byte >> 2) + 1);    // still inside the record
        const int sh = 8 * (byte & 3);
        lo = __funnelshift_r(a, b, sh);
        hi = b >> sh;
    }
}

template <int BITS>
__device__ __forceinline__ uint4 dequantize_lane(uint32_t lo, uint32_t hi, float s) {
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(field_value<BITS>(lo, hi, i * BITS), s);
    return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                      pack_bf16x2(y[6], y[7]));
}

template <int BITS, int UNROLL>
__global__ void __launch_bounds__(kThreads) laaq_dequant_kernel(const uint32_t *__restrict__ codes,
                                                                const float *__restrict__ scales,
                                                                uint4 *__restrict__ y,
                                                                int64_t nblocks) {
    constexpr int kWords = 4 * BITS;
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, j = lane & 15;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = warp * (2 * UNROLL); base < nblocks; base += nwarps * (2 * UNROLL)) {
        uint32_t lo[UNROLL], hi[UNROLL];
        float s[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            if (blk < nblocks) {
                load_chunk<BITS>(codes + blk * kWords, j, lo[u], hi[u]);
                s[u] = __ldg(scales + blk);
            } else {
                lo[u] = hi[u] = 0u;
                s[u] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            if (blk < nblocks) st_stream(y + blk * 16 + j, dequantize_lane<BITS>(lo[u], hi[u], s[u]));
        }
    }
}

template <typename K>
int resident_grid(K kernel, int *cache, int64_t work_ctas) {
    int64_t g = (int64_t)sm_count() * resident_per_sm(kernel, kThreads, 0, cache);
    if (work_ctas < g) g = work_ctas;
    return (int)(g > 0 ? g : 1);
}

template <int BITS>
cudaError_t quant_bits(const void *x, int64_t nblocks, void *codes, float *scales, cudaStream_t st) {
    constexpr int kU = AGOQ_QUANT_UNROLL;
    static int cache[kMaxDevices];
    auto k = laaq_quant_kernel<BITS, kU>;
    const int64_t per_cta = 2 * kU * (kThreads / 32);
    k<<<resident_grid(k, cache, (nblocks + per_cta - 1) / per_cta), kThreads, 0, st>>>(
        static_cast<const uint4 *>(x), static_cast<uint32_t *>(codes), scales, nblocks);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t dequant_bits(const void *codes, const float *scales, int64_t nblocks, void *y,
                         cudaStream_t st) {
    constexpr int kU = AGOQ_DEQUANT_UNROLL;
    static int cache[kMaxDevices];
    auto k = laaq_dequant_kernel<BITS, kU>;
    const int64_t per_cta = 2 * kU * (kThreads / 32);
    k<<<resident_grid(k, cache, (nblocks + per_cta - 1) / per_cta), kThreads, 0, st>>>(
        static_cast<const uint32_t *>(codes), scales, static_cast<uint4 *>(y), nblocks);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_laaq_quant(const void *x, int64_t n, int bits, void *codes, float *scales,
                              cudaStream_t st) {
    const int64_t nb = n / kBlock;
    switch (bits) {
        case 4: return quant_bits<4>(x, nb, codes, scales, st);
        case 5: return quant_bits<5>(x, nb, codes, scales, st);
        case 6: return quant_bits<6>(x, nb, codes, scales, st);
        case 8: return quant_bits<8>(x, nb, codes, scales, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_laaq_dequant(const void *codes, const float *scales, int64_t n, int bits, void *y,
                                cudaStream_t st) {
    const int64_t nb = n / kBlock;
    switch (bits) {
        case 4: return dequant_bits<4>(codes, scales, nb, y, st);
        case 5: return dequant_bits<5>(codes, scales, nb, y, st);
        case 6: return dequant_bits<6>(codes, scales, nb, y, st);
        case 8: return dequant_bits<8>(codes, scales, nb, y, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace agoq
