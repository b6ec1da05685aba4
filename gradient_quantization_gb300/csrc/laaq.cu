// laaq.cu -- LAAQ block-wise activation quantize / dequantize at 4, 5, 6 and 8
// bits ("AGoQ: Activation and Gradient Quantization for Memory-Efficient
// Distributed Training of LLMs", section 2.A: "Strategie" for 4 bits,
// "Dynamic Bit-width Compensation (DBCA-PP)" for 5, 6 and 8 bits;
// "Herberekening versus Caching" for reading the stored input back).
//
// Work decomposition: a half warp owns one 128-element block; lane j of the
// half holds elements 8j..8j+7 (one 16-byte BF16 load), so a warp moves two
// adjacent blocks (512 contiguous bytes) per load instruction and UNROLL pairs
// of blocks are in flight per warp.  The block absmax is a 4-step shuffle
// reduction inside the half warp.  Lane j's eight codes form a chunk of 8*bits
// bits at bit 8*bits*j of the block record; for 4 and 8 bits the chunk is one
// aligned 4- or 8-byte word, for 5 and 6 bits the record's 32-bit words are
// assembled from two neighbouring chunks fetched with shuffles.
// The grid is sized to one resident wave and strides over the blocks.
#include "agoq_device.cuh"
#include "agoq_launch.h"

namespace agoq {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

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

template <int BITS>
__device__ __forceinline__ uint64_t quantize_chunk(const uint4 v, float &scale_out) {
    constexpr int kQmax = (1 << (BITS - 1)) - 1;
    constexpr uint32_t kMask = (1u << BITS) - 1u;
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
    scale_out = s;
    uint64_t chunk = 0;
    if (am != 0.0f) {
        float k[8];
        if (s >= 0x1p-126f) {
            const float r = __frcp_rn(s);
#pragma unroll
            for (int i = 0; i < 8; ++i) k[i] = rint_quotient(f[i], s, r);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) k[i] = rintf(__fdiv_rn(f[i], s));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float kc = fminf(fmaxf(k[i], -(float)kQmax), (float)kQmax);
            const uint32_t field = (uint32_t)__float2int_rn(kc) & kMask;
            chunk |= (uint64_t)field << (i * BITS);
        }
    }
    return chunk;
}

// Write lane j's chunk into the block record (4*BITS 32-bit words at `rec`).
// Every lane of the warp must call this (it shuffles); `valid` gates the stores.
template <int BITS>
__device__ __forceinline__ void store_chunk(uint32_t *rec, int lane, uint64_t chunk, bool valid) {
    const int j = lane & 15;
    if constexpr (BITS == 4) {
        if (valid) rec[j] = (uint32_t)chunk;
    } else if constexpr (BITS == 8) {
        if (valid) reinterpret_cast<uint2 *>(rec)[j] = make_uint2((uint32_t)chunk, (uint32_t)(chunk >> 32));
    } else {
        constexpr int kWords = 4 * BITS;
        constexpr int kChunkBits = 8 * BITS;
        const uint32_t lo = (uint32_t)chunk, hi = (uint32_t)(chunk >> 32);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int w = j + 16 * t;                       // record word this lane writes
            const int wc = w < kWords ? w : kWords - 1;     // keep the shuffle sources in range
            const int l0 = (32 * wc) / kChunkBits;          // chunk holding the word's first bit
            const int off = 32 * wc - kChunkBits * l0;      // that bit's position in chunk l0
            const int l1 = l0 < 15 ? l0 + 1 : 15;
            const int base = lane & 16;
            const uint32_t a_lo = __shfl_sync(kFull, lo, base | l0);
            const uint32_t a_hi = __shfl_sync(kFull, hi, base | l0);
            const uint32_t b_lo = __shfl_sync(kFull, lo, base | l1);
            const uint32_t b_hi = __shfl_sync(kFull, hi, base | l1);
            uint64_t word = (((uint64_t)a_hi << 32) | a_lo) >> off;
            const int sh = kChunkBits - off;                // chunk l1 starts sh bits into the word
            if (sh < 32) word |= (((uint64_t)b_hi << 32) | b_lo) << sh;
            if (valid && w < kWords) rec[w] = (uint32_t)word;
        }
    }
}

template <int BITS, int UNROLL>
__global__ void __launch_bounds__(256) laaq_quant_kernel(const uint4 *__restrict__ x,
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
            const uint64_t chunk = quantize_chunk<BITS>(v[u], s);
            store_chunk<BITS>(codes + blk * kWords, lane, chunk, valid);
            if (valid && j == 0) scales[blk] = s;
        }
    }
}

template <int BITS>
__device__ __forceinline__ uint64_t load_chunk(const uint32_t *rec, int j) {
    if constexpr (BITS == 4) {
        return __ldg(rec + j);
    } else if constexpr (BITS == 8) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(rec) + j);
        return ((uint64_t)w.y << 32) | w.x;
    } else {
        const int byte = BITS * j;                         // chunk starts at this byte
        const uint32_t lo = __ldg(rec + (byte >> 2));
        const uint32_t hi = __ldg(rec + (byte >> 2) + 1);  // still inside the record
        return ((((uint64_t)hi << 32) | lo) >> (8 * (byte & 3)));
    }
}

template <int BITS>
__device__ __forceinline__ uint4 dequantize_chunk(uint64_t chunk, float s) {
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t field = (uint32_t)(chunk >> (i * BITS));
        const int32_t c = (int32_t)(field << (32 - BITS)) >> (32 - BITS);  // sign-extend
        y[i] = __fmul_rn((float)c, s);
    }
    return make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                      pack_bf16x2(y[6], y[7]));
}

template <int BITS, int UNROLL>
__global__ void __launch_bounds__(256) laaq_dequant_kernel(const uint32_t *__restrict__ codes,
                                                           const float *__restrict__ scales,
                                                           uint4 *__restrict__ y,
                                                           int64_t nblocks) {
    constexpr int kWords = 4 * BITS;
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, j = lane & 15;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = warp * (2 * UNROLL); base < nblocks; base += nwarps * (2 * UNROLL)) {
        uint64_t ch[UNROLL];
        float s[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            if (blk < nblocks) {
                ch[u] = load_chunk<BITS>(codes + blk * kWords, j);
                s[u] = __ldg(scales + blk);
            } else {
                ch[u] = 0;
                s[u] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t blk = base + 2 * u + half;
            if (blk < nblocks) st_stream(y + blk * 16 + j, dequantize_chunk<BITS>(ch[u], s[u]));
        }
    }
}

constexpr int kThreads = 256;
constexpr int kUnroll = 2;

template <typename K>
int resident_grid(K kernel, int *cache, int64_t work_ctas) {
    int64_t g = (int64_t)sm_count() * resident_per_sm(kernel, kThreads, 0, cache);
    if (work_ctas < g) g = work_ctas;
    return (int)(g > 0 ? g : 1);
}

template <int BITS>
cudaError_t quant_bits(const void *x, int64_t nblocks, void *codes, float *scales, cudaStream_t st) {
    static int cache[kMaxDevices];
    auto k = laaq_quant_kernel<BITS, kUnroll>;
    const int64_t ctas = (nblocks + 2 * kUnroll * (kThreads / 32) - 1) / (2 * kUnroll * (kThreads / 32));
    k<<<resident_grid(k, cache, ctas), kThreads, 0, st>>>(static_cast<const uint4 *>(x),
                                                   static_cast<uint32_t *>(codes), scales, nblocks);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t dequant_bits(const void *codes, const float *scales, int64_t nblocks, void *y,
                         cudaStream_t st) {
    static int cache[kMaxDevices];
    auto k = laaq_dequant_kernel<BITS, kUnroll>;
    const int64_t ctas = (nblocks + 2 * kUnroll * (kThreads / 32) - 1) / (2 * kUnroll * (kThreads / 32));
    k<<<resident_grid(k, cache, ctas), kThreads, 0, st>>>(static_cast<const uint32_t *>(codes), scales,
                                                   static_cast<uint4 *>(y), nblocks);
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
