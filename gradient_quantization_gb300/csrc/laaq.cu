// laaq.cu -- LAAQ block-wise activation quantize / dequantize at 4, 5, 6 and 8
// bits ("AGoQ: Activation and Gradient Quantization for Memory-Efficient
// Distributed Training of LLMs", section 2.A: "Strategie" for 4 bits,
// "Dynamic Bit-width Compensation (DBCA-PP)" for 5, 6 and 8 bits;
// "Herberekening versus Caching" for reading the stored input back).
//
// Work decomposition: an octet of lanes owns one 128-element block; lane j
// holds chunks j and j+8 (elements 8j..8j+7 and 64+8j..64+8j+7, two 16-byte
// BF16 loads or stores), so a warp covers four adjacent blocks and UNROLL
// such groups are in flight per warp.  The block absmax is a bf16x2 max over
// the lane's words and a 3-step shuffle reduction inside the octet.  A chunk
// of eight codes is 8*bits bits at bit 8*bits*c of the block record:
//   bits 4, 8 : one aligned 4- or 8-byte word;
//   bits 5    : 4 chunks (160 bits) fill 5 aligned words; the lane holding
//               chunk q of the group writes word q from its chunk and the
//               previous lane's, and the lane of chunk 3 also writes word 4;
//   bits 6    : 2 chunks (96 bits) fill 3 words the same way.
// The grid is one resident wave striding over the blocks.
#include "agoq_device.cuh"
#include "agoq_launch.h"

// Measured choices: quantize 2 block groups per warp in flight with the next
// group's loads issued before the current group's arithmetic (3 CTAs of 256
// threads per SM); dequantize 2 groups per warp, software-pipelined; SiLU
// backward 1 group (4 CTAs per SM, 3 with the recomputed forward output); one
// block group per warp prefetched into L2 before the wait on the preceding grid.
constexpr int kQuantUnroll = 2, kDequantUnroll = 2, kSiluUnroll = 1;
constexpr int kQuantMinCtas = 3, kSiluMinCtas = 4, kSiluYMinCtas = 3;


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

// Write one 8-code chunk set into the block record `rec` (4*BITS words):
// lane j of the octet holds chunk (j + 8*set) as (lo, hi).  Every lane of the
// warp must call this (5 and 6 bits shuffle); `valid` gates the stores.
template <int BITS>
__device__ __forceinline__ void store_chunk_set(uint32_t *rec, int j, int set, uint32_t lo,
                                                uint32_t hi, bool valid) {
    const int c = j + 8 * set;                              // chunk index in the block
    if constexpr (BITS == 4) {
        if (valid) rec[c] = lo;
    } else if constexpr (BITS == 8) {
        if (valid) reinterpret_cast<uint2 *>(rec)[c] = make_uint2(lo, hi);
    } else if constexpr (BITS == 5) {
        // 4 chunks (160 bits) fill 5 words; chunk q of the group starts at bit
        // 40q.  Word q >= 1 is the top 8q bits of chunk q-1 below the low
        // 32-8q bits of chunk q, and word 4 is the top 32 bits of chunk 3.
        // Each lane sends the next one its top 8(q+1) bits (for q = 3 that is
        // word 4 itself); hi holds only the chunk's bits 32-39.
        const int q = c & 3;
        const uint32_t top = __funnelshift_rc(lo, hi, 32 - 8 * q);
        const uint32_t prev = __shfl_up_sync(kFull, top, 1);
        const uint32_t word = (q == 0 ? 0u : prev) | (lo << (8 * q));
        uint32_t *w = rec + 5 * (c >> 2);
        if (valid) {
            w[q] = word;
            if (q == 3) w[4] = top;
        }
    } else {  // BITS == 6: 2 chunks (96 bits) fill 3 words; chunk 1 starts at bit 48
        const uint32_t phi = __shfl_up_sync(kFull, hi, 1);
        uint32_t *w = rec + 3 * (c >> 1);
        if (valid) {
            if ((c & 1) == 0) {
                w[0] = lo;
            } else {
                w[1] = phi | (lo << 16);
                w[2] = __funnelshift_r(lo, hi, 16);
            }
        }
    }
}

// A block is owned by an octet of lanes; lane j holds elements 8j..8j+7
// (chunk j) and 64+8j..64+8j+7 (chunk j+8), so each 16-byte load instruction
// of a warp reads 4 x 128 contiguous bytes and the per-block work (absmax
// shuffles, scale division, reciprocal) is shared by 16 elements per lane.
//
// Block indices are 32-bit: the launcher splits inputs of more than
// kMaxLaunchBlocks blocks into several launches.
template <int BITS, int UNROLL>
__global__ void __launch_bounds__(kThreads, kQuantMinCtas)
laaq_quant_kernel(const uint4 *__restrict__ x, uint32_t *__restrict__ codes,
                  float *__restrict__ scales, int nblocks) {
    {
        // this warp's first group of 4 * UNROLL blocks (256 bytes each)
        const int b0 = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * (4 * UNROLL);
        if ((threadIdx.x & 31) == 0 && b0 < nblocks) {
            const int nb = nblocks - b0 < 4 * UNROLL ? nblocks - b0 : 4 * UNROLL;
            prefetch_l2(x + (size_t)(unsigned)b0 * 16, (uint32_t)nb * 256u);
        }
    }
    pdl_wait_and_release();
    constexpr int kWords = 4 * BITS;
    constexpr int kQmax = (1 << (BITS - 1)) - 1;
    constexpr bool kBiased = BITS < 8;
    constexpr int kBias = kBiased ? (1 << (BITS - 1)) : 0;
    const int lane = threadIdx.x & 31;
    const int oct = lane >> 3, j = lane & 7;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    const int stride = nwarps * (4 * UNROLL);
    auto load_group = [&](int b0, uint4 (&a)[UNROLL], uint4 (&b)[UNROLL]) {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int blk = b0 + 4 * u + oct;
            if (blk < nblocks) {
                const uint4 *p = x + (size_t)(unsigned)blk * 16 + j;
                a[u] = ld_stream(p);
                b[u] = ld_stream(p + 8);
            } else {
                a[u] = b[u] = make_uint4(0, 0, 0, 0);
            }
        }
    };
    // The next group's loads are issued before this group's arithmetic.
    uint4 va[UNROLL], vb[UNROLL];
    load_group(warp * (4 * UNROLL), va, vb);
    for (int base = warp * (4 * UNROLL); base < nblocks; base += stride) {
        uint4 na[UNROLL], nb[UNROLL];
        load_group(base + stride, na, nb);
        uint32_t w[UNROLL][8];
        float s[UNROLL];
        bool fast = true;
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            w[u][0] = va[u].x; w[u][1] = va[u].y; w[u][2] = va[u].z; w[u][3] = va[u].w;
            w[u][4] = vb[u].x; w[u][5] = vb[u].y; w[u][6] = vb[u].z; w[u][7] = vb[u].w;
            const float am = octet_max(bf16_absmax<8>(w[u]));
            s[u] = bf16_div_qmax<kQmax>(am);               // +0 for an all-zero block
            fast &= s[u] >= 0x1p-96f;
        }
        uint32_t cb[UNROLL][16];
        if (fast) {
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) corrected_codes16<kBias>(w[u], s[u], cb[u]);
        } else {
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                float f[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    f[2 * i] = bf16_lo(w[u][i]);
                    f[2 * i + 1] = bf16_hi(w[u][i]);
                }
                if (s[u] >= 0x1p-96f)
                    corrected_codes16<kBias>(w[u], s[u], cb[u]);
                else
                    integer_codes_n<kQmax, 16, kBias>(f, s[u], cb[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int blk = base + 4 * u + oct;
            const bool valid = blk < nblocks;
            uint32_t lo, hi;
            uint32_t *rec = codes + (size_t)(unsigned)blk * kWords;
            if constexpr (kBiased) pack_biased8<BITS>(cb[u], lo, hi);
            else pack_fields8<BITS>(cb[u], lo, hi);
            store_chunk_set<BITS>(rec, j, 0, lo, hi, valid);
            if constexpr (kBiased) pack_biased8<BITS>(cb[u] + 8, lo, hi);
            else pack_fields8<BITS>(cb[u] + 8, lo, hi);
            store_chunk_set<BITS>(rec, j, 1, lo, hi, valid);
            if (valid && j == 0) scales[blk] = s[u];
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            va[u] = na[u];
            vb[u] = nb[u];
        }
    }
}

// Loads of one dequantization batch: UNROLL groups of 4 blocks per warp.
template <int BITS, int UNROLL>
struct DequantBatch {
    uint32_t alo[UNROLL], ahi[UNROLL], blo[UNROLL], bhi[UNROLL];
    float s[UNROLL];

    __device__ __forceinline__ void load(const uint32_t *__restrict__ codes,
                                         const float *__restrict__ scales, int base, int oct,
                                         int j, int nblocks) {
        constexpr int kWords = 4 * BITS;
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int blk = base + 4 * u + oct;
            if (blk < nblocks) {
                const uint32_t *rec = codes + (size_t)(unsigned)blk * kWords;
                load_chunk<BITS>(rec, j, alo[u], ahi[u]);
                load_chunk<BITS>(rec, j + 8, blo[u], bhi[u]);
                s[u] = __ldg(scales + blk);
            } else {
                alo[u] = ahi[u] = blo[u] = bhi[u] = 0u;
                s[u] = 0.0f;
            }
        }
    }
};

// Software-pipelined: the next batch's code and scale loads are issued before
// the current batch is converted and stored, so loads stay in flight.
template <int BITS, int UNROLL>
__global__ void __launch_bounds__(kThreads, 1) laaq_dequant_kernel(const uint32_t *__restrict__ codes,
                                                                const float *__restrict__ scales,
                                                                uint4 *__restrict__ y,
                                                                int nblocks) {
    {
        // codes and scales of this warp's first group of 4 * UNROLL blocks
        const int b0 = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * (4 * UNROLL);
        if ((threadIdx.x & 31) == 0 && b0 < nblocks) {
            const int nb = nblocks - b0 < 4 * UNROLL ? nblocks - b0 : 4 * UNROLL;
            prefetch_l2(codes + (size_t)(unsigned)b0 * (4 * BITS), (uint32_t)nb * (16u * BITS));
            // scales need only 4-byte alignment: prefetched when 16-byte aligned
            if (nb % 4 == 0 && (reinterpret_cast<uintptr_t>(scales + b0) & 15u) == 0)
                prefetch_l2(scales + b0, (uint32_t)nb * 4u);
        }
    }
    pdl_wait_and_release();
    const int lane = threadIdx.x & 31;
    const int oct = lane >> 3, j = lane & 7;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    const int stride = nwarps * (4 * UNROLL);
    int base = warp * (4 * UNROLL);
    if (base >= nblocks) return;
    DequantBatch<BITS, UNROLL> cur, nxt;
    cur.load(codes, scales, base, oct, j, nblocks);
    for (; base < nblocks; base += stride) {
        const bool more = base + stride < nblocks;
        if (more) nxt.load(codes, scales, base + stride, oct, j, nblocks);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int blk = base + 4 * u + oct;
            if (blk < nblocks) {
                uint4 *out = y + (size_t)(unsigned)blk * 16 + j;
                st_stream(out, dequantize_chunk<BITS>(cur.alo[u], cur.ahi[u], cur.s[u]));
                st_stream(out + 8, dequantize_chunk<BITS>(cur.blo[u], cur.bhi[u], cur.s[u]));
            }
        }
        if (more) cur = nxt;
    }
}

// ---- SiLU backward recomputed from the stored input ("Herberekening versus
// Caching", section 2.A: only the low-bit input is kept; the backward pass
// dequantizes it and recomputes the intermediates).  For the 8 dequantized
// values xh of a chunk and the matching upstream gradients dy, in binary32:
//   sigma = 1 / (1 + exp(-xh));  silu'(xh) = sigma * (1 + xh * (1 - sigma));
//   dx = bf16(dy * silu'(xh));   y = bf16(xh * sigma)  (the recomputed forward output).
// e^-x as 2^(-x log2 e) by the hardware's approximate base-2 exponential, and
// the approximate reciprocal (each within a few binary32 ulps; subnormal
// results flush to zero, which leaves sigma at 1 or 0 where they occur).
__device__ __forceinline__ float ex2_approx(float a) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}
__device__ __forceinline__ float rcp_approx(float a) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(a));
    return r;
}

template <bool WITH_Y>
__device__ __forceinline__ void silu_backward_chunk(uint4 xh, uint4 dy, uint4 &dx, uint4 &y) {
    const uint32_t xw[4] = {xh.x, xh.y, xh.z, xh.w};
    const uint32_t dw[4] = {dy.x, dy.y, dy.z, dy.w};
    uint32_t o[4], yo[4];
    constexpr float kNegLog2e = -1.4426950408889634f;
    const uint64_t nl2e = f32x2(kNegLog2e, kNegLog2e), one = f32x2(1.0f, 1.0f);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        // element pairs in packed binary32; every operation rounds separately
        const uint64_t x = f32x2(bf16_lo(xw[p]), bf16_hi(xw[p]));
        const uint64_t d = f32x2(bf16_lo(dw[p]), bf16_hi(dw[p]));
        const uint64_t t = mul_f32x2(x, nl2e);
        const uint64_t den = add_f32x2(f32x2(ex2_approx(lo_f32(t)), ex2_approx(hi_f32(t))), one);
        const uint64_t sg = f32x2(rcp_approx(lo_f32(den)), rcp_approx(hi_f32(den)));
        const uint64_t g = mul_f32x2(sg, fma_f32x2(x, sub_f32x2(one, sg), one));
        const uint64_t r = mul_f32x2(d, g);
        o[p] = pack_bf16x2(lo_f32(r), hi_f32(r));
        if constexpr (WITH_Y) {
            const uint64_t yy = mul_f32x2(x, sg);
            yo[p] = pack_bf16x2(lo_f32(yy), hi_f32(yy));
        }
    }
    dx = make_uint4(o[0], o[1], o[2], o[3]);
    if constexpr (WITH_Y) y = make_uint4(yo[0], yo[1], yo[2], yo[3]);
}

// Same decomposition as the dequantizer (an octet per block, lane j holding
// chunks j and j+8), plus the 16-byte upstream-gradient loads of those chunks;
// the next batch's code, scale and gradient loads are issued before the
// current batch's arithmetic.
template <int BITS, int UNROLL, bool WITH_Y>
__global__ void __launch_bounds__(kThreads, WITH_Y ? kSiluYMinCtas : kSiluMinCtas) laaq_silu_backward_kernel(
    const uint32_t *__restrict__ codes, const float *__restrict__ scales,
    const uint4 *__restrict__ dy, uint4 *__restrict__ dx, uint4 *__restrict__ y,
    int nblocks) {
    pdl_wait_and_release();
    const int lane = threadIdx.x & 31;
    const int oct = lane >> 3, j = lane & 7;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    const int stride = nwarps * (4 * UNROLL);
    int base = warp * (4 * UNROLL);
    if (base >= nblocks) return;
    auto load_dy = [&](int b0, uint4 (&a)[UNROLL], uint4 (&b)[UNROLL]) {
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int blk = b0 + 4 * u + oct;
            if (blk < nblocks) {
                const uint4 *p = dy + (size_t)(unsigned)blk * 16 + j;
                a[u] = ld_stream(p);
                b[u] = ld_stream(p + 8);
            } else {
                a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    };
    DequantBatch<BITS, UNROLL> cur, nxt;
    uint4 da[UNROLL], db[UNROLL], na[UNROLL], nb[UNROLL];
    cur.load(codes, scales, base, oct, j, nblocks);
    load_dy(base, da, db);
    for (; base < nblocks; base += stride) {
        const bool more = base + stride < nblocks;
        if (more) {
            nxt.load(codes, scales, base + stride, oct, j, nblocks);
            load_dy(base + stride, na, nb);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int blk = base + 4 * u + oct;
            if (blk < nblocks) {
                const size_t off = (size_t)(unsigned)blk * 16 + j;
                uint4 ga, gb, ya, yb;
                silu_backward_chunk<WITH_Y>(dequantize_chunk<BITS>(cur.alo[u], cur.ahi[u], cur.s[u]),
                                            da[u], ga, ya);
                silu_backward_chunk<WITH_Y>(dequantize_chunk<BITS>(cur.blo[u], cur.bhi[u], cur.s[u]),
                                            db[u], gb, yb);
                st_stream(dx + off, ga);
                st_stream(dx + off + 8, gb);
                if constexpr (WITH_Y) {
                    st_stream(y + off, ya);
                    st_stream(y + off + 8, yb);
                }
            }
        }
        if (more) {
            cur = nxt;
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                da[u] = na[u];
                db[u] = nb[u];
            }
        }
    }
}

template <typename K>
int resident_grid(K kernel, int *cache, int64_t work_ctas) {
    int64_t g = (int64_t)sm_count() * resident_per_sm(kernel, kThreads, 0, cache);
    if (work_ctas < g) g = work_ctas;
    return (int)(g > 0 ? g : 1);
}

// Largest block count of one quantization launch (32-bit block indices, with
// headroom for the stride arithmetic).
constexpr int64_t kMaxLaunchBlocks = int64_t(1) << 30;

template <int BITS>
cudaError_t quant_bits(const void *x, int64_t nblocks, void *codes, float *scales, cudaStream_t st) {
    constexpr int kU = kQuantUnroll;
    static int cache[kMaxDevices];
    auto k = laaq_quant_kernel<BITS, kU>;
    const int64_t per_cta = 4 * kU * (kThreads / 32);
    for (int64_t b0 = 0; b0 < nblocks; b0 += kMaxLaunchBlocks) {
        const int64_t nb = nblocks - b0 < kMaxLaunchBlocks ? nblocks - b0 : kMaxLaunchBlocks;
        const cudaError_t e = launch_pdl(
            k, resident_grid(k, cache, (nb + per_cta - 1) / per_cta), kThreads, 0, st,
            static_cast<const uint4 *>(x) + b0 * 16,
            static_cast<uint32_t *>(codes) + b0 * 4 * BITS, scales + b0, static_cast<int>(nb));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int BITS>
cudaError_t dequant_bits(const void *codes, const float *scales, int64_t nblocks, void *y,
                         cudaStream_t st) {
    constexpr int kU = kDequantUnroll;
    static int cache[kMaxDevices];
    auto k = laaq_dequant_kernel<BITS, kU>;
    const int64_t per_cta = 4 * kU * (kThreads / 32);
    for (int64_t b0 = 0; b0 < nblocks; b0 += kMaxLaunchBlocks) {
        const int64_t nb = nblocks - b0 < kMaxLaunchBlocks ? nblocks - b0 : kMaxLaunchBlocks;
        const cudaError_t e = launch_pdl(
            k, resident_grid(k, cache, (nb + per_cta - 1) / per_cta), kThreads, 0, st,
            static_cast<const uint32_t *>(codes) + b0 * 4 * BITS, scales + b0,
            static_cast<uint4 *>(y) + b0 * 16, static_cast<int>(nb));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int BITS, bool WITH_Y>
cudaError_t silu_backward_bits(const void *codes, const float *scales, const void *dy,
                               int64_t nblocks, void *dx, void *y, cudaStream_t st) {
    constexpr int kU = kSiluUnroll;
    static int cache[kMaxDevices];
    auto k = laaq_silu_backward_kernel<BITS, kU, WITH_Y>;
    const int64_t per_cta = 4 * kU * (kThreads / 32);
    for (int64_t b0 = 0; b0 < nblocks; b0 += kMaxLaunchBlocks) {
        const int64_t nb = nblocks - b0 < kMaxLaunchBlocks ? nblocks - b0 : kMaxLaunchBlocks;
        const cudaError_t e = launch_pdl(
            k, resident_grid(k, cache, (nb + per_cta - 1) / per_cta), kThreads, 0, st,
            static_cast<const uint32_t *>(codes) + b0 * 4 * BITS, scales + b0,
            static_cast<const uint4 *>(dy) + b0 * 16, static_cast<uint4 *>(dx) + b0 * 16,
            y ? static_cast<uint4 *>(y) + b0 * 16 : nullptr, static_cast<int>(nb));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int BITS>
cudaError_t silu_backward_dispatch(const void *codes, const float *scales, const void *dy,
                                   int64_t nblocks, void *dx, void *y, cudaStream_t st) {
    return y ? silu_backward_bits<BITS, true>(codes, scales, dy, nblocks, dx, y, st)
             : silu_backward_bits<BITS, false>(codes, scales, dy, nblocks, dx, y, st);
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

namespace agoq {

cudaError_t launch_silu_backward(const void *codes, const float *scales, const void *dy, int64_t n,
                                 int bits, void *dx, void *y, cudaStream_t st) {
    const int64_t nb = n / kBlock;
    switch (bits) {
        case 4: return silu_backward_dispatch<4>(codes, scales, dy, nb, dx, y, st);
        case 5: return silu_backward_dispatch<5>(codes, scales, dy, nb, dx, y, st);
        case 6: return silu_backward_dispatch<6>(codes, scales, dy, nb, dx, y, st);
        case 8: return silu_backward_dispatch<8>(codes, scales, dy, nb, dx, y, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace agoq
