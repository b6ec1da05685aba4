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
// of every shard per load instruction.  Two kernels feed that arithmetic: one
// loads the codes into registers itself, several shards ahead; the other
// (used whenever the scale rows allow 16-byte bulk copies) has a producer warp
// stream (tile, shard group) stages into a shared-memory ring with bulk async
// copies, so that far more bytes are in flight per SM than registers can hold.
#include <type_traits>

#include "agoq_device.cuh"
#include "agoq_launch.h"
#include "gemm_common.cuh"

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

// fl(e4m3(code_i) * s) for the 4 codes of word w.
__device__ __forceinline__ void decode_mul4(uint32_t w, float s, float v[4]) {
    float e[4];
    e4m3x2_to_f32(w & 0xFFFFu, e[0], e[1]);
    e4m3x2_to_f32(w >> 16, e[2], e[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __fmul_rn(e[i], s);
}

// Intermediate formats of the accumulation: MID 0 binary32 (t = fl(m + g));
// MID 1 BF16 and MID 2 FP16 (m and g rounded to the format, their sum rounded
// once to it: the page's "dequantize to FP16/BF16, add").
constexpr int kMidF32 = 0, kMidBf16 = 1, kMidF16 = 2;

// In place on t[8] (binary32 products fl(e4m3(c) * s)) and the 8 BF16 gradient
// values of g: t = R(R(t) + R(g)) with R the rounding to the MID format.  The
// format's own add rounds the exact sum once.
template <int MID>
__device__ __forceinline__ void add_in_format(float t[8], const uint4 &g) {
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t r;
        if constexpr (MID == kMidBf16) {
            const uint32_t m = pack_bf16x2(t[2 * p], t[2 * p + 1]);
            asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(gw[p]));
            t[2 * p] = bf16_lo(r);
            t[2 * p + 1] = bf16_hi(r);
        } else {
            uint32_t m, gh;
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(m) : "f"(t[2 * p + 1]), "f"(t[2 * p]));
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(gh) : "f"(bf16_hi(gw[p])), "f"(bf16_lo(gw[p])));
            asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(gh));
            asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\t"
                "cvt.f32.f16 %1, b;\n\t}"
                : "=f"(t[2 * p]), "=f"(t[2 * p + 1])
                : "r"(r));
        }
    }
}

// One lane's 8 elements of a block (every lane of the warp calls it, a half
// warp per block): t = the master's products plus the gradient in the MID
// format, the block's new scale (returned in snew) and the 8 new codes.
template <int MID>
__device__ __forceinline__ uint2 accum_block(const uint2 &mc, const uint4 &g, float s, float &snew) {
    const float gv[8] = {bf16_lo(g.x), bf16_hi(g.x), bf16_lo(g.y), bf16_hi(g.y),
                         bf16_lo(g.z), bf16_hi(g.z), bf16_lo(g.w), bf16_hi(g.w)};
    float t[8];
    decode_mul4(mc.x, s, t);
    decode_mul4(mc.y, s, t + 4);
    float am = 0.0f;
    if constexpr (MID == kMidF32) {
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = __fadd_rn(t[i], gv[i]);
    } else {
        add_in_format<MID>(t, g);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(t[i]));
    am = halfwarp_max(am);
    snew = __fdiv_rn(am, kE4M3Max);
    // BF16-valued sums take the corrected quotient (a bracket near an E4M3
    // rounding boundary is common for them): the BF16 intermediate, and any
    // sum onto an all-zero master block, t = 0 + g in binary32 or
    // t = fp16(g) in FP16 (a BF16 value rounded to the FP16 grid keeps at
    // most 8 significant bits; an FP16 overflow is outside the contract).
    if (MID == kMidBf16 || s == 0.0f) return e4m3_codes8_bf16(t, snew);
    return e4m3_codes8(t, snew);
}

// The register-staged accumulation (master scales not 16-byte aligned, or a
// block count that is not a multiple of 4): each half warp keeps UNROLL blocks
// in flight.
template <int UNROLL, int MID>
__global__ void __launch_bounds__(kThreads) grad_accum_kernel(uint2 *__restrict__ master,
                                                              float *__restrict__ scales,
                                                              const uint4 *__restrict__ grad,
                                                              int64_t nblocks) {
    pdl_wait_and_release();
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, j = lane & 15;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t stride = nwarps * (2 * UNROLL);
    for (int64_t base = warp * (2 * UNROLL); base < nblocks; base += stride) {
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
            float snew;
            const uint2 out = accum_block<MID>(mc[u], g[u], s[u], snew);
            if (blk < nblocks) {
                master[blk * 16 + j] = out;
                if (j == 0) scales[blk] = snew;
            }
        }
    }
}

// ---- the local reduce: per-lane arithmetic -----------------------------------

// Two E4M3 codes (bits 0-15 of v) to an FP16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)v));
    return h2;
}

// An FP16 pair to a binary32 pair held in one 64-bit register (half 0 in the
// low word), exactly.
__device__ __forceinline__ uint64_t f16x2_to_f32x2(uint32_t h2) {
    uint64_t d;
    asm("{\n\t.reg .f16 a, b;\n\t.reg .f32 x, y;\n\tmov.b32 {a, b}, %1;\n\t"
        "cvt.f32.f16 x, a;\n\tcvt.f32.f16 y, b;\n\tmov.b64 %0, {x, y};\n\t}"
        : "=l"(d)
        : "r"(h2));
    return d;
}

// d_k = fl(f32(half k of h2) + c_k): binary32 additions of an FP16 operand.
__device__ __forceinline__ void add_f16x2_f32(uint32_t h2, float c0, float c1, float &d0,
                                              float &d1) {
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "add.rn.f32.f16 %0, a, %3;\n\tadd.rn.f32.f16 %1, b, %4;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(h2), "f"(c0), "f"(c1));
}

// One lane's share of the reduce of one block: 16 elements (one 16-byte load
// of codes per shard), their binary32 running sums over the shards in rank
// order and, with the naive count, the naive FP8 running sums.
//
// The running sums are kept as binary32 pairs.  A shard's products are formed
// as fma(e4m3(c), s, +0) on pairs: that is fl(e4m3(c) * s) except that an
// exactly -0 product becomes +0, which changes nothing here -- the sums start
// at +0 and a binary32 sum is -0 only if both operands are, so no running sum
// is ever -0 and adding +0 or -0 to it gives the same value.  (A multiply
// would be equivalent too, but a packed multiply followed by a packed add has
// been seen contracted into one fused operation by the assembler; a fused
// multiply-add with +0 is not a multiply.)  Each sum is then fl(acc + p), a
// packed round-to-nearest add.
//
// The naive FP8 sum (one shared scale, summed in the code domain) is kept as
// FP16 pairs (every E4M3 value is an FP16 value): step r forms the exact sum
// t = n + e4m3(c_r) in binary32 (mixed FP16 + binary32 add; both operands are
// E4M3 values, so the sum is exact), keeps the largest |t| seen per element
// (an element overflows iff that maximum exceeds 448, which is the first
// overflow's test; later steps cannot undo it), and rounds t to E4M3 through a
// saturating cvt.  Shards are taken two at a time so that one three-input
// maximum covers both steps of an element.
template <bool NAIVE>
struct ReduceLane {
    uint64_t acc[8];   // binary32 running sums, elements (2p, 2p+1)
    uint32_t nvh[8];   // naive running sums, FP16 pairs
    float nmax[16];    // largest |exact naive sum| seen per element

    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int p = 0; p < 8; ++p) acc[p] = 0ull;
        if constexpr (NAIVE) {
#pragma unroll
            for (int i = 0; i < 16; ++i) nmax[i] = 0.0f;
        }
    }

    // Pair p (elements 2p, 2p+1) of one shard: its codes as an FP16 pair h and
    // a binary32 pair e, and its products added to the running sums.
    __device__ __forceinline__ void decode_add(const uint4 &c, uint64_t s2, int p, uint32_t &h,
                                               uint64_t &e) {
        const uint32_t w = p < 2 ? c.x : p < 4 ? c.y : p < 6 ? c.z : c.w;
        h = e4m3x2_to_f16x2((p & 1) ? w >> 16 : w & 0xFFFFu);
        e = f16x2_to_f32x2(h);
        acc[p] = add_f32x2(acc[p], fma_f32x2(e, s2, 0ull));
    }

    // One naive step of pair p with the shard values e (binary32 pair): returns
    // the exact sums t0, t1 and rounds them to E4M3 (nearest even, saturating).
    __device__ __forceinline__ void naive_step(int p, uint64_t e, float &t0, float &t1) {
        add_f16x2_f32(nvh[p], lo_f32(e), hi_f32(e), t0, t1);
        nvh[p] = e4m3x2_to_f16x2(e4m3x2_from_f32(t0, t1));
    }

    // One shard; `first` says it is rank 0.
    __device__ __forceinline__ void add(const uint4 &c, float sc, bool first) {
        const uint64_t s2 = f32x2(sc, sc);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            uint32_t h;
            uint64_t e;
            decode_add(c, s2, p, h, e);
            if constexpr (NAIVE) {
                if (first) {
                    nvh[p] = h;
                } else {
                    float t0, t1;
                    naive_step(p, e, t0, t1);
                    nmax[2 * p] = fmaxf(nmax[2 * p], fabsf(t0));
                    nmax[2 * p + 1] = fmaxf(nmax[2 * p + 1], fabsf(t1));
                }
            }
        }
    }

    // Two consecutive shards a, b (a of rank 0 if `first`).  Elements are
    // independent, so each pair takes a then b before the next pair.
    __device__ __forceinline__ void add2(const uint4 &ca, float sa, const uint4 &cb, float sb,
                                         bool first) {
        const uint64_t sa2 = f32x2(sa, sa), sb2 = f32x2(sb, sb);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            uint32_t ha, hb;
            uint64_t ea, eb;
            decode_add(ca, sa2, p, ha, ea);
            decode_add(cb, sb2, p, hb, eb);
            if constexpr (NAIVE) {
                if (first) {
                    nvh[p] = ha;
                    float t0, t1;
                    naive_step(p, eb, t0, t1);
                    nmax[2 * p] = fmaxf(nmax[2 * p], fabsf(t0));
                    nmax[2 * p + 1] = fmaxf(nmax[2 * p + 1], fabsf(t1));
                } else {
                    float a0, a1, b0, b1;
                    naive_step(p, ea, a0, a1);
                    naive_step(p, eb, b0, b1);
                    nmax[2 * p] = max3_abs(nmax[2 * p], a0, b0);
                    nmax[2 * p + 1] = max3_abs(nmax[2 * p + 1], a1, b1);
                }
            }
        }
    }

    // All W shards are in: requantize with a fresh block scale (the block's 8
    // lanes are an aligned octet of the warp, all of which call this), store
    // the lane's 16 codes and, from the octet's first lane, the scale; count
    // the lane's overflowed naive sums.  Every lane of the warp must call it.
    __device__ __forceinline__ void finish(bool valid, uint4 *out16, float *out_scale, bool first,
                                           unsigned long long &overflowed) {
        float t[16];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            t[2 * p] = lo_f32(acc[p]);
            t[2 * p + 1] = hi_f32(acc[p]);
        }
        // |max| of the 16 sums as a tree of three-input maxima
        float m[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) m[i] = max3_abs(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
        float am = max3_abs(max3_abs(m[0], m[1], m[2]), max3_abs(m[3], m[4], t[15]), 0.0f);
        am = octet_max(am);
        const float snew = __fdiv_rn(am, kE4M3Max);
        const uint2 lo = e4m3_codes8(t, snew);
        const uint2 hi = e4m3_codes8(t + 8, snew);
        if (valid) {
            *out16 = make_uint4(lo.x, lo.y, hi.x, hi.y);
            if (first) *out_scale = snew;
            if constexpr (NAIVE) {
                int k = 0;
#pragma unroll
                for (int i = 0; i < 16; ++i) k += nmax[i] > kE4M3Max;
                overflowed += (unsigned long long)k;
            }
        }
    }
};

// Shards c[0..k-1] of a group whose first shard has rank r0, two at a time.
template <bool NAIVE, int KMAX>
__device__ __forceinline__ void add_group(ReduceLane<NAIVE> &st, const uint4 (&c)[KMAX],
                                          const float (&sc)[KMAX], int k, int r0) {
#pragma unroll
    for (int j = 0; j < KMAX; j += 2) {
        if (j + 1 < k) st.add2(c[j], sc[j], c[j + 1], sc[j + 1], r0 + j == 0);
        else if (j < k) st.add(c[j], sc[j], r0 + j == 0);
    }
}

// Sum of the warp's overflow counts, added to *naive_count by lane 0.
__device__ __forceinline__ void flush_count(unsigned long long overflowed,
                                            unsigned long long *naive_count) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) overflowed += __shfl_xor_sync(kFull, overflowed, o);
    if ((threadIdx.x & 31) == 0 && overflowed) atomicAdd(naive_count, overflowed);
}

// ---- the register-staged reduce ---------------------------------------------
// Used when the scale rows are not 16-byte aligned or n/128 is not a multiple
// of 4.  Block indices are 32-bit (the launcher splits larger inputs); shard r
// of block b is at shards[r * shard_vec + 8 b ...] and its scale at
// shard_scales[r * scale_stride + b].  Each warp keeps the loads of its next
// (block group, chunk of RUNROLL shards) in flight while it accumulates the
// current chunk.
template <bool NAIVE, int RUNROLL>
__global__ void __launch_bounds__(kThreads, 2)
reduce_shards_kernel(
    const uint4 *__restrict__ shards, const float *__restrict__ shard_scales, int W,
    int64_t shard_vec, int64_t scale_stride, int nblocks, uint4 *__restrict__ out,
    float *__restrict__ out_scales, unsigned long long *__restrict__ naive_count) {
    pdl_wait_and_release();
    const int lane = threadIdx.x & 31;
    const int oct = lane >> 3, t8 = lane & 7;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    const int stride = nwarps * 4;
    const int nchunk = (W + RUNROLL - 1) / RUNROLL;
    // Codes and scales of shards ch*RUNROLL .. +RUNROLL-1 for the octet's block
    // of the group at b0 (clamped in range; the results of idle lanes are dropped).
    auto load = [&](int b0, int ch, uint4 (&c)[RUNROLL], float (&sc)[RUNROLL]) {
        const int blk = b0 + oct;
        const int blk_c = blk < nblocks ? blk : nblocks - 1;
        const uint4 *p = shards + (size_t)(unsigned)blk_c * 8 + t8;
        const float *q = shard_scales + blk_c;
#pragma unroll
        for (int u = 0; u < RUNROLL; ++u) {
            const int r = ch * RUNROLL + u < W ? ch * RUNROLL + u : W - 1;
            c[u] = ld_stream(p + (int64_t)r * shard_vec);
            sc[u] = __ldg(q + (int64_t)r * scale_stride);
        }
    };
    unsigned long long overflowed = 0;
    int base = warp * 4;
    if (base < nblocks) {
        uint4 cn[RUNROLL];
        float sn[RUNROLL];
        load(base, 0, cn, sn);
        int ch = 0;
        ReduceLane<NAIVE> st;
        st.clear();
        for (;;) {
            uint4 c[RUNROLL];
            float sc[RUNROLL];
#pragma unroll
            for (int u = 0; u < RUNROLL; ++u) {
                c[u] = cn[u];
                sc[u] = sn[u];
            }
            int nbase = base;
            int nch = ch + 1;
            if (nch == nchunk) {
                nch = 0;
                nbase = base + stride;
            }
            if (nbase < nblocks) load(nbase, nch, cn, sn);
            const int k = W - ch * RUNROLL < RUNROLL ? W - ch * RUNROLL : RUNROLL;
            add_group<NAIVE, RUNROLL>(st, c, sc, k, ch * RUNROLL);
            if (nch == 0) {
                // all W shards of the block group are in: requantize and store
                const int blk = base + oct;
                st.finish(blk < nblocks, out + (size_t)(unsigned)blk * 8 + t8, out_scales + blk,
                          t8 == 0, overflowed);
                st.clear();
            }
            if (nbase >= nblocks) break;
            base = nbase;
            ch = nch;
        }
    }
    if constexpr (NAIVE) flush_count(overflowed, naive_count);
}

// ---- the staged reduce ------------------------------------------------------
// A CTA is kStWarps consumer warps and one producer warp (16 + 1 without the
// naive count; 15 + 1 with it, so that the CTA is 16 warps and a thread may
// hold 128 registers).  Work is cut into tiles of kStTile blocks (a consumer
// warp owns 4 blocks of a tile, laid out as in reduce_shards_kernel); the CTAs
// take tiles round-robin.  The producer walks (tile, group of kStShards shards)
// items in the order the consumers take them and copies each shard's codes
// (kStTile * 128 bytes) and scales (kStTile * 4 bytes) with cp.async.bulk into
// the next free stage of a kStStages-deep ring (one barrier wait per group of
// shards): full[s] completes when both copies have landed, empty[s] when every
// consumer warp has read the stage.  Every wait is time-limited: on expiry the
// wait records a timeout in g_reduce_status and raises the CTA's abort flag,
// the warps stop, and the producer waits (time-limited) for its copies still
// in flight before the CTA exits.
constexpr int kStStages = 2;
constexpr int kStShards = 8;          // shards per stage
template <bool NAIVE>
struct StagedShape {
    static constexpr int kWarps = NAIVE ? 15 : 16;
    static constexpr int kThreads = (kWarps + 1) * 32;
    static constexpr int kTile = 4 * kWarps;
    static constexpr int kCodeBytes = kStShards * kTile * 128;
    static constexpr int kScaleBytes = kStShards * kTile * 4;
    static constexpr size_t kSmem = (size_t)kStStages * (kCodeBytes + kScaleBytes + 16);
    static_assert((kTile * 4) % 16 == 0, "a full tile's scales must be whole 16-byte units");
};

__device__ unsigned g_reduce_status;

// Bulk copy of `bytes` (a multiple of 16) from global `src` to shared `dst`
// (both 16-byte aligned), completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(gemm::smem_u32(dst)), "l"(src), "r"(bytes), "r"(gemm::smem_u32(bar))
        : "memory");
}

// shards: byte base; shard r of block b at shards + r * shard_bytes + 128 b.
// Requires shard_scales 16-byte aligned, scale_stride and nblocks multiples of
// 4 (so every scale copy is whole 16-byte units).
template <bool NAIVE>
__global__ void __launch_bounds__(StagedShape<NAIVE>::kThreads, 1)
reduce_shards_staged_kernel(
    const uint8_t *__restrict__ shards, const float *__restrict__ shard_scales, int W,
    int64_t shard_bytes, int64_t scale_stride, int nblocks, uint4 *__restrict__ out,
    float *__restrict__ out_scales, unsigned long long *__restrict__ naive_count) {
    using namespace gemm;
    using Sh = StagedShape<NAIVE>;
    constexpr int kStWarps = Sh::kWarps, kStTile = Sh::kTile;
    constexpr int kStCodeBytes = Sh::kCodeBytes, kStScaleBytes = Sh::kScaleBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *codes = smem;
    float *scl = reinterpret_cast<float *>(smem + (size_t)kStStages * kStCodeBytes);
    uint64_t *full =
        reinterpret_cast<uint64_t *>(smem + (size_t)kStStages * (kStCodeBytes + kStScaleBytes));
    uint64_t *empty = full + kStStages;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kStWarps);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_wait_and_release();
    volatile int *abort = &abort_flag;
    const int ntiles = (nblocks + kStTile - 1) / kStTile;

    if (warp == kStWarps) {
        // producer: one lane issues every copy
        if (lane == 0) {
            uint32_t issued = 0;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
                const int b0 = tile * kStTile;
                const int nb = nblocks - b0 < kStTile ? nblocks - b0 : kStTile;
                const uint8_t *src_c = shards + (int64_t)b0 * 128;
                const float *src_s = shard_scales + b0;
                for (int r0 = 0; r0 < W; r0 += kStShards) {
                    const int k = W - r0 < kStShards ? W - r0 : kStShards;
                    if (issued >= (uint32_t)kStStages &&
                        !wait_bar(&empty[stage], phase ^ 1u, abort, &g_reduce_status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&full[stage], (uint32_t)(k * nb) * (128u + 4u));
                    for (int j = 0; j < k; ++j) {
                        bulk_g2s(codes + (size_t)stage * kStCodeBytes + (size_t)j * kStTile * 128,
                                 src_c + (int64_t)(r0 + j) * shard_bytes, (uint32_t)nb * 128u,
                                 &full[stage]);
                        bulk_g2s(scl + ((size_t)stage * kStShards + j) * kStTile,
                                 src_s + (int64_t)(r0 + j) * scale_stride, (uint32_t)nb * 4u,
                                 &full[stage]);
                    }
                    ++issued;
                    if (++stage == kStStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // copies still in flight land before the CTA may exit
            const uint32_t first = issued > (uint32_t)kStStages ? issued - kStStages : 0u;
            for (uint32_t j = first; j < issued; ++j)
                wait_bar(&full[j % kStStages], (j / kStStages) & 1u, abort, &g_reduce_status, true);
        }
        return;
    }

    // consumers
    const int oct = lane >> 3, t8 = lane & 7;
    const int lb = warp * 4 + oct;   // the lane's block within a tile
    int stage = 0;
    uint32_t phase = 0;
    unsigned long long overflowed = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
        const int blk = tile * kStTile + lb;
        ReduceLane<NAIVE> st;
        st.clear();
        for (int r0 = 0; r0 < W; r0 += kStShards) {
            const int k = W - r0 < kStShards ? W - r0 : kStShards;
            if (!warp_wait(&full[stage], phase, abort, &g_reduce_status)) {
                ok = false;
                break;
            }
            mbar_try_wait(&full[stage], phase, 0);   // each lane observes the completed phase
            const uint8_t *cs = codes + (size_t)stage * kStCodeBytes + (size_t)(warp * 32 + lane) * 16;
            const float *ss = scl + (size_t)stage * kStShards * kStTile + lb;
            auto ld = [&](int j) { return *reinterpret_cast<const uint4 *>(cs + (size_t)j * kStTile * 128); };
            // Shards are read from the stage two at a time, the next pair's
            // loads issued before the current pair is added; the stage is
            // released once its last loads are issued (the arrive orders them).
            if (k == kStShards) {
                // a full stage: every bound and the rank-0 test are compile-time
                auto full_stage = [&](auto first_stage) {
                    constexpr bool kFirst = decltype(first_stage)::value;
                    uint4 c0 = ld(0), c1 = ld(1);
                    float s0 = ss[0], s1 = ss[kStTile];
#pragma unroll
                    for (int j = 0; j < kStShards; j += 2) {
                        uint4 n0 = c0, n1 = c1;
                        float t0 = s0, t1 = s1;
                        if (j + 2 < kStShards) {
                            n0 = ld(j + 2);
                            n1 = ld(j + 3);
                            t0 = ss[(j + 2) * kStTile];
                            t1 = ss[(j + 3) * kStTile];
                        } else {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&empty[stage]);
                        }
                        st.add2(c0, s0, c1, s1, kFirst && j == 0);
                        c0 = n0;
                        c1 = n1;
                        s0 = t0;
                        s1 = t1;
                    }
                };
                if (r0 == 0)
                    full_stage(std::true_type{});
                else
                    full_stage(std::false_type{});
            } else {
                uint4 c0 = ld(0);
                float s0 = ss[0];
                uint4 c1 = make_uint4(0u, 0u, 0u, 0u);
                float s1 = 0.0f;
                if (k > 1) {
                    c1 = ld(1);
                    s1 = ss[kStTile];
                }
#pragma unroll
                for (int j = 0; j < kStShards; j += 2) {
                    if (j >= k) break;
                    uint4 n0 = c0, n1 = c1;
                    float t0 = s0, t1 = s1;
                    if (j + 2 < k) {
                        n0 = ld(j + 2);
                        t0 = ss[(j + 2) * kStTile];
                        if (j + 3 < k) {
                            n1 = ld(j + 3);
                            t1 = ss[(j + 3) * kStTile];
                        }
                    } else {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[stage]);
                    }
                    if (j + 1 < k) st.add2(c0, s0, c1, s1, r0 + j == 0);
                    else st.add(c0, s0, r0 + j == 0);
                    c0 = n0;
                    c1 = n1;
                    s0 = t0;
                    s1 = t1;
                }
            }
            if (++stage == kStStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        st.finish(blk < nblocks, out + (size_t)(unsigned)blk * 8 + t8, out_scales + blk, t8 == 0,
                  overflowed);
    }
    if constexpr (NAIVE) flush_count(overflowed, naive_count);
}

// ---- the staged accumulation ------------------------------------------------
// A CTA is kAcWarps consumer warps and one producer warp.  Tiles of kAcTile
// blocks go round-robin to the CTAs; the producer copies each tile's BF16
// gradient, master codes and master scales with cp.async.bulk into a
// kAcStages-deep ring, and half warp h takes blocks h, h + 2 kAcWarps, ... of
// the tile (lane j: elements 8j .. 8j+7), loads them from shared memory,
// releases the stage and writes the new codes and scale straight back over the
// master (the producer never reads a tile twice, so the in-place update races
// nothing).  The arithmetic is accum_block, as in grad_accum_kernel.  Waits are
// time-limited (status in g_reduce_status, this file's pipeline status word).
constexpr int kAcWarps = 16;
constexpr int kAcThreads = (kAcWarps + 1) * 32;
constexpr int kAcRep = 3;                               // blocks per half warp per stage
constexpr int kAcTile = 2 * kAcWarps * kAcRep;
constexpr int kAcStages = 3;
constexpr int kAcGradBytes = kAcTile * 256, kAcCodeBytes = kAcTile * 128;
constexpr int kAcStageBytes = kAcGradBytes + kAcCodeBytes + kAcTile * 4;
constexpr size_t kAcSmem = (size_t)kAcStages * (kAcStageBytes + 16);
static_assert(kAcTile % 4 == 0 && kAcStageBytes % 16 == 0, "whole 16-byte copies");

template <int MID>
__global__ void __launch_bounds__(kAcThreads, 1)
grad_accum_staged_kernel(uint8_t *__restrict__ master, float *__restrict__ scales,
                         const uint8_t *__restrict__ grad, int64_t nblocks) {
    using namespace gemm;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)kAcStages * kAcStageBytes);
    uint64_t *empty = full + kAcStages;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kAcWarps);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_wait_and_release();
    volatile int *abort = &abort_flag;
    const int64_t ntiles = (nblocks + kAcTile - 1) / kAcTile;

    if (warp == kAcWarps) {
        if (lane == 0) {
            uint32_t issued = 0;
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                if (issued >= (uint32_t)kAcStages &&
                    !wait_bar(&empty[stage], phase ^ 1u, abort, &g_reduce_status))
                    break;
                const int64_t b0 = tile * kAcTile;
                const uint32_t nb = (uint32_t)(nblocks - b0 < kAcTile ? nblocks - b0 : kAcTile);
                uint8_t *st = smem + (size_t)stage * kAcStageBytes;
                mbar_expect_tx(&full[stage], nb * (256u + 128u + 4u));
                bulk_g2s(st, grad + b0 * 256, nb * 256u, &full[stage]);
                bulk_g2s(st + kAcGradBytes, master + b0 * 128, nb * 128u, &full[stage]);
                bulk_g2s(st + kAcGradBytes + kAcCodeBytes, scales + b0, nb * 4u, &full[stage]);
                ++issued;
                if (++stage == kAcStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            const uint32_t first = issued > (uint32_t)kAcStages ? issued - kAcStages : 0u;
            for (uint32_t j = first; j < issued; ++j)
                wait_bar(&full[j % kAcStages], (j / kAcStages) & 1u, abort, &g_reduce_status, true);
        }
        return;
    }

    const int half = lane >> 4, j = lane & 15, hw = 2 * warp + half;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        if (!warp_wait(&full[stage], phase, abort, &g_reduce_status)) break;
        mbar_try_wait(&full[stage], phase, 0);   // each lane observes the completed phase
        const uint8_t *st = smem + (size_t)stage * kAcStageBytes;
        uint2 mc[kAcRep];
        uint4 g[kAcRep];
        float sc[kAcRep];
#pragma unroll
        for (int r = 0; r < kAcRep; ++r) {
            const int lb = hw + 2 * kAcWarps * r;
            g[r] = reinterpret_cast<const uint4 *>(st)[lb * 16 + j];
            mc[r] = reinterpret_cast<const uint2 *>(st + kAcGradBytes)[lb * 16 + j];
            sc[r] = reinterpret_cast<const float *>(st + kAcGradBytes + kAcCodeBytes)[lb];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == kAcStages) {
            stage = 0;
            phase ^= 1u;
        }
        const int64_t b0 = tile * kAcTile;
#pragma unroll
        for (int r = 0; r < kAcRep; ++r) {
            const int64_t blk = b0 + hw + 2 * kAcWarps * r;
            float snew;
            const uint2 out = accum_block<MID>(mc[r], g[r], sc[r], snew);
            if (blk < nblocks) {
                reinterpret_cast<uint2 *>(master)[blk * 16 + j] = out;
                if (j == 0) scales[blk] = snew;
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

}  // namespace

namespace {
template <int MID>
cudaError_t launch_grad_accum_mid(void *master, float *master_scales, const void *grad, int64_t n,
                                  cudaStream_t st) {
    if ((n / kBlock) % 4 == 0 && reinterpret_cast<uintptr_t>(master_scales) % 16 == 0) {
        static bool smem_set[kMaxDevices];
        static int cache_st[kMaxDevices];
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 0 || dev >= kMaxDevices) dev = 0;
        auto ks = grad_accum_staged_kernel<MID>;
        if (!smem_set[dev]) {
            cudaError_t e =
                cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAcSmem);
            if (e != cudaSuccess) return e;
            smem_set[dev] = true;
        }
        const int64_t nbs = n / kBlock, tiles = (nbs + kAcTile - 1) / kAcTile;
        int64_t grid = (int64_t)sm_count() * resident_per_sm(ks, kAcThreads, kAcSmem, cache_st);
        if (tiles < grid) grid = tiles;
        return launch_pdl(ks, (int)(grid > 0 ? grid : 1), kAcThreads, kAcSmem, st,
                          static_cast<uint8_t *>(master), master_scales,
                          static_cast<const uint8_t *>(grad), nbs);
    }
    constexpr int kUnroll = 4;
    static int cache[kMaxDevices];
    const int64_t nb = n / kBlock;
    auto k = grad_accum_kernel<kUnroll, MID>;
    const int64_t per_cta = 2 * kUnroll * (kThreads / 32);
    return launch_pdl(k, resident_grid(k, cache, (nb + per_cta - 1) / per_cta), kThreads, 0, st,
                      static_cast<uint2 *>(master), master_scales,
                      static_cast<const uint4 *>(grad), nb);
}
}  // namespace

cudaError_t launch_grad_accum(void *master, float *master_scales, const void *grad, int64_t n,
                              int mid, cudaStream_t st) {
    switch (mid) {
        case kMidBf16: return launch_grad_accum_mid<kMidBf16>(master, master_scales, grad, n, st);
        case kMidF16: return launch_grad_accum_mid<kMidF16>(master, master_scales, grad, n, st);
        default: return launch_grad_accum_mid<kMidF32>(master, master_scales, grad, n, st);
    }
}

namespace {
// The staged reduce (the caller has zeroed naive_count); nblocks a multiple of 4.
cudaError_t launch_reduce_staged(const void *shards, const float *shard_scales, int W, int64_t n,
                                 void *out, float *out_scales, unsigned long long *naive_count,
                                 cudaStream_t st) {
    constexpr int64_t kMaxLaunchBlocks = int64_t(1) << 30;
    static bool smem_set[2][kMaxDevices];
    static int cache[2][kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    const int which = naive_count ? 1 : 0;
    auto kernel = naive_count ? reduce_shards_staged_kernel<true> : reduce_shards_staged_kernel<false>;
    const int threads = naive_count ? StagedShape<true>::kThreads : StagedShape<false>::kThreads;
    const int tile = naive_count ? StagedShape<true>::kTile : StagedShape<false>::kTile;
    const size_t smem = naive_count ? StagedShape<true>::kSmem : StagedShape<false>::kSmem;
    if (!smem_set[which][dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set[which][dev] = true;
    }
    const int per_sm = resident_per_sm(kernel, threads, smem, cache[which]);
    const int64_t nb_all = n / kBlock;
    for (int64_t b0 = 0; b0 < nb_all; b0 += kMaxLaunchBlocks) {
        const int64_t nb = nb_all - b0 < kMaxLaunchBlocks ? nb_all - b0 : kMaxLaunchBlocks;
        const int64_t tiles = (nb + tile - 1) / tile;
        int64_t grid = (int64_t)sm_count() * per_sm;
        if (tiles < grid) grid = tiles;
        const cudaError_t e = launch_pdl(
            kernel, (int)grid, threads, smem, st, static_cast<const uint8_t *>(shards) + b0 * 128,
            shard_scales + b0, W, n, nb_all, (int)nb, static_cast<uint4 *>(out) + b0 * 8,
            out_scales + b0, naive_count);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
}  // namespace

cudaError_t read_and_clear_reduce_status(unsigned *status) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_reduce_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_reduce_status, &zero, sizeof zero);
        if (e != cudaSuccess) return e;
    }
    *status = v;
    return cudaSuccess;
}

cudaError_t launch_reduce_shards(const void *shards, const float *shard_scales, int W, int64_t n,
                                 void *out, float *out_scales, unsigned long long *naive_count,
                                 cudaStream_t st) {
    constexpr int kRUnroll = 8, kRUnrollCount = 4;
    constexpr int64_t kMaxLaunchBlocks = int64_t(1) << 30;
    const int64_t nb_all = n / kBlock;
    const int64_t per_cta = 4 * (kThreads / 32);
    if (naive_count) {
        cudaError_t e = cudaMemsetAsync(naive_count, 0, sizeof(unsigned long long), st);
        if (e != cudaSuccess) return e;
    }
    if (nb_all % 4 == 0 && reinterpret_cast<uintptr_t>(shard_scales) % 16 == 0)
        return launch_reduce_staged(shards, shard_scales, W, n, out, out_scales, naive_count, st);
    static int cache_count[kMaxDevices], cache_plain[kMaxDevices];
    auto kc = reduce_shards_kernel<true, kRUnrollCount>;
    auto kp = reduce_shards_kernel<false, kRUnroll>;
    for (int64_t b0 = 0; b0 < nb_all; b0 += kMaxLaunchBlocks) {
        const int64_t nb = nb_all - b0 < kMaxLaunchBlocks ? nb_all - b0 : kMaxLaunchBlocks;
        const int64_t ctas = (nb + per_cta - 1) / per_cta;
        const uint4 *sh = static_cast<const uint4 *>(shards) + b0 * 8;
        uint4 *o = static_cast<uint4 *>(out) + b0 * 8;
        const cudaError_t e =
            naive_count
                ? launch_pdl(kc, resident_grid(kc, cache_count, ctas), kThreads, 0, st, sh,
                             shard_scales + b0, W, n / 16, nb_all, (int)nb, o, out_scales + b0,
                             naive_count)
                : launch_pdl(kp, resident_grid(kp, cache_plain, ctas), kThreads, 0, st, sh,
                             shard_scales + b0, W, n / 16, nb_all, (int)nb, o, out_scales + b0,
                             static_cast<unsigned long long *>(nullptr));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace agoq
