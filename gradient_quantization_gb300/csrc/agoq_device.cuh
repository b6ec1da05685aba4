// agoq_device.cuh -- device helpers of the AGoQ element-wise kernels (sm_103a).
//
// Number formats and rounding follow the conventions stated in include/agoq.h:
// BF16 inputs, FP32 block scales, round-to-nearest-even integer codes and
// saturating E4M3 "FN" codes, every intermediate a separately rounded binary32
// operation.  Conversions use the hardware cvt instructions (inline PTX);
// divisions use the IEEE-rounded __fdiv_rn / __frcp_rn intrinsics.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace agoq {

constexpr int kBlock = 128;          // elements per quantization block
constexpr float kE4M3Max = 448.0f;   // largest finite E4M3 magnitude

// ---- programmatic dependent launch -------------------------------------------
// Wait until the grids this one depends on have completed and their memory is
// visible, then let the next grid in the stream be scheduled (its own wait
// keeps it from touching memory before this grid completes).
__device__ __forceinline__ void pdl_wait_and_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Ask the L2 to start fetching [p, p + bytes) (p 16-byte aligned, bytes a
// multiple of 16).  A hint with no effect on results: the L2 is the point of
// coherence, so a line fetched before a preceding grid writes it is updated by
// that write.  Kernels issue it for their first inputs before
// pdl_wait_and_release, so that the fetch overlaps the preceding grid's tail.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- BF16 ------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two binary32 values to a BF16 pair (round to nearest even); `lo` in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---- packed binary32 pairs (sm_100+): two IEEE round-to-nearest operations
// per instruction, bit-identical to the scalar __fadd_rn/__fsub_rn/__fmul_rn.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t u32x2(uint32_t lo, uint32_t hi) {
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// a*b + c per lane with a single rounding (fused multiply-add).
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// max(|a|, |b|, |c|) in one instruction.
__device__ __forceinline__ float max3_abs(float a, float b, float c) {
    float d;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---- E4M3 ------------------------------------------------------------------
// Two binary32 values to two E4M3 codes, round to nearest even, saturating to
// +-448; `lo` in bits 0-7.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 codes (bits 0-7 and 8-15 of v) to binary32, exactly (every E4M3
// value is an FP16 value, and every FP16 value a binary32 value).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t v, float &lo, float &hi) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)v));
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

// E4M3 codes of 8 values t[] requantized with block scale s = fl(absmax/448):
// code_i = e4m3_rne_satfinite(fl(t_i / s)).  Returns two words of 4 codes.
//
// For a normal s the quotient is formed as q = fl(t * r), r = fl(1/s); q lies
// within 3 * 2^-24 |t/s| of the binary32 quotient (plus a negligible absolute
// term if subnormal).  The codes of fl(q * (1 - 2^-20)) and fl(q * (1 + 2^-20))
// bracket that quotient on both sides; E4M3 rounding is monotonic, so when the
// two codes agree they equal the quotient's code.  Only the values whose two
// codes disagree (a quotient at or next to an E4M3 rounding boundary) are
// recomputed with IEEE division.  Such values are not rare when t has few
// significant bits: t/s is then close to 448 times a ratio of short integers,
// and on the gradient workload about one BF16-valued sum in 200 lands within
// 2^-20 of a boundary (one binary32 sum in 2000), so a per-value fallback keeps
// most lanes of a warp on the fast path.  Values whose products
// underflow are far below the smallest E4M3 midpoint (2^-10) and give a signed
// zero either way.  s subnormal takes the division; s == 0 (all-zero block)
// gives zero codes.
__device__ __forceinline__ uint2 e4m3_codes8(const float t[8], float s) {
    if (s >= 0x1p-126f) {
        const float r = __frcp_rn(s);
        constexpr float kDown = 1.0f - 0x1p-20f, kUp = 1.0f + 0x1p-20f;
        uint32_t c[2] = {0u, 0u}, d[2] = {0u, 0u};   // codes; nonzero byte: bracket differs
        // the same products in packed pairs (multiplies only: nothing to contract)
        const uint64_t r2 = f32x2(r, r), dn2 = f32x2(kDown, kDown), up2 = f32x2(kUp, kUp);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const uint64_t q2 = mul_f32x2(f32x2(t[2 * p], t[2 * p + 1]), r2);
            const uint64_t a2 = mul_f32x2(q2, dn2), b2 = mul_f32x2(q2, up2);
            const uint32_t lo = e4m3x2_from_f32(lo_f32(a2), hi_f32(a2));
            const uint32_t hi = e4m3x2_from_f32(lo_f32(b2), hi_f32(b2));
            c[p >> 1] |= lo << (16 * (p & 1));
            d[p >> 1] |= (lo ^ hi) << (16 * (p & 1));
        }
        if (d[0] | d[1]) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int sh = 8 * (k & 3);
                if ((d[k >> 2] >> sh) & 0xFFu) {
                    const uint32_t code = e4m3x2_from_f32(__fdiv_rn(t[k], s), 0.0f);
                    c[k >> 2] = (c[k >> 2] & ~(0xFFu << sh)) | (code << sh);
                }
            }
        }
        return make_uint2(c[0], c[1]);
    }
    if (s > 0.0f) {
        uint32_t c[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            c[p] = e4m3x2_from_f32(__fdiv_rn(t[2 * p], s), __fdiv_rn(t[2 * p + 1], s));
        return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
    return make_uint2(0u, 0u);
}

// The same codes when every t is a BF16 value (and so is the block absmax that
// gave s): the binary32 quotient by Markstein's correction of the reciprocal
// product (P. Markstein, IBM J. Res. Dev. 34(1), 1990), with no bracket and no
// division.  It is formed negated, -q' = fma(rho, -r, -q) with r = fl(1/s),
// -q = fl(t * -r) and rho = fma(-q, s, t), and the codes' sign bits are
// flipped at the end (E4M3 is sign-magnitude): that is q' = fma(rho, r, q)
// for every t except a zero t, where rho is +0 and only the negated form keeps
// the sign of -0/s = -0.  For s >= 2^-96, q' = fl(t/s) for every such t: the
// library's tests run every pair of BF16 values (t, absmax), |t| <= absmax,
// signed zeros included, through it and through e4m3_codes8 and compare the
// codes.  Below 2^-96 the residual can fall into the subnormal range, so those
// blocks take e4m3_codes8.
__device__ __forceinline__ uint2 e4m3_codes8_bf16(const float t[8], float s) {
    if (!(s >= 0x1p-96f)) return e4m3_codes8(t, s);
    const float nr = -__frcp_rn(s);
    const uint64_t nr2 = f32x2(nr, nr), s2 = f32x2(s, s);
    uint32_t c[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint64_t tt = f32x2(t[2 * p], t[2 * p + 1]);
        const uint64_t nq = mul_f32x2(tt, nr2);
        const uint64_t rho = fma_f32x2(nq, s2, tt);
        const uint64_t nq1 = fma_f32x2(rho, nr2, nq);
        c[p] = e4m3x2_from_f32(lo_f32(nq1), hi_f32(nq1));
    }
    return make_uint2((c[0] | (c[1] << 16)) ^ 0x80808080u, (c[2] | (c[3] << 16)) ^ 0x80808080u);
}

// Largest |value| of the BF16 pairs in w[0..N-1], as a binary32 (exact: the
// maximum of BF16 magnitudes is a BF16 value).  max.xorsign.abs compares
// magnitudes directly; its sign bit, the XOR of the inputs', is masked once at
// the end.
template <int N>
__device__ __forceinline__ float bf16_absmax(const uint32_t *w) {
    uint32_t m = w[0];
#pragma unroll
    for (int i = 1; i < N; ++i) {
        uint32_t r;
        asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w[i]));
        m = r;
    }
    m &= 0x7FFF7FFFu;
    return fmaxf(bf16_lo(m), bf16_hi(m));
}

// fl(am / QMAX) for a BF16 magnitude am (a binary32 holding a non-negative
// BF16 value, +0 included) and QMAX in {7, 15, 31, 127}, by Markstein's
// correction of the reciprocal product (P. Markstein, IBM J. Res. Dev. 34(1),
// 1990): y = fl(1/QMAX), q = fl(am*y), rho = fma(-q, QMAX, am), result
// fma(rho, y, q).  For these divisors rho is exact and the result equals the
// IEEE quotient for every BF16 am, subnormals included (checked against exact
// rational arithmetic for all 32,640 finite magnitudes per divisor; the
// library's exhaustive quantization test checks the scales of every BF16
// absmax against IEEE division on the device).
template <int QMAX>
__device__ __forceinline__ float bf16_div_qmax(float am) {
    static_assert(QMAX == 7 || QMAX == 15 || QMAX == 31 || QMAX == 127, "checked divisors only");
    constexpr float kY = 1.0f / (float)QMAX;
    const float q = __fmul_rn(am, kY);
    const float rho = __fmaf_rn(-q, (float)QMAX, am);
    return __fmaf_rn(rho, kY, q);
}

// ---- block reductions --------------------------------------------------------
// Maximum over the 16 lanes of a half warp (lanes 0-15 or 16-31).
__device__ __forceinline__ float halfwarp_max(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Maximum over aligned groups of 8 lanes.
__device__ __forceinline__ float octet_max(float v) {
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// ---- integer codes ----------------------------------------------------------
// Adding 1.5 * 2^23 to a binary32 of magnitude below 2^22 rounds it to an
// integer (round to nearest even, the addition's own rounding) and leaves that
// integer in the low mantissa bits in two's complement: the bit pattern is
// 0x4B400000 + k.  Subtracting the constant again recovers k exactly.
constexpr float kRoundMagic = 12582912.0f;

// Integer codes of 8 values of one block: code_i = rne_int(fl(x_i / s)), clamped
// to [-qmax, qmax].  Returns each code as the bit pattern of fl(code + 1.5*2^23),
// whose low bits are the code in two's complement.
//
// For a normal scale s the quotient is formed as fl(x * r), r = fl(1/s), and
// rounded with the magic addition; only if some product lies within 2^-14 of
// a half-integer are the eight quotients recomputed with IEEE division.  Why
// the shortcut is exact: with r = (1/s)(1+e1) and fl(x*r) = x*r*(1+e2),
// |e1|,|e2| <= 2^-24, the product differs from x/s by at most 2^-23 |x/s| (plus
// 2^-150 absolute if it is subnormal), and fl(x/s) differs from x/s by at most
// 2^-24 |x/s|.  Here |x/s| <= qmax(1+2^-23) <= 128, so product and quotient
// differ by less than 3 * 2^-17 < 2^-14; away from the half-integers (the only
// points where integer rounding changes) both round to the same integer.  The
// same bound keeps every code within [-qmax, qmax] without a clamp.  A
// subnormal scale (absolute rounding error up to 2^-150) takes the division
// and an explicit clamp; an all-zero block (s = 0) gives zero codes.
template <int QMAX>
__device__ __forceinline__ void integer_codes8(const float x[8], float s, uint32_t code_bits[8]) {
    if (s >= 0x1p-126f) {
        const float r = __frcp_rn(s);
        bool near = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float q = __fmul_rn(x[i], r);
            const float t = __fadd_rn(q, kRoundMagic);
            const float k = __fsub_rn(t, kRoundMagic);
            near |= fabsf(__fsub_rn(q, k)) > 0.5f - 0x1p-14f;
            code_bits[i] = __float_as_uint(t);
        }
        if (near) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                code_bits[i] = __float_as_uint(__fadd_rn(__fdiv_rn(x[i], s), kRoundMagic));
        }
    } else if (s > 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float k = fminf(fmaxf(rintf(__fdiv_rn(x[i], s)), -(float)QMAX), (float)QMAX);
            code_bits[i] = __float_as_uint(__fadd_rn(k, kRoundMagic));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) code_bits[i] = 0u;
    }
}

// Integer codes of N values (N even) sharing the scale s: the same result as
// integer_codes8, code = clamp(rne_int(fl(x/s)), -qmax, qmax), with a cheaper
// shortcut.  With r = fl(1/s) and r+- = fl(r * (1 +- 2^-20)), each value gives
// t+- = fl(x * r+- + 1.5*2^23) by one fused multiply-add: the exact product
// plus the magic constant, rounded once, i.e. x*r+- rounded to an integer held
// in the low mantissa bits.  r+- exceed and undercut 1/s by at least 14*2^-24
// relative (two roundings of 2^-24 each), while fl(x/s) is within 2^-24 of x/s;
// so for |x/s| >= 1/4 the binary32 quotient lies strictly between x*r- and x*r+,
// and rounding (monotonic) maps it between t- and t+.  When t- == t+ for all N
// values that common integer is the code; otherwise the N quotients are formed
// with IEEE division.  Values with |x/s| < 1/4 give 0 on every route.  The code
// never exceeds qmax: |x * r+| <= qmax (1 + 2^-19) < qmax + 1/2.  Subnormal s
// takes the division and an explicit clamp; s = 0 gives zero codes.
//
// With BIAS > 0 every result is the bit pattern of fl(code + BIAS + 1.5*2^23)
// instead (see kRoundMagic): the same rounding, as BIAS is an even integer.
template <int QMAX, int N, int BIAS = 0>
__device__ __forceinline__ void integer_codes_n(const float *x, float s, uint32_t *code_bits) {
    constexpr float kMagic = kRoundMagic + (float)BIAS;
    if (s >= 0x1p-126f) {
        const float r = __frcp_rn(s);
        const float rhi = __fmaf_rn(r, 0x1p-20f, r), rlo = __fmaf_rn(r, -0x1p-20f, r);
        const uint64_t rhi2 = f32x2(rhi, rhi), rlo2 = f32x2(rlo, rlo);
        const uint64_t m2 = f32x2(kMagic, kMagic);
        uint64_t differ = 0;
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const uint64_t xx = f32x2(x[i], x[i + 1]);
            const uint64_t th = fma_f32x2(xx, rhi2, m2);
            const uint64_t tl = fma_f32x2(xx, rlo2, m2);
            differ |= th ^ tl;
            code_bits[i] = static_cast<uint32_t>(th);
            code_bits[i + 1] = static_cast<uint32_t>(th >> 32);
        }
        if (differ) {
#pragma unroll
            for (int i = 0; i < N; ++i)
                code_bits[i] = __float_as_uint(__fadd_rn(__fdiv_rn(x[i], s), kMagic));
        }
    } else if (s > 0.0f) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float k = fminf(fmaxf(rintf(__fdiv_rn(x[i], s)), -(float)QMAX), (float)QMAX);
            code_bits[i] = __float_as_uint(__fadd_rn(k, kMagic));
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) code_bits[i] = __float_as_uint(kMagic);   // code 0
    }
}

// Pack the low BITS bits of 8 words into a 64-bit little-endian chunk held as
// two 32-bit words (field i at bit i*BITS, two's complement).
//   8 bits: byte permutes gather the low bytes.
//   4 bits: byte permutes gather the even and the odd elements' low bytes, and
//           one shift and one logic op interleave their nibbles (element 2j in
//           the low nibble of byte j).
//   5, 6 bits: compile-time shifts (measured faster than integer multiply-add
//           packing on this GPU).
template <int BITS>
__device__ __forceinline__ void pack_fields8(const uint32_t w[8], uint32_t &lo, uint32_t &hi) {
    if constexpr (BITS == 8) {
        lo = __byte_perm(__byte_perm(w[0], w[1], 0x0040), __byte_perm(w[2], w[3], 0x0040), 0x5410);
        hi = __byte_perm(__byte_perm(w[4], w[5], 0x0040), __byte_perm(w[6], w[7], 0x0040), 0x5410);
    } else if constexpr (BITS == 4) {
        const uint32_t ev =
            __byte_perm(__byte_perm(w[0], w[2], 0x0040), __byte_perm(w[4], w[6], 0x0040), 0x5410);
        const uint32_t od =
            __byte_perm(__byte_perm(w[1], w[3], 0x0040), __byte_perm(w[5], w[7], 0x0040), 0x5410);
        lo = (ev & 0x0F0F0F0Fu) | ((od << 4) & 0xF0F0F0F0u);
        hi = 0u;
    } else {
        constexpr uint32_t kMask = (1u << BITS) - 1u;
        lo = 0u;
        hi = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t f = w[i] & kMask;
            const int pos = i * BITS;
            if (pos + BITS <= 32) {
                lo |= f << pos;
            } else if (pos >= 32) {
                hi |= f << (pos - 32);
            } else {
                lo |= f << pos;
                hi |= f >> (32 - pos);
            }
        }
    }
}

// Sums over the fields of an 8-field chunk of BITS-bit fields: v shifted to
// each field's position, the part landing in bits 0-31 (packed_lo) or in bits
// 32-63 (packed_hi, as a 32-bit word), modulo 2^32.
template <int BITS>
__host__ __device__ constexpr uint32_t packed_lo(uint32_t v) {
    uint32_t r = 0u;
    for (int i = 0; i < 8; ++i)
        if (i * BITS < 32) r += v << (i * BITS);
    return r;
}
template <int BITS>
__host__ __device__ constexpr uint32_t packed_hi(uint32_t v) {
    uint32_t r = 0u;
    for (int i = 0; i < 8; ++i) {
        const int pos = i * BITS;
        if (pos >= 32) r += v << (pos - 32);
        else if (pos + BITS > 32) r += v >> (32 - pos);
    }
    return r;
}

// The same chunk as pack_fields8 (BITS in {4, 5, 6}), from words t[i] that hold
// 0x4B400000 + code_i + 2^(BITS-1), as integer_codes_n and corrected_codes16
// return them with BIAS = 2^(BITS-1).  The field code + 2^(BITS-1) lies in
// [0, 2^BITS) and nothing above it differs from 0x4B400000, so the words are
// added at their shifts without masking (no field carries into the next) and
// the constant's contribution is subtracted once; flipping each field's top
// bit then turns offset binary into two's complement.  The low 22 bits of
// 0x4B400000 are zero, so the right shift of a field that straddles bit 32
// splits t into the constant's and the field's parts exactly.
// The shifted additions are written as integer multiply-adds, which the
// compiler can place on the FMA pipe (measured faster than shifts and adds).
template <int BITS>
__device__ __forceinline__ void pack_biased8(const uint32_t t[8], uint32_t &lo, uint32_t &hi) {
    constexpr uint32_t kC = 0x4B400000u;
    constexpr uint32_t kSign = 1u << (BITS - 1);
    constexpr uint32_t kCLo = packed_lo<BITS>(kC), kCHi = packed_hi<BITS>(kC);
    constexpr uint32_t kSLo = packed_lo<BITS>(kSign), kSHi = packed_hi<BITS>(kSign);
    uint32_t l = 0u - kCLo, h = 0u - kCHi;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int pos = i * BITS;
        // integer multiply-adds (power-of-two multipliers)
        if (pos < 32) asm("mad.lo.u32 %0, %1, %2, %0;" : "+r"(l) : "r"(t[i]), "r"(1u << pos));
        if (pos >= 32) asm("mad.lo.u32 %0, %1, %2, %0;" : "+r"(h) : "r"(t[i]), "r"(1u << (pos - 32)));
        else if (pos + BITS > 32) h += t[i] >> (32 - pos);
    }
    lo = l ^ kSLo;
    hi = h ^ kSHi;
}

// binary32 value of the signed BITS-bit field at bit `pos` of (hi:lo), exact:
// flipping the field's sign bit gives c + 2^(BITS-1) as an unsigned number,
// which becomes the mantissa of 2^23 + c + 2^(BITS-1); subtracting that bias
// leaves c.
template <int BITS>
__device__ __forceinline__ float field_value(uint32_t lo, uint32_t hi, int pos) {
    constexpr uint32_t kMask = (1u << BITS) - 1u;
    constexpr uint32_t kSign = 1u << (BITS - 1);
    uint32_t u;
    if (pos + BITS <= 32) {
        u = lo >> pos;
    } else if (pos >= 32) {
        u = hi >> (pos - 32);
    } else {
        u = __funnelshift_r(lo, hi, pos);
    }
    const uint32_t biased = (u & kMask) ^ (0x4B000000u | kSign);
    return __fsub_rn(__uint_as_float(biased), (float)(8388608 + kSign));
}

// ---- reading LAAQ records ----------------------------------------------------
// Chunk c (8 codes, 8*BITS bits at bit 8*BITS*c) of a block record, as (lo, hi).
template <int BITS>
__device__ __forceinline__ void load_chunk(const uint32_t *rec, int c, uint32_t &lo, uint32_t &hi) {
    if constexpr (BITS == 4) {
        lo = __ldg(rec + c);
        hi = 0u;
    } else if constexpr (BITS == 8) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(rec) + c);
        lo = w.x;
        hi = w.y;
    } else {
        const int byte = BITS * c;                          // chunk starts at this byte
        const uint32_t a = __ldg(rec + (byte >> 2));
        const uint32_t b = __ldg(rec + (byte >> 2) + 1);    // still inside the record
        const int sh = 8 * (byte & 3);
        lo = __funnelshift_r(a, b, sh);
        hi = b >> sh;
    }
}

// The 8 fields of a chunk as biased binary32 words: word i holds
// 0x4B000000 + (code_i + 2^(BITS-1)), whose value is 2^23 + code_i + 2^(BITS-1)
// (field_value's bias trick).  4- and 8-bit fields are moved into place by
// byte permutes: the sign bits of a whole word are
// flipped at once, the nibbles of 4-bit fields are first spread over the
// bytes of two words (even and odd fields), and one permute per field puts
// its byte below the constant bytes 00 00 4B.
template <int BITS>
__device__ __forceinline__ void biased_words8(uint32_t lo, uint32_t hi, uint32_t wv[8]) {
    constexpr uint32_t kHigh = 0x4B000000u;
    if constexpr (BITS == 8) {
        const uint32_t a = lo ^ 0x80808080u, b = hi ^ 0x80808080u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            wv[i] = __byte_perm(a, kHigh, 0x7650 + i);
            wv[4 + i] = __byte_perm(b, kHigh, 0x7650 + i);
        }
    } else if constexpr (BITS == 4) {
        const uint32_t a = lo ^ 0x88888888u;
        const uint32_t even = a & 0x0F0F0F0Fu, odd = (a >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            wv[2 * k] = __byte_perm(even, kHigh, 0x7650 + k);
            wv[2 * k + 1] = __byte_perm(odd, kHigh, 0x7650 + k);
        }
    } else {
        constexpr uint32_t kMask = (1u << BITS) - 1u;
        constexpr uint32_t kSign = 1u << (BITS - 1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int pos = i * BITS;
            uint32_t u;
            if (pos + BITS <= 32) u = lo >> pos;
            else if (pos >= 32) u = hi >> (pos - 32);
            else u = __funnelshift_r(lo, hi, pos);
            wv[i] = (u & kMask) ^ (kHigh | kSign);
        }
    }
}

// bf16(fl32(c_i * s)) for the 8 codes of a chunk: the biased words minus
// 2^23 + 2^(BITS-1) give the codes exactly, then one product rounding, in
// packed pairs.
template <int BITS>
__device__ __forceinline__ uint4 dequantize_chunk(uint32_t lo, uint32_t hi, float s) {
    constexpr float kK = 8388608.0f + (float)(1 << (BITS - 1));
    uint32_t wv[8];
    biased_words8<BITS>(lo, hi, wv);
    const uint64_t s2 = f32x2(s, s), k2 = f32x2(kK, kK);
    uint32_t out[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint64_t y = mul_f32x2(sub_f32x2(u32x2(wv[2 * p], wv[2 * p + 1]), k2), s2);
        out[p] = pack_bf16x2(lo_f32(y), hi_f32(y));
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Integer codes of 16 BF16 values (8 words) for a block scale s >= 2^-96:
// code = rne_int(fl(x / s)).  The binary32 quotient is formed with Markstein's
// correction of the reciprocal product (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): r = fl(1/s), q = fl(x*r), rho = fma(-q, s, x) (exact),
// q' = fma(rho, r, q); then q' + 1.5*2^23 rounds it to an integer.  For BF16
// x with |x| <= absmax and s = fl(absmax/qmax) >= 2^-96, rne_int(q') equals
// rne_int(fl(x/s)) for every x, absmax and qmax in {7, 15, 31, 127}: checked
// exhaustively against IEEE division (tests/test_gpu_laaq_exhaustive.py runs
// the same check through the library).  Below 2^-96 the residual can fall
// into the subnormal range and the correction can miss a tie, so those blocks
// take integer_codes_n.  Codes stay within +-qmax because q' = fl(x/s).
// BIAS as for integer_codes_n.
template <int BIAS = 0>
__device__ __forceinline__ void corrected_codes16(const uint32_t w[8], float s, uint32_t cb[16]) {
    constexpr float kMagic = kRoundMagic + (float)BIAS;
    const float r = __frcp_rn(s);
    const uint64_t r2 = f32x2(r, r), ns2 = f32x2(-s, -s);
    const uint64_t m2 = f32x2(kMagic, kMagic);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint64_t xx = f32x2(bf16_lo(w[i]), bf16_hi(w[i]));
        const uint64_t q = mul_f32x2(xx, r2);
        const uint64_t rho = fma_f32x2(q, ns2, xx);
        const uint64_t t = add_f32x2(fma_f32x2(rho, r2, q), m2);
        cb[2 * i] = __float_as_uint(lo_f32(t));
        cb[2 * i + 1] = __float_as_uint(hi_f32(t));
    }
}

}  // namespace agoq
