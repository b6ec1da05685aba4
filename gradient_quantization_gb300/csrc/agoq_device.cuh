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

// ---- BF16 ------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two binary32 values to a BF16 pair (round to nearest even); `lo` in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
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
// Nearest integer, ties to even, of the binary32 quotient fl(x / s), computed
// as rint(fl(x * r)) with r = fl(1/s) unless the product lies within 2^-14 of a
// half-integer, in which case the quotient is formed with an IEEE division.
//
// Why the shortcut is exact: with r = (1/s)(1+e1) and fl(x*r) = x*r*(1+e2),
// |e1|,|e2| <= 2^-24, the product differs from x/s by at most 2^-23 |x/s|
// (+ an absolute 2^-150 if it is subnormal), and fl(x/s) differs from x/s by at
// most 2^-24 |x/s|.  Quotients here satisfy |x/s| <= qmax(1+2^-23) <= 128, so
// product and quotient differ by less than 3 * 2^-17 < 2^-14.  Away from the
// half-integers (the only points where the integer rounding changes) both
// therefore round to the same integer.  Requires s normal (r finite and
// accurate); callers use the division for subnormal s.
__device__ __forceinline__ float rint_quotient(float x, float s, float r) {
    const float q = __fmul_rn(x, r);
    const float k = rintf(q);
    const float d = fabsf(__fsub_rn(q, k));     // distance to the nearest integer, <= 1/2
    if (__fsub_rn(0.5f, d) < 0x1p-14f) return rintf(__fdiv_rn(x, s));
    return k;
}

}  // namespace agoq
