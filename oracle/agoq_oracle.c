/*
 * agoq_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, scalar CPU restatement of what the AGoQ element-wise
 * quantization path computes, written to be checked against the method by eye.
 * Only the tests, the smoke check and the bench's CPU-baseline leg load it;
 * the library under gradient_quantization_gb300/ never calls it and shares no
 * code, header, table or constant generator with it.
 *
 * Source of the method: "AGoQ: Activation and Gradient Quantization for
 * Memory-Efficient Distributed Training of LLMs" (gist.science summary page),
 * cited below as [AGoQ] with its section:
 *   §2.A  Layer-Aware Activation Quantization (LAAQ): "Strategie" (4-bit
 *         block-wise activations), "Herberekening versus Caching" (the stored
 *         4-bit input is dequantized in the backward pass), "DBCA-PP" (5, 6 or
 *         8 bits for pipeline stages with fewer in-flight batches).
 *   §2.B  QuanGrad: "Lokale accumulatie" (dequantize the FP8 master gradient,
 *         add the new micro-batch gradient, requantize to FP8) and
 *         "Precision-Preserved All-Reduce" step 2 "Lokale reduce" (dequantize
 *         the received shards to FP32, sum locally, requantize to FP8).
 *   §2.C  Kernel Fusion (dequantization fused with the adjacent GEMM).
 * The summary fixes no block size, scale format, rounding or bit layout.  This
 * implementation fixes them as: blocks of 128 consecutive elements, one FP32
 * scale per block equal to the block's absolute maximum divided by qmax, codes
 * from round-to-nearest-even of the IEEE FP32 quotient x/scale, qmax =
 * 2^(b-1)-1 for b-bit integer codes and 448 for FP8 E4M3, saturating E4M3.
 * Every floating-point step below is a single IEEE binary32 operation in
 * round-to-nearest-even; the file must be compiled with -ffp-contract=off and
 * without fast-math so that no multiply-add is fused.
 *
 * The outer loops over blocks (or rows, or sampled entries) carry OpenMP
 * pragmas.  Every iteration writes only its own outputs and the naive overflow
 * count is a sum, so the single-threaded build (pragmas ignored) and the
 * all-core build (-fopenmp) compute the same bits; a test compares them.
 *
 * Parity pins: every function here is pinned by tests under tests/ (codec
 * sweeps against library casts, exact-rational brute force, closed forms and
 * invariants).  No function in this file is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_BLOCK 128

/* ------------------------------------------------------------------------- */
/* BF16: the upper 16 bits of an IEEE binary32 (1 sign, 8 exponent, 7 fraction).
 * Decoding is exact: the 16 bits become the high half of a binary32.          */
float or_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to BF16, to nearest with ties to even: the 16 discarded
 * bits are compared with one half unit in the last kept place.  A carry out of
 * the fraction correctly bumps the exponent (and reaches infinity on
 * overflow).  NaN stays NaN (quiet bit set).                                  */
uint16_t or_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        if (u & 0x007FFFFFu)
            return (uint16_t)((u >> 16) | 0x0040u);
        return (uint16_t)(u >> 16);
    }
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* ------------------------------------------------------------------------- */
/* Rounding a binary64 value to a binary floating-point format with p significand
 * bits (the leading one included), smallest normal exponent emin and largest
 * exponent emax: to nearest, ties to even, with gradual underflow below 2^emin;
 * a result beyond the largest finite value 2^emax * (2 - 2^(1-p)) becomes
 * infinity (so the midpoint above it, a tie, goes to infinity as IEEE 754
 * rounds it).  The value is scaled by its quantum (a power of two, exact),
 * rounded to an integer with nearbyint in the default rounding mode (ties to
 * even) and scaled back (exact).  BF16: p = 8, emin = -126, emax = 127;
 * FP16 (IEEE binary16): p = 11, emin = -14, emax = 15.                         */
double or_round_format(double v, int p, int emin, int emax)
{
    if (v == 0.0 || isnan(v) || isinf(v))
        return v;
    int e;
    frexp(fabs(v), &e); /* |v| in [2^(e-1), 2^e) */
    int lead = e - 1;
    if (lead < emin)
        lead = emin;
    double quantum = ldexp(1.0, lead - (p - 1));
    double out = nearbyint(v / quantum) * quantum;
    double maxf = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(out) > maxf)
        return copysign(INFINITY, v);
    return out;
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 in its "FN" form (OCP 8-bit floating point): 1 sign bit, 4 exponent
 * bits with bias 7, 3 fraction bits; exponent field 0 is subnormal with value
 * m * 2^-9; S.1111.111 is NaN; there is no infinity; the largest finite
 * magnitude is 0x7E = 1.75 * 2^8 = 448.                                       */
static double or_e4m3_magnitude(unsigned code7)
{
    unsigned e = (code7 >> 3) & 15u, m = code7 & 7u;
    if (e == 0)
        return ldexp((double)m, -9);
    return ldexp(1.0 + (double)m / 8.0, (int)e - 7);
}

float or_e4m3_to_f32(uint8_t c)
{
    if ((c & 0x7Fu) == 0x7Fu)
        return NAN;
    double mag = or_e4m3_magnitude(c & 0x7Fu);
    return (float)((c & 0x80u) ? -mag : mag); /* exact: at most 4 significant bits */
}

/* Round a finite binary32 to E4M3 to nearest, ties to even, saturating: any
 * magnitude above 448 becomes 448.  The two neighbouring representable
 * magnitudes are found by bisection over the 127 finite non-negative codes
 * (their values increase with the code), and the nearer one wins; on an exact
 * tie the code with a zero last fraction bit (an even code) wins.  The sign bit
 * is kept, so a negative value that rounds to zero gives 0x80.                 */
uint8_t or_f32_to_e4m3(float v)
{
    uint8_t sign = signbit(v) ? 0x80u : 0x00u;
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7Eu);
    unsigned lo = 0, hi = 0x7Eu; /* invariant: mag(lo) <= a < mag(hi) */
    while (hi - lo > 1) {
        unsigned mid = (lo + hi) / 2;
        if (or_e4m3_magnitude(mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - or_e4m3_magnitude(lo); /* exact in binary64 */
    double dhi = or_e4m3_magnitude(hi) - a;
    unsigned pick;
    if (dlo < dhi)
        pick = lo;
    else if (dhi < dlo)
        pick = hi;
    else
        pick = (lo & 1u) ? hi : lo;
    return (uint8_t)(sign | pick);
}

/* ------------------------------------------------------------------------- */
/* Signed b-bit codes in a dense little-endian bit stream.  Within a block
 * record of 16*b bytes, element j occupies bits [j*b, j*b+b); bit k of the
 * record is bit (k mod 8) of byte floor(k/8).  The field holds the code in
 * two's complement.  For b=4 this is "two codes per byte, low nibble first";
 * for b=8 it is one int8 per byte.                                            */
static void or_put_field(uint8_t *rec, int j, int bits, int32_t code)
{
    uint32_t field = (uint32_t)code & ((1u << bits) - 1u);
    for (int k = 0; k < bits; ++k) {
        int pos = j * bits + k;
        if ((field >> k) & 1u)
            rec[pos / 8] |= (uint8_t)(1u << (pos % 8));
    }
}

static int32_t or_get_field(const uint8_t *rec, int j, int bits)
{
    uint32_t field = 0;
    for (int k = 0; k < bits; ++k) {
        int pos = j * bits + k;
        field |= (uint32_t)((rec[pos / 8] >> (pos % 8)) & 1u) << k;
    }
    if (field & (1u << (bits - 1))) /* negative in two's complement */
        return (int32_t)field - (int32_t)(1u << bits);
    return (int32_t)field;
}

static int or_bits_ok(int bits)
{
    return bits == 4 || bits == 5 || bits == 6 || bits == 8;
}

/* Return codes of the oracle entry points. */
#define OR_OK 0
#define OR_BAD_ARG 1

/* LAAQ block-wise activation quantization, [AGoQ] §2.A "Strategie" (4 bits)
 * and "DBCA-PP" (5, 6, 8 bits).  Per block of 128 elements:
 *   absmax = max |x_i|                        (exact)
 *   s      = fl(absmax / qmax)                (binary32 division)
 *   c_i    = clamp(rne_int(fl(x_i / s)), -qmax, qmax)
 * An all-zero block stores s = +0 and all-zero codes (no 0/0).
 * Output: codes, 16*bits bytes per block (dense bit stream), scales[n/128].  */
int or_quant_act(const uint16_t *x, int64_t n, int bits, uint8_t *codes, float *scales)
{
    if (!or_bits_ok(bits) || n < 0 || n % OR_BLOCK)
        return OR_BAD_ARG;
    const int32_t qmax = (1 << (bits - 1)) - 1;
    const int64_t rec_bytes = 16 * (int64_t)bits;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n / OR_BLOCK; ++b) {
        const uint16_t *xb = x + b * OR_BLOCK;
        uint8_t *rec = codes + b * rec_bytes;
        float absmax = 0.0f;
        for (int i = 0; i < OR_BLOCK; ++i) {
            float v = fabsf(or_bf16_to_f32(xb[i]));
            if (v > absmax)
                absmax = v;
        }
        float s = absmax / (float)qmax;
        scales[b] = s; /* +0 when absmax is 0 */
        memset(rec, 0, (size_t)rec_bytes);
        for (int i = 0; i < OR_BLOCK; ++i) {
            int32_t c = 0;
            if (absmax != 0.0f) {
                float q = or_bf16_to_f32(xb[i]) / s;
                float r = rintf(q); /* ties to even in the default rounding mode */
                if (r > (float)qmax)
                    r = (float)qmax;
                if (r < -(float)qmax)
                    r = -(float)qmax;
                c = (int32_t)r;
            }
            or_put_field(rec, i, bits, c);
        }
    }
    return OR_OK;
}

/* LAAQ dequantization, [AGoQ] §2.A "Herberekening versus Caching": the
 * backward pass reads the stored low-bit input back.  y_i = bf16_rne(fl(c_i*s)). */
int or_dequant_act(const uint8_t *codes, const float *scales, int64_t n, int bits, uint16_t *y)
{
    if (!or_bits_ok(bits) || n < 0 || n % OR_BLOCK)
        return OR_BAD_ARG;
    const int64_t rec_bytes = 16 * (int64_t)bits;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n / OR_BLOCK; ++b) {
        const uint8_t *rec = codes + b * rec_bytes;
        float s = scales[b];
        for (int i = 0; i < OR_BLOCK; ++i) {
            float prod = (float)or_get_field(rec, i, bits) * s;
            y[b * OR_BLOCK + i] = or_f32_to_bf16(prod);
        }
    }
    return OR_OK;
}

/* Backward of SiLU recomputed from the stored low-bit input, [AGoQ] §2.A
 * "Herberekening versus Caching": only the quantized input x is kept; the
 * backward pass dequantizes it and recomputes what it needs.  With
 * xh = bf16(fl(c * s)) (exactly or_dequant_act), sigma = 1 / (1 + exp(-xh)):
 *   silu(xh)  = xh * sigma                          -> y[i]  (binary64)
 *   silu'(xh) = sigma * (1 + xh * (1 - sigma))      (the derivative of x * sigma(x))
 *   dx[i]     = dy[i] * silu'(xh)                   -> dx[i] (binary64)
 * in binary64 throughout: the reference values the GPU's rounded BF16
 * outputs are measured against.  y may be NULL.                              */
int or_silu_backward(const uint8_t *codes, const float *scales, const uint16_t *dy, int64_t n,
                     int bits, double *dx, double *y)
{
    if (!or_bits_ok(bits) || n < 0 || n % OR_BLOCK)
        return OR_BAD_ARG;
    const int64_t rec_bytes = 16 * (int64_t)bits;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n / OR_BLOCK; ++b) {
        const uint8_t *rec = codes + b * rec_bytes;
        float s = scales[b];
        for (int i = 0; i < OR_BLOCK; ++i) {
            const int64_t k = b * OR_BLOCK + i;
            double xh = (double)or_bf16_to_f32(or_f32_to_bf16((float)or_get_field(rec, i, bits) * s));
            double sigma = 1.0 / (1.0 + exp(-xh));
            dx[k] = (double)or_bf16_to_f32(dy[k]) * (sigma * (1.0 + xh * (1.0 - sigma)));
            if (y)
                y[k] = xh * sigma;
        }
    }
    return OR_OK;
}

/* Backward of RMSNorm recomputed from the stored low-bit input, [AGoQ] §2.A
 * "Herberekening versus Caching".  The forward pass normalises each row t of
 * the [T][H] input as  y[t][i] = x[t][i] * r_t * w[i],  r_t = 1 / sqrt(mean_i
 * x[t][i]^2 + eps)  and keeps only the quantized x; the backward pass uses
 * xh = or_dequant_act of the codes (row t = blocks t*H/128 ..) and, with
 * g[i] = dy[t][i] * w[i]:
 *   rstd[t]  = r_t
 *   dx[t][i] = r_t * g[i] - xh[t][i] * r_t^3 * (sum_j g[j] * xh[t][j]) / H
 *   dw[i]    = sum_t dy[t][i] * xh[t][i] * r_t
 * all in binary64 (the exact derivatives of y with respect to x and w).
 * dy and w are BF16.  H must be a multiple of 128.                            */
int or_rmsnorm_backward(const uint8_t *codes, const float *scales, const uint16_t *dy,
                        const uint16_t *w, int64_t T, int64_t H, int bits, double eps, double *dx,
                        double *rstd, double *dw)
{
    if (!or_bits_ok(bits) || T < 0 || H <= 0 || H % OR_BLOCK)
        return OR_BAD_ARG;
    uint16_t *xrow = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)H);
    if (!xrow)
        return OR_BAD_ARG;
    const int64_t rec_bytes = 16 * (int64_t)bits, per_row = H / OR_BLOCK;
    for (int64_t i = 0; i < H; ++i)
        dw[i] = 0.0;
    for (int64_t t = 0; t < T; ++t) {
        or_dequant_act(codes + t * per_row * rec_bytes, scales + t * per_row, H, bits, xrow);
        double sxx = 0.0, sgx = 0.0;
        for (int64_t i = 0; i < H; ++i) {
            double x = or_bf16_to_f32(xrow[i]);
            double g = (double)or_bf16_to_f32(dy[t * H + i]) * or_bf16_to_f32(w[i]);
            sxx += x * x;
            sgx += g * x;
        }
        double r = 1.0 / sqrt(sxx / (double)H + eps);
        rstd[t] = r;
        for (int64_t i = 0; i < H; ++i) {
            double x = or_bf16_to_f32(xrow[i]);
            double d = or_bf16_to_f32(dy[t * H + i]);
            double g = d * or_bf16_to_f32(w[i]);
            dx[t * H + i] = r * g - x * r * r * r * sgx / (double)H;
            dw[i] += d * x * r;
        }
    }
    free(xrow);
    return OR_OK;
}

/* Requantize 128 binary32 values to E4M3 with a fresh block scale:
 * s' = fl(absmax / 448); c_i = e4m3_rne_satfinite(fl(t_i / s')).
 * An all-zero block (absmax 0, whatever the signs) stores s' = +0, codes 0x00. */
static void or_requant_block(const float *t, uint8_t *out_codes, float *out_scale)
{
    float absmax = 0.0f;
    for (int i = 0; i < OR_BLOCK; ++i) {
        float v = fabsf(t[i]);
        if (v > absmax)
            absmax = v;
    }
    float s = absmax / 448.0f;
    *out_scale = s;
    for (int i = 0; i < OR_BLOCK; ++i)
        out_codes[i] = (absmax == 0.0f) ? (uint8_t)0x00u : or_f32_to_e4m3(t[i] / s);
}

/* QuanGrad local accumulation, [AGoQ] §2.B "Lokale accumulatie", in place on
 * the FP8 master gradient.  Per block:
 *   m_i = fl(e4m3(c_i) * s)       t_i = fl(m_i + bf16(g_i))
 *   then requantize t with a fresh block scale (or_requant_block).
 * The summary names FP16/BF16 for the dequantized master; this implementation
 * keeps the intermediate in binary32, which holds every FP16/BF16 value.      */
int or_grad_accum_fp8(uint8_t *master, float *master_scales, const uint16_t *grad, int64_t n)
{
    if (n < 0 || n % OR_BLOCK)
        return OR_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n / OR_BLOCK; ++b) {
        float t[OR_BLOCK];
        uint8_t *cb = master + b * OR_BLOCK;
        float s = master_scales[b];
        for (int i = 0; i < OR_BLOCK; ++i) {
            float m = or_e4m3_to_f32(cb[i]) * s;
            t[i] = m + or_bf16_to_f32(grad[b * OR_BLOCK + i]);
        }
        or_requant_block(t, cb, &master_scales[b]);
    }
    return OR_OK;
}

/* QuanGrad local accumulation with the intermediate held in BF16 or FP16, as
 * the summary states it ([AGoQ] §2.B "Lokale accumulatie": the FP8 master is
 * dequantized to FP16/BF16, the new local gradient is added, the sum is
 * quantized back to FP8).  With R the rounding to the intermediate format
 * (mid = 1: BF16, mid = 2: FP16; or_round_format), per element:
 *   m = R(fl(e4m3(c_i) * s))      the dequantized master (binary32 product, then R)
 *   g = R(bf16(g_i))              the BF16 gradient in the intermediate format
 *   t = R(m + g)                  the sum, rounded once
 * then or_requant_block on t.  m and g have at most 11 significant bits, so
 * their binary64 sum is exact unless the smaller is below 2^-42 of the larger,
 * where it cannot move the rounding to the format; R of the binary64 sum is
 * therefore R of the exact sum.  In FP16 the intermediate overflows to
 * infinity beyond 65504 (a precondition of that format, not checked).          */
int or_grad_accum_fp8_mid(uint8_t *master, float *master_scales, const uint16_t *grad, int64_t n,
                          int mid)
{
    if (n < 0 || n % OR_BLOCK || (mid != 1 && mid != 2))
        return OR_BAD_ARG;
    const int p = mid == 1 ? 8 : 11, emin = mid == 1 ? -126 : -14, emax = mid == 1 ? 127 : 15;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n / OR_BLOCK; ++b) {
        float t[OR_BLOCK];
        uint8_t *cb = master + b * OR_BLOCK;
        float s = master_scales[b];
        for (int i = 0; i < OR_BLOCK; ++i) {
            float m32 = or_e4m3_to_f32(cb[i]) * s;
            double m = or_round_format((double)m32, p, emin, emax);
            double g = or_round_format((double)or_bf16_to_f32(grad[b * OR_BLOCK + i]), p, emin, emax);
            t[i] = (float)or_round_format(m + g, p, emin, emax); /* exact in binary32 */
        }
        or_requant_block(t, cb, &master_scales[b]);
    }
    return OR_OK;
}

/* Local reduce of the precision-preserved all-reduce, [AGoQ] §2.B
 * "Precision-Preserved All-Reduce" step 2 ("Lokale reduce"), with the W
 * received shards laid out shard-major: shard r's codes at shards[r*n ...],
 * its scales at shard_scales[r*(n/128) ...].  Per element:
 *   acc = +0;  for r = 0 .. W-1:  acc = fl(acc + fl(e4m3(c_r) * s_r))
 * then requantize acc per block (or_requant_block).
 *
 * naive_overflow (may be NULL) receives the number of elements for which the
 * naive FP8 all-reduce the page contrasts with overflows: the FP8 values are
 * summed directly in rank order in the FP8 domain (all shards share one scale),
 * acc = e4m3(c_0); for r = 1 .. W-1: t = acc + e4m3(c_r) (exact in binary32);
 * if |t| > 448 the element has overflowed (counted once); otherwise
 * acc = e4m3(rne(t)).                                                          */
int or_reduce_fp8_shards(const uint8_t *shards, const float *shard_scales, int W, int64_t n,
                         uint8_t *out, float *out_scales, uint64_t *naive_overflow)
{
    if (W < 1 || n < 0 || n % OR_BLOCK)
        return OR_BAD_ARG;
    const int64_t nb = n / OR_BLOCK;
    uint64_t overflow = 0;
#pragma omp parallel for schedule(static) reduction(+ : overflow)
    for (int64_t b = 0; b < nb; ++b) {
        float acc[OR_BLOCK];
        for (int i = 0; i < OR_BLOCK; ++i)
            acc[i] = 0.0f;
        for (int r = 0; r < W; ++r) {
            const uint8_t *cb = shards + (int64_t)r * n + b * OR_BLOCK;
            float s = shard_scales[(int64_t)r * nb + b];
            for (int i = 0; i < OR_BLOCK; ++i) {
                float v = or_e4m3_to_f32(cb[i]) * s;
                acc[i] = acc[i] + v;
            }
        }
        or_requant_block(acc, out + b * OR_BLOCK, &out_scales[b]);
        if (naive_overflow) {
            for (int i = 0; i < OR_BLOCK; ++i) {
                float a = or_e4m3_to_f32(shards[b * OR_BLOCK + i]);
                for (int r = 1; r < W; ++r) {
                    float t = a + or_e4m3_to_f32(shards[(int64_t)r * n + b * OR_BLOCK + i]);
                    if (fabsf(t) > 448.0f) {
                        ++overflow;
                        break;
                    }
                    a = or_e4m3_to_f32(or_f32_to_e4m3(t));
                }
            }
        }
    }
    if (naive_overflow)
        *naive_overflow = overflow;
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Weight-gradient product with an INT4 LAAQ operand, [AGoQ] §2.C "Kernel
 * Fusion": dW = dY^T * Xhat, where dY is BF16 [K][M] row-major (K tokens),
 * Xhat[k][j] is exactly the LAAQ 4-bit dequantization of X (or_dequant_act on
 * row k: codes [K][N/2], scales [K][N/128]), and dW[i][j] = sum_k dY[k][i] *
 * Xhat[k][j] is accumulated in binary64 in k order.  Output dW is binary64
 * [M][N] row-major: the unrounded reference the GPU result is measured against. */
static double or_xhat(const uint8_t *xc, const float *xs, int N, int64_t k, int64_t j)
{
    const uint8_t *rec = xc + k * (int64_t)(N / 2) + (j / OR_BLOCK) * 64;
    int32_t c = or_get_field(rec, (int)(j % OR_BLOCK), 4);
    float prod = (float)c * xs[k * (N / OR_BLOCK) + j / OR_BLOCK];
    return (double)or_bf16_to_f32(or_f32_to_bf16(prod));
}

int or_wgrad_gemm_int4_f64(const uint16_t *dY, const uint8_t *xc, const float *xs, int M, int N,
                           int K, double *dW)
{
    if (M <= 0 || N <= 0 || K <= 0 || N % OR_BLOCK)
        return OR_BAD_ARG;
    double *xhat = (double *)malloc(sizeof(double) * (size_t)K * (size_t)N);
    if (!xhat)
        return OR_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j)
            xhat[k * N + j] = or_xhat(xc, xs, N, k, j);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)or_bf16_to_f32(dY[k * M + i]) * xhat[k * N + j];
            dW[i * N + j] = acc;
        }
    free(xhat);
    return OR_OK;
}

/* The same product for a list of entries (rows[e], cols[e]), one plain dot
 * product each, for checking sampled entries of a full-size result.           */
int or_wgrad_gemm_int4_f64_entries(const uint16_t *dY, const uint8_t *xc, const float *xs, int M,
                                   int N, int K, const int32_t *rows, const int32_t *cols,
                                   int64_t count, double *out)
{
    if (M <= 0 || N <= 0 || K <= 0 || N % OR_BLOCK || count < 0)
        return OR_BAD_ARG;
    for (int64_t e = 0; e < count; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N)
            return OR_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t e = 0; e < count; ++e) {
        int64_t i = rows[e], j = cols[e];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += (double)or_bf16_to_f32(dY[k * M + i]) * or_xhat(xc, xs, N, k, j);
        out[e] = acc;
    }
    return OR_OK;
}

/* QuanGrad local accumulation with a binary32 gradient, the form it takes when
 * it is fused into the epilogue of the weight-gradient product ([AGoQ] §2.B
 * "Lokale accumulatie" together with §2.C "Kernel Fusion": the new gradient is
 * the product's FP32 accumulator, never rounded to BF16).  Per block:
 *   m_i = fl(e4m3(c_i) * s)       t_i = fl(m_i + g_i)
 *   then requantize t with a fresh block scale (or_requant_block).             */
int or_grad_accum_fp8_f32(uint8_t *master, float *master_scales, const float *grad, int64_t n)
{
    if (n < 0 || n % OR_BLOCK)
        return OR_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n / OR_BLOCK; ++b) {
        float t[OR_BLOCK];
        uint8_t *cb = master + b * OR_BLOCK;
        float s = master_scales[b];
        for (int i = 0; i < OR_BLOCK; ++i) {
            float m = or_e4m3_to_f32(cb[i]) * s;
            t[i] = m + grad[b * OR_BLOCK + i];
        }
        or_requant_block(t, cb, &master_scales[b]);
    }
    return OR_OK;
}

/* The weight-gradient product with the QuanGrad accumulation as its epilogue
 * ([AGoQ] §2.B "Lokale accumulatie", §2.C "Kernel Fusion"), in place on an FP8
 * master gradient [M][N] (E4M3 codes, scales [M][N/128]):
 *   g[i][j] = fl32(sum_k dY[k][i] * Xhat[k][j])   (binary64 sum in k order,
 *             rounded once to binary32: the FP32 accumulator the product hands
 *             to the epilogue, without the GEMM's own summation error)
 *   then or_grad_accum_fp8_f32 on every 128-element block of row i.
 * `blocks` (may be NULL) restricts the work to `count` blocks of the flat
 * master, block b covering row b / (N/128), columns (b % (N/128))*128 ..+127;
 * master and master_scales then hold only those blocks, [count][128] and
 * [count].  With blocks == NULL every block is done (count is ignored).      */
int or_wgrad_accum_fp8(const uint16_t *dY, const uint8_t *xc, const float *xs, int M, int N,
                       int K, const int64_t *blocks, int64_t count, uint8_t *master,
                       float *master_scales)
{
    if (M <= 0 || N <= 0 || K <= 0 || N % OR_BLOCK || count < 0)
        return OR_BAD_ARG;
    const int64_t per_row = N / OR_BLOCK;
    if (!blocks) {
        /* every block: the full binary64 product (same k-order sums), then
         * round each entry once and accumulate */
        double *dw = (double *)malloc(sizeof(double) * (size_t)M * (size_t)N);
        float *g32 = (float *)malloc(sizeof(float) * (size_t)M * (size_t)N);
        int rc = (dw && g32) ? or_wgrad_gemm_int4_f64(dY, xc, xs, M, N, K, dw) : OR_BAD_ARG;
        if (rc == OR_OK) {
            for (int64_t e = 0; e < (int64_t)M * N; ++e)
                g32[e] = (float)dw[e];
            rc = or_grad_accum_fp8_f32(master, master_scales, g32, (int64_t)M * N);
        }
        free(dw);
        free(g32);
        return rc;
    }
    float g[OR_BLOCK];
    for (int64_t e = 0; e < count; ++e) {
        const int64_t b = blocks[e];
        if (b < 0 || b >= (int64_t)M * per_row)
            return OR_BAD_ARG;
        const int64_t i = b / per_row, j0 = (b % per_row) * OR_BLOCK;
        for (int jj = 0; jj < OR_BLOCK; ++jj) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)or_bf16_to_f32(dY[k * M + i]) * or_xhat(xc, xs, N, k, j0 + jj);
            g[jj] = (float)acc;
        }
        or_grad_accum_fp8_f32(master + e * OR_BLOCK, master_scales + e, g, OR_BLOCK);
    }
    return OR_OK;
}

/* A linear layer's forward product with the LAAQ quantization of its output
 * fused into the GEMM ([AGoQ] §2.C "Kernel Fusion" with §2.A "Strategie" /
 * "DBCA-PP": the activation kept for the backward pass is quantized where it
 * is produced).  X is BF16 [T][K], W is BF16 [N][K] (K contiguous in both):
 *   Y[t][n] = bf16(fl32(sum_k X[t][k] * W[n][k]))   (binary64 sum in k order,
 *             rounded once to binary32, then to BF16)
 *   codes, scales = or_quant_act(Y, T*N, bits)      (row t = blocks t*N/128 ..)
 * y receives Y's BF16 bit patterns [T][N].                                    */
int or_fwd_gemm_quant(const uint16_t *x, const uint16_t *w, int T, int N, int K, int bits,
                      uint16_t *y, uint8_t *codes, float *scales)
{
    if (T <= 0 || N <= 0 || K <= 0 || N % OR_BLOCK || !or_bits_ok(bits))
        return OR_BAD_ARG;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)or_bf16_to_f32(x[t * K + k]) * or_bf16_to_f32(w[n * K + k]);
            y[t * N + n] = or_f32_to_bf16((float)acc);
        }
    return or_quant_act(y, (int64_t)T * N, bits, codes, scales);
}

/* ------------------------------------------------------------------------- */
/* Array forms of the codecs, for the codec sweeps in the tests.               */
void or_f32_to_bf16_array(const float *src, uint16_t *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_f32_to_bf16(src[i]);
}

void or_f32_to_e4m3_array(const float *src, uint8_t *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_f32_to_e4m3(src[i]);
}

void or_round_format_array(const double *src, double *dst, int64_t n, int p, int emin, int emax)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_round_format(src[i], p, emin, emax);
}

void or_e4m3_to_f32_array(const uint8_t *src, float *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_e4m3_to_f32(src[i]);
}

/* Threads the loops above may use: 1 in the single-threaded build.            */
int or_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
