/*
 * agoq.h -- C ABI of libagoq.so: the AGoQ element-wise quantization kernels
 * and the INT4-dequant-fused weight-gradient GEMM, for NVIDIA GB300 (sm_103a).
 *
 * Method: "AGoQ: Activation and Gradient Quantization for Memory-Efficient
 * Distributed Training of LLMs" (gist.science summary page), sections
 * 2.A (LAAQ, DBCA-PP), 2.B (QuanGrad: local accumulation, precision-preserved
 * all-reduce) and 2.C (kernel fusion).  The page fixes no numeric format; this
 * library fixes:
 *   - blocks of 128 consecutive elements of the flat tensor;
 *   - one FP32 scale per block = (block absmax) / qmax, rounded once (IEEE
 *     binary32 division); an all-zero block stores scale +0 and zero codes;
 *   - integer codes c = clamp(round_half_even(fl32(x / scale)), -qmax, qmax)
 *     with qmax = 2^(bits-1) - 1, stored as two's-complement bit fields in a
 *     dense little-endian stream: element j of a block occupies bits
 *     [j*bits, j*bits+bits) of the block's 16*bits-byte record, bit k being
 *     bit (k mod 8) of byte k/8 (for bits=4: two codes per byte, low nibble
 *     first; for bits=8: one int8 per byte);
 *   - FP8 codes are OCP E4M3 "FN" (bias 7, max 448, no infinity), produced by
 *     round-to-nearest-even with saturation to +-448; qmax = 448;
 *   - every intermediate is a separately rounded binary32 operation (no fused
 *     multiply-add), so results are bit-identical to a plain scalar
 *     implementation of the same steps.
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers (memory the GPU can address) owned
 *     by the caller.  The library allocates no memory and keeps no state
 *     between calls.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous and stream-ordered: they return after
 *     the launch; results are valid once the stream has been synchronised.
 *   - Arguments are validated before anything is launched.  On any error the
 *     call returns a non-zero status and touches no buffer.
 *   - n counts elements; n must be a multiple of 128 (ragged tails are not
 *     supported: AGOQ_ERR_SHAPE); n == 0 is a valid no-op.
 *   - Data pointers must be 16-byte aligned (AGOQ_ERR_ALIGN); scale arrays 4-byte.
 *   - Outputs must not overlap inputs (AGOQ_ERR_ALIAS), except where a call is
 *     documented as in place.
 *   - Inputs must be finite; NaN or infinite inputs give unspecified codes.
 */
#ifndef AGOQ_H
#define AGOQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    AGOQ_OK = 0,
    AGOQ_ERR_NULL = 1,    /* a required pointer is NULL */
    AGOQ_ERR_SHAPE = 2,   /* n not a multiple of 128, negative size, or GEMM tile rule broken */
    AGOQ_ERR_BITS = 3,    /* bits not in {4, 5, 6, 8} */
    AGOQ_ERR_ALIGN = 4,   /* pointer not aligned as required */
    AGOQ_ERR_ALIAS = 5,   /* an output overlaps an input */
    AGOQ_ERR_CUDA = 6,    /* the CUDA runtime reported an error at launch */
    AGOQ_ERR_TIMEOUT = 7, /* a pipeline wait gave up (see agoq_device_status) */
    AGOQ_ERR_FORMAT = 8   /* unsupported intermediate format (agoq_grad_accum_fp8_mid) */
} agoq_status;

/* Intermediate formats of the QuanGrad accumulation (agoq_grad_accum_fp8_mid). */
typedef enum {
    AGOQ_MID_FP32 = 0,  /* binary32 (agoq_grad_accum_fp8) */
    AGOQ_MID_BF16 = 1,
    AGOQ_MID_FP16 = 2
} agoq_mid_format;

/* Human-readable name of a status code (static string, never NULL). */
const char *agoq_status_string(agoq_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int agoq_version(void);

/*
 * LAAQ block-wise activation quantization (AGoQ section 2.A, "Strategie" for
 * 4 bits; "Dynamic Bit-width Compensation (DBCA-PP)" for 5, 6 and 8 bits).
 *   x_bf16 : in,  n BF16 values (the flattened activation, row-major).
 *   n      : number of elements, multiple of 128.
 *   bits   : 4, 5, 6 or 8.
 *   codes  : out, (n/128) * 16 * bits bytes: one packed record per block.
 *   scales : out, n/128 FP32 block scales.
 */
agoq_status agoq_quant_act(const void *x_bf16, int64_t n, int bits, void *codes, float *scales,
                           void *stream);

/*
 * LAAQ dequantization (AGoQ section 2.A, "Herberekening versus Caching": the
 * stored low-bit input is read back in the backward pass).
 *   y_i = bf16_round_nearest_even(fl32(c_i * scale)).
 *   codes, scales : in, as written by agoq_quant_act with the same n and bits.
 *   y_bf16        : out, n BF16 values.
 */
agoq_status agoq_dequant_act(const void *codes, const float *scales, int64_t n, int bits,
                             void *y_bf16, void *stream);

/*
 * SiLU backward recomputed from the stored low-bit input (AGoQ section 2.A,
 * "Herberekening versus Caching": only the quantized input is kept; the
 * backward pass dequantizes it and recomputes the intermediates).  With
 * xh_i = bf16(fl32(c_i * scale)) (exactly agoq_dequant_act), in binary32:
 *   sigma_i = 1 / (1 + exp(-xh_i));
 *   dx_i = bf16_rne(dy_i * sigma_i * (1 + xh_i * (1 - sigma_i)));   (dy * silu'(xh))
 *   y_i  = bf16_rne(xh_i * sigma_i);                                 (silu(xh), optional)
 *   codes, scales : in, as written by agoq_quant_act with the same n and bits.
 *   dy_bf16       : in, n BF16 upstream gradients (of the SiLU output).
 *   dx_bf16       : out, n BF16 gradients of the SiLU input.
 *   y_bf16        : out, n BF16 recomputed SiLU outputs, or NULL to skip them.
 * exp is the hardware base-2 exponential of xh * log2(e) (__expf), 1/(1+e) the
 * approximate division, and 1 + xh * (1 - sigma) a fused multiply-add; each
 * output is within half a BF16 ulp plus 2^-20 * |dy| * (1 + |xh|) (dx) or
 * 2^-20 * |xh| (y) of the exact value.
 * Outputs must not overlap the inputs or each other.
 */
agoq_status agoq_silu_backward(const void *codes, const float *scales, const void *dy_bf16,
                               int64_t n, int bits, void *dx_bf16, void *y_bf16, void *stream);

/*
 * RMSNorm backward recomputed from the stored low-bit input (AGoQ section 2.A,
 * "Herberekening versus Caching").  The forward pass computed, per row t of
 * the [T][H] input x, y[t][i] = x[t][i] * r_t * w[i] with r_t = 1/sqrt(mean_i
 * x[t][i]^2 + eps), and kept only agoq_quant_act(x, bits) (row t = blocks
 * t*H/128 ..).  With xh its dequantization (exactly agoq_dequant_act) and
 * g[i] = dy[t][i] * w[i], in binary32:
 *   rstd[t]  = 1 / sqrt(sum_i xh[t][i]^2 / H + eps)
 *   dx[t][i] = bf16_rne(rstd[t] * g[i] - xh[t][i] * rstd[t]^3 * (sum_j g[j] xh[t][j]) / H)
 *   dw[i]    = sum_t dy[t][i] * xh[t][i] * rstd[t]
 *   codes, scales : in, the stored input (n = T*H elements, `bits` wide).
 *   dy_bf16       : in, BF16 [T][H] upstream gradients.   w_bf16 : in, BF16 [H] weight.
 *   dx_bf16       : out, BF16 [T][H].  rstd : out, FP32 [T].
 *   dw            : out, FP32 [H] (set, not accumulated), or NULL to skip it.
 * Sums are formed in a fixed order (fused multiply-adds where that only
 * removes roundings), so results are deterministic; they differ from exact
 * values by binary32 summation error (bounded by (H + 16) * 2^-24 relative to
 * the sums of absolute terms for the row sums, (T/64 + H + 32) * 2^-24 for dw)
 * plus the output rounding.  H must be a multiple of 256 and at
 * most 8192, eps finite and >= 0 (AGOQ_ERR_SHAPE otherwise).  The input is read
 * once for dx and rstd; dw reads the codes and dy a second time.  Outputs must
 * not overlap the inputs or each other.  When T is a multiple of 32, H of 512,
 * and scales and rstd are 16-byte aligned, dw streams its rows through shared
 * memory by TMA with time-limited pipeline waits (see agoq_device_status); the
 * bound above holds either way.
 */
agoq_status agoq_rmsnorm_backward(const void *codes, const float *scales, const void *dy_bf16,
                                  const void *w_bf16, int64_t T, int64_t H, int bits, float eps,
                                  void *dx_bf16, float *rstd, float *dw, void *stream);

/*
 * Bytes of scratch agoq_rmsnorm_backward_ws needs for rows of H elements (the
 * same for every T): 304 * H * 4 for H <= 4096, 0 for larger H (which takes the
 * two-pass path of agoq_rmsnorm_backward), -1 if H is not a multiple of 256 in
 * 256 .. 8192.
 */
int64_t agoq_rmsnorm_backward_workspace_bytes(int64_t H);

/*
 * The same backward as agoq_rmsnorm_backward, with dw (required here), in ONE
 * read of the input for H <= 4096: a group of 128 threads takes a row, keeps its
 * dequantized input, dy and w in registers from the row sums through dx, and
 * adds the row's dw terms dy * xh * rstd to per-thread sums; each of the G
 * CTAs (as many as are resident at once, at most 304) writes its sums as one row
 * of the workspace, and a second small kernel adds those rows in a fixed order
 * (eight contiguous ranges, each in row order, then the range sums in order)
 * into dw.  Results are deterministic on a given GPU model; each dw sum is a
 * chain of at most ceil(T/2G) + 1 + ceil(G/8) + 8 binary32 additions, and dx
 * and rstd obey the bounds stated for agoq_rmsnorm_backward.
 *   workspace       : caller-owned device scratch, 16-byte aligned, of at least
 *                     agoq_rmsnorm_backward_workspace_bytes(H) bytes (else
 *                     AGOQ_ERR_SHAPE); contents on entry are ignored and on
 *                     return unspecified; it must not overlap any argument.
 *   workspace_bytes : its size in bytes.
 * Other arguments, rules and errors as agoq_rmsnorm_backward; dw NULL is
 * AGOQ_ERR_NULL.  For H > 4096 (workspace size 0) the call is
 * agoq_rmsnorm_backward.  Calls that share a workspace must not overlap in time
 * on the GPU.
 */
agoq_status agoq_rmsnorm_backward_ws(const void *codes, const float *scales, const void *dy_bf16,
                                     const void *w_bf16, int64_t T, int64_t H, int bits, float eps,
                                     void *dx_bf16, float *rstd, float *dw, void *workspace,
                                     int64_t workspace_bytes, void *stream);

/*
 * agoq_rmsnorm_backward_ws without the workspace argument, for callers that
 * cannot allocate device memory where they call it: a hook inside another
 * framework's allocator-free path, code running while device memory is
 * reserved or accounted by someone else, or a plain C caller with no device
 * allocator of its own.  The page has no counterpart: it is a packaging of the
 * single-read kernel above.  The scratch that workspace would hold is a
 * static array inside the library, sized for the largest rows it accepts:
 * H must be a multiple of 256 and at most 4096 (AGOQ_ERR_SHAPE beyond that;
 * about 5 MB per GPU, held from the first use of the library on that GPU until
 * the process exits).  The library allocates nothing in this call.  The first
 * call on each device looks up the array's device address (with that device
 * current), so make that first call before capturing a stream into a graph.
 * All calls on a device share the array: calls that may run at the same time
 * on the GPU (on different streams without ordering between them) race and
 * give wrong dw; order them, or use agoq_rmsnorm_backward_ws with separate
 * workspaces.  Nothing in the array needs to start at zero (every call writes
 * the part it reads).  Arguments, results and the other errors as
 * agoq_rmsnorm_backward_ws; dw NULL is AGOQ_ERR_NULL.
 */
agoq_status agoq_rmsnorm_backward_noalloc(const void *codes, const float *scales,
                                          const void *dy_bf16, const void *w_bf16, int64_t T,
                                          int64_t H, int bits, float eps, void *dx_bf16,
                                          float *rstd, float *dw, void *stream);

/*
 * QuanGrad local accumulation (AGoQ section 2.B, "Lokale accumulatie"), IN
 * PLACE on an FP8 master gradient.  Per block of 128:
 *   m_i = fl32(e4m3(c_i) * scale);  t_i = fl32(m_i + g_i);
 *   scale' = fl32(absmax(t) / 448); c_i' = e4m3_rne_satfinite(fl32(t_i / scale')).
 *   master_e4m3   : in/out, n E4M3 codes.  A zeroed buffer is a zero gradient.
 *   master_scales : in/out, n/128 FP32 scales.
 *   grad_bf16     : in, n BF16 micro-batch gradient values (must not overlap the master).
 * The page dequantizes to FP16/BF16; this library keeps the sum in FP32.
 * When master_scales is 16-byte aligned and n/128 is a multiple of 4, the
 * blocks stream through shared memory with time-limited pipeline waits (see
 * agoq_device_status; the results are the same either way).  If such a wait
 * runs out, the update stops part-way: some blocks of the master then hold the
 * new sum and others the old one, and the old values of the updated blocks are
 * gone.  A caller that must be able to recover from AGOQ_ERR_TIMEOUT keeps a
 * copy of the master (codes and scales) from before the call.
 */
agoq_status agoq_grad_accum_fp8(void *master_e4m3, float *master_scales, const void *grad_bf16,
                                int64_t n, void *stream);

/*
 * The same accumulation with the intermediate held in the format the page
 * names (AGoQ section 2.B, "Lokale accumulatie": the FP8 master gradient is
 * dequantized to FP16/BF16, the new gradient added, the sum requantized).
 * With R the rounding to nearest even to the intermediate format, per element
 *   m_i = R(fl32(e4m3(c_i) * scale));  g_i' = R(g_i);  t_i = R(m_i + g_i')
 * (the exact sum rounded once), then the requantization of
 * agoq_grad_accum_fp8.  mid_format: AGOQ_MID_FP32 (identical to
 * agoq_grad_accum_fp8), AGOQ_MID_BF16 or AGOQ_MID_FP16; anything else returns
 * AGOQ_ERR_FORMAT.  FP16 has gradual underflow below 2^-14 and overflows to
 * infinity beyond 65504: magnitudes must stay below that (not checked).
 * Other arguments and errors as agoq_grad_accum_fp8.
 */
agoq_status agoq_grad_accum_fp8_mid(void *master_e4m3, float *master_scales,
                                    const void *grad_bf16, int64_t n, int mid_format,
                                    void *stream);

/*
 * Local reduce of the precision-preserved all-reduce (AGoQ section 2.B,
 * "Precision-Preserved All-Reduce", step 2 "Lokale reduce"): the W shards an
 * all-to-all delivered, summed in FP32 in rank order and requantized to FP8.
 *   shards_e4m3  : in, W * n E4M3 codes, shard-major ([W][n]).
 *   shard_scales : in, W * (n/128) FP32 scales ([W][n/128]).
 *   W            : number of shards, >= 1.
 *   out_e4m3     : out, n codes;  out_scales : out, n/128 scales.
 *   Per element acc = +0; for r = 0..W-1: acc = fl32(acc + fl32(e4m3(c_r) * s_r));
 *   then the requantization of agoq_grad_accum_fp8.
 *   naive_overflow_count : out (device pointer to one uint64) or NULL.  When
 *     given, it is set (not accumulated) to the number of elements at which a
 *     naive FP8 all-reduce -- the W FP8 values summed directly in rank order,
 *     the running sum rounded back to E4M3 after each add -- exceeds 448.
 *     The library zeroes it on `stream` before the reduce.
 * When shard_scales is 16-byte aligned and n/128 is a multiple of 4, the
 * reduce streams the shards through shared memory with time-limited pipeline
 * waits (see agoq_device_status); the results are the same either way.
 */
agoq_status agoq_reduce_fp8_shards(const void *shards_e4m3, const float *shard_scales, int W,
                                   int64_t n, void *out_e4m3, float *out_scales,
                                   unsigned long long *naive_overflow_count, void *stream);

/*
 * Weight-gradient GEMM with the LAAQ 4-bit activation dequantized inside the
 * kernel's operand path (AGoQ section 2.C, "Kernel Fusion"):
 *   dW[M][N] = sum_k dY[k][m] * Xhat[k][n],
 *   Xhat[k][n] = bf16_rne(fl32(c[k][n] * scale[k][n/128])), exactly what
 *   agoq_dequant_act(bits=4) gives for row k;  FP32 accumulation in tensor
 *   memory, BF16 round-to-nearest-even output.
 *   dY_bf16  : in, BF16 [K][M] row-major (K tokens).
 *   x_codes  : in, [K][N/2] bytes: row k is agoq_quant_act(bits=4) of X row k.
 *   x_scales : in, FP32 [K][N/128].
 *   dW_bf16  : out, BF16 [M][N] row-major.
 *   M and N must be multiples of 128 and K of 64, all > 0 (AGOQ_ERR_SHAPE
 *   otherwise).  dY, x_codes and dW must be 16-byte aligned, x_scales 4-byte
 *   aligned (AGOQ_ERR_ALIGN).  When N is a multiple of 512 and x_scales is
 *   16-byte aligned the scales are staged by TMA with the codes; otherwise the
 *   kernel reads them directly.  A 32-byte-aligned dW (as every torch
 *   allocation is) is written with 32-byte stores, a 16-byte-aligned one with
 *   16-byte stores (slower; the same values).  Pipeline waits are
 *   time-limited: see agoq_device_status.
 */
agoq_status agoq_wgrad_gemm_int4(const void *dY_bf16, const void *x_codes, const float *x_scales,
                                 int M, int N, int K, void *dW_bf16, void *stream);

/*
 * The same GEMM with the FP32 accumulator written out unrounded
 * (dW_f32 : out, FP32 [M][N] row-major).  For verification: it isolates the
 * accumulation error from the BF16 output rounding.
 */
agoq_status agoq_wgrad_gemm_int4_f32out(const void *dY_bf16, const void *x_codes,
                                        const float *x_scales, int M, int N, int K, float *dW_f32,
                                        void *stream);

/*
 * The same product with the QuanGrad local accumulation as its epilogue (AGoQ
 * section 2.B "Lokale accumulatie" fused per section 2.C "Kernel Fusion"), IN
 * PLACE on an FP8 master gradient laid out like dW: for each 128-column block
 * of each row m (block b = m * N/128 + n/128 of the flat [M][N] master),
 *   g_i   = the FP32 accumulator of dW[m][n] (never rounded to BF16);
 *   m_i   = fl32(e4m3(c_i) * scale);  t_i = fl32(m_i + g_i);
 *   scale' = fl32(absmax(t) / 448);   c_i' = e4m3_rne_satfinite(fl32(t_i / scale')),
 * i.e. agoq_grad_accum_fp8 with the accumulator as the gradient.
 *   master_e4m3   : in/out, [M][N] E4M3 codes, 16-byte aligned (32-byte aligned:
 *                   read and written in 32-byte accesses).
 *   master_scales : in/out, [M][N/128] FP32 scales.
 * Shape rules and the other arguments as agoq_wgrad_gemm_int4; the master must
 * not overlap the operands.  The FP32 accumulation order is the tensor cores'
 * (not specified), so codes match a reference that rounds the exact product
 * once to FP32 only where that accumulation is exact.
 */
agoq_status agoq_wgrad_gemm_int4_accum_fp8(const void *dY_bf16, const void *x_codes,
                                           const float *x_scales, int M, int N, int K,
                                           void *master_e4m3, float *master_scales, void *stream);

/*
 * A linear layer's forward GEMM with the LAAQ quantization of its output fused
 * into the epilogue (AGoQ section 2.C, "Kernel Fusion", with section 2.A: the
 * activation kept for the backward pass is stored in `bits`-wide codes):
 *   Y[t][n] = bf16_rne(acc[t][n]),  acc = sum_k X[t][k] * W[n][k] accumulated
 *             in FP32 on the tensor cores (order unspecified);
 *   codes, scales = agoq_quant_act(Y, T*N, bits) (row t = blocks t*N/128 ..).
 *   x_bf16 : in, BF16 [T][K] (K contiguous).   w_bf16 : in, BF16 [N][K] (K contiguous,
 *            the torch Linear weight layout).
 *   y_bf16 : out, BF16 [T][N].   codes : out, (T*N/128) records of 16*bits bytes.
 *   scales : out, FP32 [T][N/128].
 * T must be a multiple of 128, N of 256, K of 64, all > 0 (AGOQ_ERR_SHAPE);
 * bits in {4, 5, 6, 8}; all pointers 16-byte aligned (scales 4-byte).  Outputs
 * must not overlap the operands or each other.  Pipeline waits are
 * time-limited: see agoq_device_status.
 */
agoq_status agoq_fwd_gemm_quant(const void *x_bf16, const void *w_bf16, int T, int N, int K,
                                int bits, void *y_bf16, void *codes, float *scales, void *stream);

/*
 * DBCA-PP bit-width assignment (AGoQ section 2.A, "Dynamic Bit-width
 * Compensation (DBCA-PP)": pipeline stages that hold fewer activation batches
 * get wider codes, the stages with the most batches the base width, so that
 * no stage stores more activation bytes than the fullest one).  Host-side, no
 * GPU work.  Under the one-forward-one-backward schedule, stage s (0 = first)
 * holds live_s = min(stages - s, microbatches) micro-batches of activations at
 * its peak; stage 0 holds the most.  Each stage gets the largest width b in
 * {4, 5, 6, 8}, b >= base_bits, with live_s * b <= live_0 * base_bits.
 *   bits : out, `stages` ints (the width for agoq_quant_act on that stage).
 * AGOQ_ERR_SHAPE if stages or microbatches < 1, AGOQ_ERR_BITS for a base
 * width outside {4, 5, 6, 8}.
 */
agoq_status agoq_dbca_pp_bits(int stages, int microbatches, int base_bits, int *bits);

/*
 * Synchronise `stream`, then read and clear the library's device-side status
 * words for the current device.  Returns AGOQ_ERR_TIMEOUT if a pipeline wait
 * of a GEMM (agoq_wgrad_gemm_int4*, agoq_fwd_gemm_quant), of the staged
 * shard reduce (agoq_reduce_fp8_shards), of the staged QuanGrad accumulation
 * (agoq_grad_accum_fp8, agoq_grad_accum_fp8_mid) or of the staged RMSNorm dw
 * (agoq_rmsnorm_backward) exceeded its time limit since the last call (that
 * call's output is then incomplete; for the in-place accumulations the master
 * is left partly updated),
 * AGOQ_ERR_CUDA if the synchronisation failed, else AGOQ_OK.
 */
agoq_status agoq_device_status(void *stream);

/*
 * Test-only export for the failure path: launches one thread that waits, with
 * the GEMMs' bounded mbarrier wait, for a barrier phase that never completes.
 * The wait gives up after `limit_cycles` SM clock cycles (0 < limit_cycles <=
 * 4e9, else AGOQ_ERR_SHAPE), records a timeout in the status word and the
 * kernel returns; the next agoq_device_status then reports AGOQ_ERR_TIMEOUT
 * and the CUDA context stays usable.
 */
agoq_status agoq_test_wait_timeout(int64_t limit_cycles, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* AGOQ_H */
