// wgrad_gemm_impl.cuh -- weight-gradient GEMM with the LAAQ 4-bit activation
// dequantized in the operand path ("AGoQ: Activation and Gradient Quantization
// for Memory-Efficient Distributed Training of LLMs", section 2.C "Kernel
// Fusion": the tensor cores do the GEMM while the quantization logic runs on
// the CUDA cores of the same kernel).
//
//   dW[M][N] = sum_k dY[k][m] * Xhat[k][n],  Xhat = bf16(fl32(code * scale))
//
// Blackwell design (sm_103a): one CTA per SM; the two CTAs of a cluster of
// two form a tcgen05 CTA pair that is persistent over 512 x 256 output tiles
// (256 rows per CTA, as two 128-row halves).  Per BK-deep k-block each CTA has three shared-memory rings:
//   A ring (NA stages)  its 256 dY rows x BK, four 64-wide boxes with the
//                       128-byte swizzle, loaded by TMA (rows past M read as
//                       zeros and are not multiplied);
//   X ring (NX stages)  the packed 4-bit codes of its 128 X-hat columns (BK
//                       rows x 64 bytes) and their scales, loaded by TMA;
//   B ring (NB stages)  its 128 X-hat columns (BF16), written by the
//                       dequantizers in the MN-major 128-byte-swizzled layout
//                       the MMA reads.
//   warp 0      TMA producer of the A ring.
//   warp 1      TMEM allocation for the pair; in CTA 0 one thread issues, per
//               k-block, (BK/16) x 2 pair MMAs tcgen05.mma.cta_group::2
//               kind::f16 (M=256: 128 rows from each CTA; N=256: 128 B
//               columns from each CTA; K=16; both operands MN-major, BF16 in,
//               FP32 accumulate) into two 256-column accumulators per CTA
//               (its rows of the two M-halves, all 512 TMEM columns); the
//               commits, multicast to both CTAs, free the A and B stages.
//               In CTA 1 one thread relays each landed A stage to CTA 0 with
//               a remote mbarrier arrive.
//   warp 2      TMA producer of the X ring.
//   warps 3-18  dequantizers: codes -> Xhat into the B ring, fence.proxy.async,
//               an arrive on CTA 0's B barrier (remote from CTA 1) and the
//               release of the X stage (after its codes have been consumed).
//               They also run the epilogue of the previous tile, once they
//               have written the next tile's first k-block (the MMA waits
//               for the accumulator anyway): each warp takes
//               one 32-row x 128-column item of its CTA's accumulators (its
//               TMEM lane quarter, warp % 4, and one of four 128-column
//               blocks), reads it with tcgen05.ld, one output row per thread,
//               and does one of
//               - BF16 round-to-nearest-even and global stores (the
//                 accumulator is handed back before the stores);
//               - the FP32 accumulator stored unrounded;
//               - the QuanGrad accumulation into an FP8 master gradient
//                 ("Lokale accumulatie", section 2.B): dequantize the 128
//                 E4M3 master codes of the row block, add the FP32
//                 accumulator, take the block absmax, requantize in place with
//                 the new scale.  The BF16 dW never exists.
// Every mbarrier wait has a time limit: on expiry the kernel records a code in
// g_device_status, raises a CTA-wide abort flag, lets in-flight copies and
// MMAs drain (with a limit), frees its TMEM and returns; both CTAs of a pair
// meet at a cluster barrier before either frees TMEM or exits.
#pragma once
#include <cuda.h>

#include "agoq_device.cuh"
#include "agoq_launch.h"
#include "gemm_common.cuh"

namespace agoq {
namespace AGOQ_WGRAD_NS {
namespace {

using namespace gemm;

// Device-side status word of this configuration's kernels: a pipeline wait
// that exceeds its time limit records a non-zero code here instead of
// spinning forever.
__device__ unsigned g_device_status;

// Tiling of this instance: AGOQ_GEMM_BK (k-block depth) and the ring depths
// AGOQ_GEMM_NA / NB / NX are set by the translation unit that includes this
// file (wgrad_gemm.cu: BK = 128 for K a multiple of 128; wgrad_gemm_k64.cu:
// BK = 64 for the other multiples of 64), and AGOQ_WGRAD_NS names its
// namespace.

// Epilogue kinds.
constexpr int kEpiBf16 = 0, kEpiF32 = 1, kEpiAccumFp8 = 2;

constexpr int BM = 256, BN = 256, BK = AGOQ_GEMM_BK;
constexpr int NA = AGOQ_GEMM_NA, NX = AGOQ_GEMM_NX, NB = AGOQ_GEMM_NB;
constexpr int kChunk = BK * 128;   // bytes of one 64-wide M (A) or N (B) chunk of a stage
constexpr int kTmaWarp = 0, kMmaWarp = 1, kTmaXWarp = 2, kDeqWarp0 = 3, kDeqWarps = 16;
constexpr int kThreads = (kDeqWarp0 + kDeqWarps) * 32;   // 608
// The two CTAs of a cluster of two form a tcgen05 CTA pair working on one
// 512 x 256 tile: each CTA holds 256 rows of dY (two 128-row halves) and
// dequantizes only its 128 of the 256 X-hat columns; CTA 0 issues pair MMAs
// (M = 256, N = 256) that read the A rows and the B columns of both CTAs and
// accumulate each CTA's rows in its own TMEM.  Per output element this halves
// the dequantization work and the shared-memory traffic of the B operand (a
// single-CTA design with 256 x 256 tiles measured slower: its dequantizers
// were the limit).  CTA 1's relay thread publishes each landed A stage to CTA
// 0 with one remote mbarrier arrive, its dequantizer warps arrive directly on
// CTA 0's B barrier, and every MMA commit is multicast to both CTAs' release
// barriers.
constexpr int kPair = 2;                                   // CTAs per tile
constexpr int kTileRows = BM * kPair;                      // output rows per tile
constexpr int kBCols = BN / kPair;                         // X-hat columns this CTA holds
constexpr int kWordsPerRow = kBCols / 8;                   // 4-bit code words per k-row
constexpr int kRowsPerWarp = 32 / kWordsPerRow;            // k-rows a dequant warp covers at once
constexpr int kDeqRows = BK / (kRowsPerWarp * kDeqWarps); // code words per dequant thread per stage
static_assert(kDeqRows >= 1 && kDeqRows * kRowsPerWarp * kDeqWarps == BK,
              "every k-row of a stage is dequantized exactly once");
static_assert(NB >= 2, "the B ring must let dequantization run ahead of the MMA");
static_assert(kDeqWarps == 16, "epilogue items: 4 TMEM lane quarters x 4 blocks of 128 columns");
// A waiter may only be one phase behind the barrier it polls (a parity test
// cannot tell "two phases ahead" from "complete").  Every ring here is waited
// on by all of its consumers for every phase in order, and tmem_full(t + 1)
// cannot complete before every dequant warp has waited for tmem_full(t) and
// released the accumulator.  The pair-ready ring (CTA 0 only) has as many
// slots as the relay can run ahead of the MMA: NA k-blocks (the relay waits
// for the A stage only, whose TMA producer needs the stages the MMA releases).
constexpr int NP = NA;
constexpr int kAStage = BM * BK * 2;                      // 32 KiB of dY (BF16)
constexpr int kBStage = kBCols * BK * 2;                  // this CTA's X-hat columns (BF16)
constexpr int kCStage = BK * kBCols / 2;                  // their packed codes
constexpr int kSStage = BK * 4 * 4;                       // ... and 4-wide scale boxes
static_assert(BK % 16 == 0 && BK >= 16 && BK <= 256, "k-block depth");
constexpr int kOffB = NA * kAStage;
constexpr int kOffC = kOffB + NB * kBStage;
constexpr int kOffS = kOffC + NX * kCStage;
constexpr int kOffBar = kOffS + NX * kSStage;
constexpr int kNumBars = 2 * NA + 2 * NX + 2 * NB + NP + 3;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;          // + slack for 1024-byte alignment
constexpr uint32_t kTmemCols = 512;
constexpr int kPrefetchLead = 8;   // k-blocks between master prefetch and use

static_assert(kSmemBytes <= 232448, "shared memory budget");

// Instruction descriptor: kind::f16, BF16 A and B, FP32 D, A and B MN-major,
// M = 256 (128 rows from each CTA of the pair), N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                            ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((128 * kPair) >> 4) << 24);

struct Shared {
    uint8_t *a, *b, *c;
    float *s;
    uint64_t *full_a, *empty_a, *full_x, *empty_x, *full_b, *empty_b;
    uint64_t *tmem_full, *tmem_empty, *drain, *pair_ready;
    uint32_t *tmem_addr;
    volatile int *abort;
};

// Dequantize one word of eight 4-bit codes (two's complement, element 2i in
// the low nibble of byte i) with scale s into eight BF16:
// bf16_rne(fl32(c * s)).  The code plus 8 is placed in the mantissa of 2^23
// with a byte permute; subtracting 2^23 + 8 leaves c exactly; the multiply by
// s is the one rounding before the BF16 conversion.
__device__ __forceinline__ uint4 dequant_word(uint32_t w, float s) {
    const uint32_t v = w ^ 0x88888888u;                 // c + 8 in each nibble
    const uint32_t ev = v & 0x0F0F0F0Fu;                // elements 0, 2, 4, 6
    const uint32_t od = (v >> 4) & 0x0F0F0F0Fu;         // elements 1, 3, 5, 7
    const uint64_t bias = f32x2(8388616.0f, 8388616.0f);
    const uint64_t ss = f32x2(s, s);
    uint32_t out[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t fe = __byte_perm(ev, 0x4B000000u, 0x7540u + b);   // element 2b
        const uint32_t fo = __byte_perm(od, 0x4B000000u, 0x7540u + b);   // element 2b+1
        const uint64_t y = mul_f32x2(sub_f32x2(u32x2(fe, fo), bias), ss);
        out[b] = pack_bf16x2(lo_f32(y), hi_f32(y));
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p));
}

// t_i = fl(fl(e4m3(c_i) * s) + acc_i) for the four E4M3 codes of word w and
// four binary32 accumulator values (bit patterns).  The two roundings must
// stay separate (a fused multiply-add gives a different t, e.g. a signed zero
// where m and acc cancel): packed multiplies, scalar adds (a packed multiply
// followed by a packed add was contracted into one rounding by the compiler).
__device__ __forceinline__ void master_plus_acc4(uint32_t w, float s, const uint32_t *acc,
                                                 float t[4]) {
    float e[4];
    e4m3x2_to_f32(w & 0xFFFFu, e[0], e[1]);
    e4m3x2_to_f32(w >> 16, e[2], e[3]);
    // products in packed pairs, each sum a scalar round-to-nearest add
    const uint64_t s2 = f32x2(s, s);
    const uint64_t p01 = mul_f32x2(f32x2(e[0], e[1]), s2), p23 = mul_f32x2(f32x2(e[2], e[3]), s2);
    t[0] = __fadd_rn(lo_f32(p01), __uint_as_float(acc[0]));
    t[1] = __fadd_rn(hi_f32(p01), __uint_as_float(acc[1]));
    t[2] = __fadd_rn(lo_f32(p23), __uint_as_float(acc[2]));
    t[3] = __fadd_rn(hi_f32(p23), __uint_as_float(acc[3]));
}

__device__ __forceinline__ uint32_t word_of(const uint4 (&c)[8], int i) {
    const uint4 v = c[i >> 2];
    return (i & 3) == 0 ? v.x : (i & 3) == 1 ? v.y : (i & 3) == 2 ? v.z : v.w;
}

// The 128 E4M3 master codes and the scale of one row block, loaded before the
// accumulator is ready (the loads do not depend on it).
// WIDE: the codes are 32-byte aligned (32-byte loads).
struct MasterBlock {
    uint4 c[8];
    float s;
    template <bool WIDE>
    __device__ __forceinline__ void load(const uint8_t *codes, const float *scale) {
        if constexpr (WIDE) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t w[8];
                ld_global_32B(codes + 32 * i, w);
                c[2 * i] = make_uint4(w[0], w[1], w[2], w[3]);
                c[2 * i + 1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        } else {
            const uint4 *mc = reinterpret_cast<const uint4 *>(codes);
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = mc[i];
        }
        s = *scale;
    }
};

// QuanGrad accumulation of one 128-column block of an accumulator row into the
// FP8 master (in place): `taddr` is the TMEM address of the block's first
// column in this warp's lane quarter, `mb` the block's master codes and scale
// (already loaded), `codes`/`scale` where the new ones go.  The first pass
// forms t = fl(fl(e4m3(c) * s) + acc), takes the block absmax and writes t
// back over the accumulator in TMEM; the second pass reads t and requantizes
// with the new scale.  WIDE: `codes` is 32-byte aligned (32-byte stores).
template <bool WIDE>
__device__ __forceinline__ void accum_fp8_block(uint32_t taddr, const MasterBlock &mb,
                                                uint8_t *codes, float *scale) {
    uint4 *mc = reinterpret_cast<uint4 *>(codes);
    float am = 0.0f;
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld16_nowait(taddr + cc * 16, v);
        tmem_wait_ld();
        float t[16];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            master_plus_acc4(word_of(mb.c, cc * 4 + w), mb.s, v + 4 * w, t + 4 * w);
            am = fmaxf(am, fmaxf(fmaxf(fabsf(t[4 * w]), fabsf(t[4 * w + 1])),
                                 fmaxf(fabsf(t[4 * w + 2]), fabsf(t[4 * w + 3]))));
        }
        tmem_st16(taddr + cc * 16, t);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    const float snew = __fdiv_rn(am, kE4M3Max);
    uint32_t prev[4];   // WIDE: the even 16-code group, stored with the odd one
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
        uint32_t v[16];
        __syncwarp();   // lanes may have left the fast requantization path; tcgen05.ld is .aligned
        tmem_ld16_nowait(taddr + cc * 16, v);
        tmem_wait_ld();
        uint32_t o[4];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            float t[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = __uint_as_float(v[8 * p + i]);
            const uint2 q = e4m3_codes8(t, snew);
            o[2 * p] = q.x;
            o[2 * p + 1] = q.y;
        }
        if constexpr (WIDE) {
            if (cc & 1) {
                const uint32_t w[8] = {prev[0], prev[1], prev[2], prev[3], o[0], o[1], o[2], o[3]};
                st_global_32B(mc + cc - 1, w);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) prev[i] = o[i];
            }
        } else {
            mc[cc] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    *scale = snew;
}

// One epilogue item of the FP32-output or accumulation epilogue: row `row`,
// columns col0 .. col0+127 of the output, whose accumulators start at TMEM
// address `taddr` (this warp's lane quarter); `mb` holds the item's master
// block for the accumulation epilogue.  WIDE: the row's output is 32-byte
// aligned (32-byte stores).
template <int EPI, bool WIDE>
__device__ __forceinline__ void epilogue_item(uint32_t taddr, void *dW, float *mscales, int row,
                                              int col0, int N, const MasterBlock &mb) {
    static_assert(EPI == kEpiAccumFp8 || EPI == kEpiF32, "the BF16 epilogue is in the kernel");
    if constexpr (EPI == kEpiAccumFp8) {
        accum_fp8_block<WIDE>(taddr, mb, static_cast<uint8_t *>(dW) + (size_t)row * N + col0,
                              mscales + (size_t)row * (N / 128) + col0 / 128);
    } else {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            tmem_ld32(taddr + cc * 32, v);
            float *dst = static_cast<float *>(dW) + (size_t)row * N + col0 + cc * 32;
            if constexpr (WIDE) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w[8] = {v[8 * j], v[8 * j + 1], v[8 * j + 2], v[8 * j + 3],
                                           v[8 * j + 4], v[8 * j + 5], v[8 * j + 6], v[8 * j + 7]};
                    st_global_32B(dst + 8 * j, w);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    reinterpret_cast<uint4 *>(dst)[j] =
                        make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
        }
    }
}

// The MMAs of one k-block: BK/16 K-steps of 16, each for the M-halves (the
// second only when BOTH) sharing the K-step's B descriptor; the first K-step
// of a tile overwrites the accumulator.  The depth is a compile-time constant
// so the issuing thread runs a straight line of MMA instructions (a depth test
// in the loop measured 2-7% slower, hence one kernel per BK).
//   a0: the A stage; b0: the B stage.
template <bool BOTH>
__device__ __forceinline__ void issue_kblock_h(uint32_t tmem_base, uint32_t a0, uint32_t b0,
                                               bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
        const uint64_t bdesc = sw128_desc(b0 + kk * 2048, kChunk, 1024);
        const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
        umma_bf16_pair(tmem_base, sw128_desc(a0 + kk * 2048, kChunk, 1024), bdesc, kIdesc, acc);
        if constexpr (BOTH)
            umma_bf16_pair(tmem_base + 256, sw128_desc(a0 + 2 * kChunk + kk * 2048, kChunk, 1024),
                           bdesc, kIdesc, acc);
    }
}
__device__ __forceinline__ void issue_kblock(uint32_t tmem_base, uint32_t a0, uint32_t b0,
                                             bool accumulate, bool both) {
    if (both)
        issue_kblock_h<true>(tmem_base, a0, b0, accumulate);
    else
        issue_kblock_h<false>(tmem_base, a0, b0, accumulate);
}

// dW (EPI kEpiBf16 / kEpiF32) or the FP8 master codes (kEpiAccumFp8, with
// their scales in `mscales`) are [M][N] row-major.  M and N are multiples of
// 128: rows past M of the last tile read as zeros and are not stored, and when
// N is not a multiple of 256 the last tile's second 128-column block (codes
// and scales read as zeros) is not stored.  With TMA_SCALES the X scales come
// through the X ring by TMA (a scale row is then a multiple of 16 bytes: N a
// multiple of 512); otherwise the X producer warp reads them from `xs` into
// the same shared-memory slots.  WIDE: dW (or the master codes) is 32-byte
// aligned, so each epilogue row is written (and the master read) in 32-byte
// accesses; every output row starts on such a boundary then, as N is a
// multiple of 128.
template <int EPI, bool TMA_SCALES, bool WIDE>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad_gemm_int4_kernel(const __grid_constant__ CUtensorMap map_dy,
                           const __grid_constant__ CUtensorMap map_xc,
                           const __grid_constant__ CUtensorMap map_xs,
                           const float *__restrict__ xs, void *__restrict__ dW,
                           float *__restrict__ mscales, int M, int N, int K) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Shared sh;
    sh.a = smem;
    sh.b = smem + kOffB;
    sh.c = smem + kOffC;
    sh.s = reinterpret_cast<float *>(smem + kOffS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    sh.full_a = bars;
    sh.empty_a = sh.full_a + NA;
    sh.full_x = sh.empty_a + NA;
    sh.empty_x = sh.full_x + NX;
    sh.full_b = sh.empty_x + NX;
    sh.empty_b = sh.full_b + NB;
    sh.pair_ready = sh.empty_b + NB;
    sh.tmem_full = sh.pair_ready + NP;
    sh.tmem_empty = sh.tmem_full + 1;
    sh.drain = sh.tmem_empty + 1;
    sh.tmem_addr = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    sh.abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (N + BN - 1) / BN, kblocks = K / BK;   // K is a multiple of BK
    // Tile g covers rows m0 .. m0 + kTileRows - 1 and columns n0 .. n0 + 255;
    // this CTA (rank in the pair) holds rows half_row(h) .. +127 of M-half h
    // and X-hat columns n0 + rank * kBCols .. + kBCols - 1.  Rows at or past M
    // (the second half of the last tile) are neither multiplied nor stored.
    const int rank = (int)cluster_ctarank();
    const int cluster_id = (int)(blockIdx.x / kPair), num_clusters = (int)(gridDim.x / kPair);
    const int m_tiles = (M + kTileRows - 1) / kTileRows, num_groups = m_tiles * n_tiles;
    auto tile_of = [&](int g, int &m0, int &n0) {
        m0 = (g / n_tiles) * kTileRows;
        n0 = (g % n_tiles) * BN;
    };
    auto half_row = [&](int m0, int h) { return m0 + h * 128 * kPair + 128 * rank; };
    // some row of the pair's M-half h lies below M (its MMAs are issued)
    auto half_valid = [&](int m0, int h) { return m0 + h * 128 * kPair < M; };
    // this CTA's rows of M-half h, and the 128-column block at col0, are stored
    auto item_valid = [&](int m0, int h, int col0) { return half_row(m0, h) < M && col0 < N; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NA; ++s) {
            mbar_init(&sh.full_a[s], 1);
            mbar_init(&sh.empty_a[s], 1);
        }
        for (int s = 0; s < NX; ++s) {
            mbar_init(&sh.full_x[s], 1);
            mbar_init(&sh.empty_x[s], kDeqWarps);
        }
        for (int s = 0; s < NB; ++s) {
            mbar_init(&sh.full_b[s], kDeqWarps * kPair);   // every dequantizer warp of the pair
            mbar_init(&sh.empty_b[s], 1);
        }
        for (int s = 0; s < NP; ++s) mbar_init(&sh.pair_ready[s], 1);
        mbar_init(sh.tmem_full, 1);
        mbar_init(sh.tmem_empty, kDeqWarps * kPair);   // every epilogue warp of the pair
        mbar_init(sh.drain, 1);
        *sh.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(sh.tmem_addr)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();   // the peer's barriers are initialised
    const uint32_t tmem_base = *sh.tmem_addr;

    if (warp == kTmaWarp) {
        // Producer of the A ring (one lane).
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int g = cluster_id; ok && g < num_groups; g += num_clusters) {
                int m0, n0;
                tile_of(g, m0, n0);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % NA;
                    const uint32_t ph = (it / NA) & 1u;
                    if (!wait_bar(&sh.empty_a[s], ph ^ 1u, sh.abort, &g_device_status)) { ok = false; break; }
                    const int k0 = kb * BK;
                    const int halves = half_valid(m0, 1) ? 2 : 1;
                    mbar_expect_tx(&sh.full_a[s], halves * (kAStage / 2));
                    for (int h = 0; h < halves; ++h) {
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tma_load_2d(sh.a + s * kAStage + (2 * h + c) * kChunk, &map_dy,
                                        &sh.full_a[s], half_row(m0, h) + 64 * c, k0);
                    }
                }
            }
            // Drain: every issued load lands before the CTA may exit (a no-op
            // unless the pipeline was aborted).  Iteration it-1-d was the last
            // load into stage (it-1-d) % NA.
            for (int d = 0; d < NA && d < (int)it; ++d) {
                const uint32_t last = it - 1 - d;
                wait_bar(&sh.full_a[last % NA], (last / NA) & 1u, sh.abort, &g_device_status, true);
            }
        }
    } else if (warp == kTmaXWarp) {
        // Producer of the X ring: lane 0 waits for the stage and issues the TMA
        // loads of the codes (and, with TMA_SCALES, of the 4-wide scale box);
        // without TMA_SCALES the warp's lanes read this CTA's scale of each
        // k-row from global memory into the stage's scale slots, and the
        // arrive that follows (after __syncwarp) publishes them with the codes.
        // The scales of k-block (g, kb): lane l holds k-rows l, l + 32, ...;
        // zeros past N (where the codes read as zeros too).
        constexpr int kScPerLane = BK / 32;
        static_assert(BK % 32 == 0, "every k-row of a stage gets its scale");
        auto load_scales = [&](int g, int kb, float (&v)[kScPerLane]) {
            int m0, n0;
            tile_of(g, m0, n0);
            const int cb = n0 + rank * kBCols;
#pragma unroll
            for (int i = 0; i < kScPerLane; ++i)
                v[i] = cb < N ? __ldg(xs + (size_t)(kb * BK + lane + 32 * i) * (N / 128) + cb / 128)
                              : 0.0f;
        };
        float vsc[kScPerLane];
        if (!TMA_SCALES && cluster_id < num_groups) load_scales(cluster_id, 0, vsc);
        uint32_t it = 0;
        bool ok = true;
        for (int g = cluster_id; ok && g < num_groups; g += num_clusters) {
            int m0, n0;
            tile_of(g, m0, n0);
            const int cb = n0 + rank * kBCols;   // first X-hat column of this CTA
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % NX;
                const uint32_t ph = (it / NX) & 1u;
                float cur[kScPerLane];
                if (!TMA_SCALES) {
                    // this k-block's scales are in registers; the next one's
                    // loads are issued before the wait for the stage
#pragma unroll
                    for (int i = 0; i < kScPerLane; ++i) cur[i] = vsc[i];
                    if (kb + 1 < kblocks)
                        load_scales(g, kb + 1, vsc);
                    else if (g + num_clusters < num_groups)
                        load_scales(g + num_clusters, 0, vsc);
                }
                if (!warp_wait(&sh.empty_x[s], ph ^ 1u, sh.abort, &g_device_status)) { ok = false; break; }
                const int k0 = kb * BK;
                if (!TMA_SCALES) {
                    float *dst = sh.s + s * (kSStage / 4) + ((cb / 128) & 3);
#pragma unroll
                    for (int i = 0; i < kScPerLane; ++i) dst[4 * (lane + 32 * i)] = cur[i];
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_expect_tx(&sh.full_x[s], kCStage + (TMA_SCALES ? kSStage : 0));
                    tma_load_2d(sh.c + s * kCStage, &map_xc, &sh.full_x[s], cb / 2, k0);
                    if (TMA_SCALES)
                        tma_load_2d(sh.s + s * (kSStage / 4), &map_xs, &sh.full_x[s],
                                    (cb / 128) & ~3, k0);
                }
            }
        }
        if (lane == 0) {
            for (int d = 0; d < NX && d < (int)it; ++d) {
                const uint32_t last = it - 1 - d;
                wait_bar(&sh.full_x[last % NX], (last / NX) & 1u, sh.abort, &g_device_status, true);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && rank == 0) {
            // MMA issuer (CTA 0 of a pair issues for both CTAs).
            uint32_t it = 0, t = 0;
            bool ok = true, issued = false;
            for (int g = cluster_id; ok && g < num_groups; g += num_clusters, ++t) {
                int m0, n0;
                tile_of(g, m0, n0);
                const bool v1 = half_valid(m0, 1);
                if (!wait_bar(sh.tmem_empty, (t & 1u) ^ 1u, sh.abort, &g_device_status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int sa = it % NA, sb = it % NB;
                    if (!wait_bar(&sh.full_a[sa], (it / NA) & 1u, sh.abort, &g_device_status) ||
                        !wait_bar(&sh.pair_ready[it % NP], (it / NP) & 1u, sh.abort,
                                  &g_device_status) ||
                        !wait_bar(&sh.full_b[sb], (it / NB) & 1u, sh.abort, &g_device_status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_kblock(tmem_base, smem_u32(sh.a + sa * kAStage),
                                 smem_u32(sh.b + sb * kBStage), kb > 0, v1);
                    issued = true;
                    umma_commit_pair_multicast(&sh.empty_b[sb], 3);
                    umma_commit_pair_multicast(&sh.empty_a[sa], 3);
                }
                if (!ok) break;
                umma_commit_pair_multicast(sh.tmem_full, 3);
            }
            // Drain: all MMAs issued so far complete before TMEM is freed.
            if (issued) {
                umma_commit_pair(sh.drain);
                wait_bar(sh.drain, 0u, sh.abort, &g_device_status, true);
            }
        } else if (lane == 0) {
            // Relay (CTA 1 of a pair): once this CTA's A stage of a k-block
            // has landed, tell the issuing CTA with one remote arrive (its
            // dequantizer warps arrive on CTA 0's B barrier themselves).
            const uint32_t ready0 = mapa_shared(smem_u32(sh.pair_ready), 0);
            uint32_t it = 0;
            bool ok = true;
            for (int g = cluster_id; ok && g < num_groups; g += num_clusters) {
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    if (!wait_bar(&sh.full_a[it % NA], (it / NA) & 1u, sh.abort, &g_device_status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote(ready0 + (uint32_t)(it % NP) * 8u);
                }
            }
        }
    } else {
        // Dequantizers, which also run the epilogue of the previous tile.
        const int d = warp - kDeqWarp0;
        const int wc = lane % kWordsPerRow;             // code word column: X-hat cols 8wc .. 8wc+7
        const int rsub = lane / kWordsPerRow;
        const int chunk = wc >> 3, piece = wc & 7;
        // Epilogue item: TMEM lane quarter q (tcgen05.ld reaches lanes
        // 32*(warp%4) .. +31) and 128-column block `item` of the tile: rows
        // half_row(eh) + 32q + lane, columns n0 + 128*ejb .. +127.
        const int q = warp & 3, item = d >> 2, eh = item >> 1, ejb = item & 1;
        const uint32_t etaddr = tmem_base + ((uint32_t)(32 * q) << 16) + eh * 256 + ejb * 128;
        const uint32_t tmem_empty0 = mapa_shared(smem_u32(sh.tmem_empty), 0);
        const uint32_t full_b0 = mapa_shared(smem_u32(sh.full_b), 0);
        // The previous tile's epilogue runs once this tile's first k-block of
        // X-hat is written (measured: waiting for more of the ring, or running
        // it before, was slower).
        auto epilogue = [&](int g, uint32_t t) -> bool {
            int m0, n0;
            tile_of(g, m0, n0);
            const int row = half_row(m0, eh) + 32 * q + lane, col0 = n0 + ejb * 128;
            const bool valid = item_valid(m0, eh, col0);   // the same for the whole warp
            MasterBlock mb;
            if (!warp_wait(sh.tmem_full, t & 1u, sh.abort, &g_device_status)) return false;
            tc_fence_after();
            if constexpr (EPI == kEpiAccumFp8) {
                if (valid)
                    mb.load<WIDE>(static_cast<const uint8_t *>(dW) + (size_t)row * N + col0,
                            mscales + (size_t)row * (N / 128) + col0 / 128);
            }
            auto release = [&]() {   // the accumulator may be overwritten
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rank != 0)
                        mbar_arrive_remote(tmem_empty0);
                    else
                        mbar_arrive(sh.tmem_empty);
                }
            };
            if constexpr (EPI == kEpiBf16) {
                // Read and round the whole item into registers, hand the
                // accumulator back to the MMA, then store while the next tile's
                // MMAs run.
                uint32_t h[64];
                uint16_t *dst = static_cast<uint16_t *>(dW) + (size_t)row * N + col0;
                if (valid) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t v[32];
                        tmem_ld32(etaddr + cc * 32, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            h[16 * cc + i] =
                                pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    }
                }
                release();
                if (valid) {
                    // each lane writes its own row: 32-byte stores halve the
                    // store instructions (measured 3% on the whole kernel)
                    if constexpr (WIDE) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint32_t w[8] = {h[8 * j], h[8 * j + 1], h[8 * j + 2],
                                                   h[8 * j + 3], h[8 * j + 4], h[8 * j + 5],
                                                   h[8 * j + 6], h[8 * j + 7]};
                            st_global_32B(dst + 16 * j, w);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            reinterpret_cast<uint4 *>(dst)[j] =
                                make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
                    }
                }
            } else {
                if (valid) epilogue_item<EPI, WIDE>(etaddr, dW, mscales, row, col0, N, mb);
                release();
            }
            return true;
        };
        uint32_t it = 0, t = 0;
        bool ok = true;
        int prev = -1;
        for (int g = cluster_id; ok && g < num_groups; g += num_clusters, ++t) {
            int m0, n0;
            tile_of(g, m0, n0);
            const int cb = n0 + rank * kBCols;
            const int soff = ((cb / 128) & 3) + (wc >> 4);   // scale column inside the 4-wide box
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                if constexpr (EPI == kEpiAccumFp8) {
                    // Pull this thread's master block of the tile into L2 a few
                    // k-blocks before its epilogue needs it.
                    if (item_valid(m0, eh, n0 + ejb * 128) &&
                        kb == (kblocks > kPrefetchLead ? kblocks - kPrefetchLead : 0)) {
                        const size_t row = (size_t)(half_row(m0, eh) + 32 * q + lane);
                        prefetch_l2(static_cast<const uint8_t *>(dW) + row * N + n0 + ejb * 128);
                        prefetch_l2(mscales + row * (N / 128) + n0 / 128 + ejb);
                    }
                }
                const int sx = it % NX;
                if (!warp_wait(&sh.full_x[sx], (it / NX) & 1u, sh.abort, &g_device_status)) { ok = false; break; }
                const uint32_t *codes = reinterpret_cast<const uint32_t *>(sh.c + sx * kCStage);
                const float *scales = sh.s + sx * (kSStage / 4);
                uint32_t w[kDeqRows];
                float sc[kDeqRows];
#pragma unroll
                for (int i = 0; i < kDeqRows; ++i) {
                    const int k = kRowsPerWarp * (d + kDeqWarps * i) + rsub;   // row of the stage
                    w[i] = codes[k * kWordsPerRow + wc];
                    sc[i] = scales[k * 4 + soff];
                }
                const int sb = it % NB;
                // The B stage may be overwritten once the MMA has read it.
                if (!warp_wait(&sh.empty_b[sb], ((it / NB) & 1u) ^ 1u, sh.abort, &g_device_status)) {
                    ok = false;
                    break;
                }
                uint8_t *btile = sh.b + sb * kBStage + chunk * kChunk;
#pragma unroll
                for (int i = 0; i < kDeqRows; ++i) {
                    const int k = kRowsPerWarp * (d + kDeqWarps * i) + rsub;
                    const uint4 y = dequant_word(w[i], sc[i]);
                    uint8_t *dst = btile + k * 128 + ((piece ^ (k & 7)) << 4);
                    *reinterpret_cast<uint4 *>(dst) = y;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    if (rank != 0)
                        mbar_arrive_remote(full_b0 + (uint32_t)sb * 8u);
                    else
                        mbar_arrive(&sh.full_b[sb]);
                }
                // The X stage is released only now: its codes have been consumed
                // (the B stores depend on them), so no shared-memory load of it
                // can still be in flight when the next TMA load overwrites it.
                if (lane == 0) mbar_arrive(&sh.empty_x[sx]);
                if (kb == 0 && prev >= 0 && !epilogue(prev, t - 1)) { ok = false; break; }
            }
            prev = g;
        }
        if (ok && prev >= 0) epilogue(prev, t - 1);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Neither CTA of a pair leaves (or frees TMEM) while the other may still
    // arrive on its barriers or have the pair's MMAs read its shared memory.
    cluster_sync_all();
    if (warp == kMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// Failure-path probe: one thread waits, with the GEMM's bounded wait and a
// caller-given limit, for the first phase of an mbarrier that nothing arrives
// on; the wait runs out, records the timeout in this instance's status word
// and the kernel returns.
__global__ void wait_timeout_probe_kernel(long long limit_cycles) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0)
        wait_bar(&bar, 0u, &abort_flag, &g_device_status, false, 0u, limit_cycles);
}

// ---------------------------------------------------------------- host side
template <int EPI, bool TMA_SCALES, bool WIDE>
cudaError_t launch_impl(const void *dY, const void *xc, const float *xs, int M, int N, int K,
                        void *dW, float *mscales, cudaStream_t st) {
    CUtensorMap m_dy, m_xc, m_xs;
    if (!encode_2d(&m_dy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, (uint64_t)M, (uint64_t)K,
                   (uint64_t)M * 2, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&m_xc, CU_TENSOR_MAP_DATA_TYPE_UINT8, xc, (uint64_t)N / 2, (uint64_t)K,
                   (uint64_t)N / 2, kBCols / 2, BK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (!TMA_SCALES)
        m_xs = m_xc;   // unused by this instance
    else if (!encode_2d(&m_xs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xs, (uint64_t)N / 128, (uint64_t)K,
                        (uint64_t)(N / 128) * 4, 4, BK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    auto kernel = wgrad_gemm_int4_kernel<EPI, TMA_SCALES, WIDE>;
    static bool attr_set[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevices && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int groups = ((M + kTileRows - 1) / kTileRows) * ((N + BN - 1) / BN);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kPair;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Persistent grid: as many pairs as can be resident at once (a cluster
    // must fit in one GPC, so this can be below sm_count / 2).
    static int resident[kMaxDevices];
    if (dev >= 0 && dev < kMaxDevices && resident[dev] == 0) {
        cfg.gridDim = dim3(sm_count() / kPair * kPair);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0)
            n = sm_count() / kPair;
        resident[dev] = n;
    }
    const int clusters = (dev >= 0 && dev < kMaxDevices) ? resident[dev] : sm_count() / kPair;
    cfg.gridDim = dim3((groups < clusters ? groups : clusters) * kPair);
    return cudaLaunchKernelEx(&cfg, kernel, m_dy, m_xc, m_xs, xs, dW, mscales, M, N, K);
}

// Scales by TMA when a scale row is a multiple of 16 bytes and 16-byte aligned;
// 32-byte epilogue accesses when the output is 32-byte aligned.
template <int EPI>
cudaError_t launch_any(const void *dY, const void *xc, const float *xs, int M, int N, int K,
                       void *dW, float *mscales, cudaStream_t st) {
    const bool tma = (N / 128) % 4 == 0 && (reinterpret_cast<uintptr_t>(xs) & 15u) == 0;
    const bool wide = (reinterpret_cast<uintptr_t>(dW) & 31u) == 0;
    if (wide)
        return tma ? launch_impl<EPI, true, true>(dY, xc, xs, M, N, K, dW, mscales, st)
                   : launch_impl<EPI, false, true>(dY, xc, xs, M, N, K, dW, mscales, st);
    return tma ? launch_impl<EPI, true, false>(dY, xc, xs, M, N, K, dW, mscales, st)
               : launch_impl<EPI, false, false>(dY, xc, xs, M, N, K, dW, mscales, st);
}

}  // namespace

cudaError_t launch_gemm(const void *dY, const void *xc, const float *xs, int M, int N, int K,
                        void *dW, bool f32_out, cudaStream_t st) {
    return f32_out ? launch_any<kEpiF32>(dY, xc, xs, M, N, K, dW, nullptr, st)
                   : launch_any<kEpiBf16>(dY, xc, xs, M, N, K, dW, nullptr, st);
}

cudaError_t launch_accum_fp8(const void *dY, const void *xc, const float *xs, int M, int N, int K,
                             void *master, float *master_scales, cudaStream_t st) {
    return launch_any<kEpiAccumFp8>(dY, xc, xs, M, N, K, master, master_scales, st);
}

cudaError_t launch_wait_timeout_probe(long long limit_cycles, cudaStream_t st) {
    wait_timeout_probe_kernel<<<1, 32, 0, st>>>(limit_cycles);
    return cudaGetLastError();
}

// Read and clear this instance's status word (the stream is synchronised).
cudaError_t read_and_clear_status(unsigned *status) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
        if (e != cudaSuccess) return e;
    }
    *status = v;
    return cudaSuccess;
}

}  // namespace AGOQ_WGRAD_NS
}  // namespace agoq
