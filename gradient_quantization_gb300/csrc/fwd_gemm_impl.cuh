// fwd_gemm_impl.cuh -- a linear layer's forward GEMM with the LAAQ quantization of
// its output fused into the epilogue ("AGoQ: Activation and Gradient
// Quantization for Memory-Efficient Distributed Training of LLMs", section 2.C
// "Kernel Fusion": the quantization runs on the CUDA cores of the GEMM kernel;
// section 2.A: the activation kept for the backward pass is stored in b bits).
//
//   Y[t][n] = bf16(fl32(sum_k X[t][k] * W[n][k]))     X [T][K], W [N][K], BF16
//   codes, scales = LAAQ b-bit quantization of Y (128-column blocks of each row)
//
// Blackwell design (sm_103a), persistent, one CTA per SM; the two CTAs of a
// cluster of two form a tcgen05 CTA pair on 256 x 256 output tiles, both
// operands K-major:
//   warp 0      TMA producer: per BK-deep k-block, this CTA's 128 rows of X
//               and its 128 of the tile's 256 rows of W (64-wide boxes with
//               the 128-byte swizzle) into an NS-stage ring;
//   warp 1      TMEM allocation for the pair; in CTA 0 one thread issues BK/16
//               pair MMAs tcgen05.mma.cta_group::2 kind::f16 (M=256: 128 rows
//               from each CTA; N=256: 128 W rows from each CTA; K=16) per
//               k-block into one of two 256-column accumulators per CTA, so the
//               epilogue of a tile overlaps the mainloop of the next; the
//               commits are multicast to both CTAs.  In CTA 1 one thread
//               relays each landed stage to CTA 0 (remote mbarrier arrive).
//   warps 2-5   epilogue, in each CTA for its own rows: one output row per
//               thread (its TMEM lane quarter is warp % 4); per 128-column
//               block, a first pass reads the accumulator (tcgen05.ld), rounds
//               it to BF16, stores Y and takes the block absmax; a second pass
//               reads it again, forms the codes (corrected-reciprocal quotient,
//               as the LAAQ quantizer) and stores the packed record and the
//               scale.  CTA 1's warps release an accumulator with a remote
//               arrive on CTA 0's barrier.
// Every mbarrier wait is time-limited (status word, CTA abort flag, drains); the
// two CTAs of a pair meet at a cluster barrier before either frees TMEM.
#pragma once
#include "agoq_device.cuh"
#include "agoq_launch.h"
#include "gemm_common.cuh"

namespace agoq {
namespace AGOQ_FWD_INSTANCE {
namespace {

using namespace gemm;

// Device-side status word of this instance's kernels (read with the GEMM's by
// agoq_device_status).
__device__ unsigned g_fwd_status;

// The two CTAs of a cluster of two form a tcgen05 CTA pair on 256 x 256
// tiles: each CTA loads 128 rows of X and 128 of the tile's 256 rows of W, and
// CTA 0 issues pair MMAs (M = 256, N = 256) that read both CTAs' shared memory,
// so each SM streams half of the W tile from L2 and reads half as many B bytes
// from shared memory per MMA (a single-CTA design on 128 x 256 tiles measured
// slower).  CTA 1 publishes each landed stage to CTA 0 with a remote mbarrier
// arrive.
// AGOQ_FWD_BK (k-block depth) and AGOQ_FWD_STAGES (ring depth) are set by the
// translation unit that includes this file (fwd_gemm.cu: BK = 128 for K a
// multiple of 128; fwd_gemm_k64.cu: BK = 64 for the other multiples of 64),
// and AGOQ_FWD_INSTANCE names the instance's namespace.
constexpr int kPair = 2;
constexpr int BM = 128, BN = 256, BK = AGOQ_FWD_BK, NS = AGOQ_FWD_STAGES;
constexpr int kTileRows = BM * kPair;                     // output rows per tile
constexpr int kBRows = BN / kPair;                        // W rows this CTA loads per tile
constexpr int kAtoms = BK / 64;                           // 64-wide K atoms (128-byte swizzle span)
constexpr int kThreads = 192;
constexpr int kTmaWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kEpiWarps = 4;
constexpr int kAAtom = BM * 128, kBAtom = kBRows * 128;   // bytes of one K atom of A / B
constexpr int kAStage = kAtoms * kAAtom;
constexpr int kBStage = kAtoms * kBAtom;
constexpr int kOffB = NS * kAStage;
constexpr int kOffBar = kOffB + NS * kBStage;
constexpr int kNumBars = 3 * NS + 4 + 1;                  // full/empty/pair-ready, tmem full/empty x2, drain
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
static_assert(BK % 64 == 0, "k-blocks are whole 64-wide swizzle atoms");
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Tile order: bands of kBand consecutive N-panels; within a band the tiles run
// N-fastest, then M, so the CTAs working at the same time share a few W panels
// and X row blocks (a working set that stays in L2; bands of 4, 8 or 32
// measured slower).
constexpr int kBand = 16;

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &m0, int &n0) {
    const int band = tile / (kBand * num_m);
    const int nb = min(kBand, num_n - band * kBand);            // panels in this band
    const int r = tile - band * kBand * num_m;
    m0 = (r / nb) * kTileRows;
    n0 = (band * kBand + r % nb) * BN;
}

// Streaming (evict-first) store of the outputs, which no later part of the
// kernel reads.
__device__ __forceinline__ void st_stream16(void *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// kind::f16, BF16 A and B, FP32 D, both K-major, M = 256 (128 rows from each
// CTA of the pair), N = 256.
constexpr uint32_t kIdescK = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                             ((uint32_t)(kTileRows >> 4) << 24);

// Append `n` (<= 64 - pending) low bits of v to a little-endian bit stream held
// in acc, emitting full 32-bit words to out[] as they fill.
struct BitSink {
    uint64_t acc = 0;
    int bits = 0, nw = 0;
    uint32_t *out;
    __device__ __forceinline__ explicit BitSink(uint32_t *o) : out(o) {}
    __device__ __forceinline__ void put(uint64_t v, int n) {
        acc |= v << bits;
        bits += n;
        while (bits >= 32) {
            out[nw++] = static_cast<uint32_t>(acc);
            acc >>= 32;
            bits -= 32;
        }
    }
};

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_gemm_quant_kernel(const __grid_constant__ CUtensorMap map_x,
                          const __grid_constant__ CUtensorMap map_w, int T, int N, int K,
                          uint16_t *__restrict__ y, uint32_t *__restrict__ codes,
                          float *__restrict__ scales) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sa = smem, *sb = smem + kOffB;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *full = bars, *empty = bars + NS, *ready = bars + 2 * NS, *tfull = bars + 3 * NS,
             *tempty = tfull + 2, *drain = tempty + 2;
    uint32_t *tmem_addr = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    unsigned *status = &g_fwd_status;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tile (m0, n0) covers rows m0 .. m0 + kTileRows - 1; this CTA (rank in the
    // pair) holds rows m0 + 128 rank .. +127 and loads W rows
    // n0 + kBRows rank .. + kBRows - 1.  Rows at or past T read as zeros and
    // are not stored.
    const int rank = (int)cluster_ctarank();
    const int cid = (int)(blockIdx.x / kPair), ncl = (int)(gridDim.x / kPair);
    const int num_m = (T + kTileRows - 1) / kTileRows, num_n = N / BN;
    const int num_tiles = num_m * num_n, kblocks = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&ready[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps * kPair);
        }
        mbar_init(drain, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_addr)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();   // the peer's barriers are initialised
    const uint32_t tmem_base = *tmem_addr;

    if (warp == kTmaWarp) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = cid; ok && tile < num_tiles; tile += ncl) {
                int m0, n0;
                tile_coords(tile, num_m, num_n, m0, n0);
                const int ar = m0 + BM * rank, br = n0 + kBRows * rank;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % NS;
                    if (!wait_bar(&empty[s], ((it / NS) & 1u) ^ 1u, abort, status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&full[s], kAStage + kBStage);
#pragma unroll
                    for (int a = 0; a < kAtoms; ++a) {
                        tma_load_2d(sa + s * kAStage + a * kAAtom, &map_x, &full[s], kb * BK + 64 * a, ar);
                        tma_load_2d(sb + s * kBStage + a * kBAtom, &map_w, &full[s], kb * BK + 64 * a, br);
                    }
                }
            }
            for (int d = 0; d < NS && d < (int)it; ++d) {
                const uint32_t last = it - 1 - d;
                wait_bar(&full[last % NS], (last / NS) & 1u, abort, status, true);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && rank == 0) {
            // MMA issuer (CTA 0 of a pair issues for both CTAs)
            uint32_t it = 0, t = 0;
            bool ok = true, issued = false;
            for (int tile = cid; ok && tile < num_tiles; tile += ncl, ++t) {
                const int buf = t & 1;
                if (!wait_bar(&tempty[buf], ((t >> 1) & 1u) ^ 1u, abort, status)) break;
                tc_fence_after();
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % NS;
                    if (!wait_bar(&full[s], (it / NS) & 1u, abort, status) ||
                        !wait_bar(&ready[s], (it / NS) & 1u, abort, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sa + s * kAStage), b0 = smem_u32(sb + s * kBStage);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // K-step kk: atom kk / 4, 32 bytes per step inside the atom
                        const uint64_t adesc = sw128_kmajor_desc(a0 + (kk >> 2) * kAAtom + 32 * (kk & 3));
                        const uint64_t bdesc = sw128_kmajor_desc(b0 + (kk >> 2) * kBAtom + 32 * (kk & 3));
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        umma_bf16_pair(tmem_base + buf * BN, adesc, bdesc, kIdescK, acc);
                    }
                    issued = true;
                    umma_commit_pair_multicast(&empty[s], 3);
                }
                if (!ok) break;
                umma_commit_pair_multicast(&tfull[buf], 3);
            }
            if (issued) {
                umma_commit_pair(drain);
                wait_bar(drain, 0u, abort, status, true);
            }
        } else if (lane == 0) {
            // Relay (CTA 1): each landed stage is announced to CTA 0.
            const uint32_t ready0 = mapa_shared(smem_u32(ready), 0);
            uint32_t it = 0;
            bool ok = true;
            for (int tile = cid; ok && tile < num_tiles; tile += ncl) {
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % NS;
                    if (!wait_bar(&full[s], (it / NS) & 1u, abort, status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote(ready0 + (uint32_t)s * 8u);
                }
            }
        }
    } else {
        // epilogue: TMEM lane quarter q = warp % 4, one output row per thread
        constexpr int kQmax = (1 << (BITS - 1)) - 1;
        const int q = warp & 3;
        const int rec_per_row = N / kBlock;
        const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
        uint32_t t = 0;
        for (int tile = cid; tile < num_tiles; tile += ncl, ++t) {
            const int buf = t & 1;
            if (!warp_wait(&tfull[buf], (t >> 1) & 1u, abort, status)) break;
            tc_fence_after();
            int m0, n0;
            tile_coords(tile, num_m, num_n, m0, n0);
            const bool valid = m0 + BM * rank < T;   // the same for the whole CTA
            const int row = m0 + BM * rank + 32 * q + lane;
            const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + buf * BN;
#pragma unroll 1
            for (int jb = 0; valid && jb < BN / kBlock; ++jb) {
                const int col0 = n0 + jb * kBlock;
                // pass 1: Y in BF16 and the block absmax
                float am = 0.0f;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_ld32(tbase + jb * kBlock + cc * 32, v);
                    uint32_t h[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        h[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    uint4 *dst = reinterpret_cast<uint4 *>(y + (size_t)row * N + col0 + cc * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_stream16(dst + i, make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]));
                    am = fmaxf(am, bf16_absmax<16>(h));
                }
                const float s = __fdiv_rn(am, (float)kQmax);   // +0 for an all-zero block
                uint32_t *rec = codes + ((size_t)row * rec_per_row + col0 / kBlock) * (4 * BITS);
                // pass 2: codes of the BF16 values, packed BITS words per 32 values
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    __syncwarp();   // lanes may have taken different quotient paths
                    tmem_ld32(tbase + jb * kBlock + cc * 32, v);
                    uint32_t out[BITS];
                    BitSink sink(out);
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        uint32_t h[8], cb[16];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            h[i] = pack_bf16x2(__uint_as_float(v[16 * g + 2 * i]),
                                               __uint_as_float(v[16 * g + 2 * i + 1]));
                        if (s >= 0x1p-96f) {
                            corrected_codes16(h, s, cb);
                        } else {
                            float f[16];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                f[2 * i] = bf16_lo(h[i]);
                                f[2 * i + 1] = bf16_hi(h[i]);
                            }
                            integer_codes_n<kQmax, 16>(f, s, cb);
                        }
#pragma unroll
                        for (int c8 = 0; c8 < 2; ++c8) {
                            uint32_t lo, hi;
                            pack_fields8<BITS>(cb + 8 * c8, lo, hi);
                            sink.put((static_cast<uint64_t>(hi) << 32) | lo, 8 * BITS);
                        }
                    }
                    if constexpr (BITS % 4 == 0) {
#pragma unroll
                        for (int i = 0; i < BITS; i += 4)
                            st_stream16(rec + cc * BITS + i,
                                        make_uint4(out[i], out[i + 1], out[i + 2], out[i + 3]));
                    } else {
#pragma unroll
                        for (int i = 0; i < BITS; ++i) rec[cc * BITS + i] = out[i];
                    }
                }
                scales[(size_t)row * rec_per_row + col0 / kBlock] = s;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank != 0)
                    mbar_arrive_remote(tempty0 + (uint32_t)buf * 8u);
                else
                    mbar_arrive(&tempty[buf]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Neither CTA of a pair frees TMEM or exits while the other may still
    // arrive on its barriers or have the pair's MMAs read its shared memory.
    cluster_sync_all();
    if (warp == kMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
    }
}

template <int BITS>
cudaError_t launch_bits(const void *x, const void *w, int T, int N, int K, void *y, void *codes,
                        float *scales, cudaStream_t st) {
    CUtensorMap m_x, m_w;
    if (!encode_2d(&m_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)T,
                   (uint64_t)K * 2, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&m_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, (uint64_t)K, (uint64_t)N,
                   (uint64_t)K * 2, 64, kBRows, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    auto kernel = fwd_gemm_quant_kernel<BITS>;
    static bool attr_set[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevices && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int num_tiles = ((T + kTileRows - 1) / kTileRows) * (N / BN);
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
    // persistent: as many pairs as can be resident at once
    static int resident[kMaxDevices];
    if (dev >= 0 && dev < kMaxDevices && resident[dev] == 0) {
        cfg.gridDim = dim3(sm_count() / kPair * kPair);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0)
            n = sm_count() / kPair;
        resident[dev] = n;
    }
    const int clusters = (dev >= 0 && dev < kMaxDevices) ? resident[dev] : sm_count() / kPair;
    cfg.gridDim = dim3((num_tiles < clusters ? num_tiles : clusters) * kPair);
    return cudaLaunchKernelEx(&cfg, kernel, m_x, m_w, T, N, K, static_cast<uint16_t *>(y),
                              static_cast<uint32_t *>(codes), scales);
}

}  // namespace

cudaError_t launch(const void *x, const void *w, int T, int N, int K, int bits, void *y,
                   void *codes, float *scales, cudaStream_t st) {
    switch (bits) {
        case 4: return launch_bits<4>(x, w, T, N, K, y, codes, scales, st);
        case 5: return launch_bits<5>(x, w, T, N, K, y, codes, scales, st);
        case 6: return launch_bits<6>(x, w, T, N, K, y, codes, scales, st);
        case 8: return launch_bits<8>(x, w, T, N, K, y, codes, scales, st);
        default: return cudaErrorInvalidValue;
    }
}

// Read and clear this instance's status word (the caller has synchronised).
cudaError_t read_and_clear_status(unsigned *status) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fwd_status, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof zero);
        if (e != cudaSuccess) return e;
    }
    *status = v;
    return cudaSuccess;
}

}  // namespace AGOQ_FWD_INSTANCE
}  // namespace agoq
