// fwd_gemm.cu -- a linear layer's forward GEMM with the LAAQ quantization of
// its output fused into the epilogue ("AGoQ: Activation and Gradient
// Quantization for Memory-Efficient Distributed Training of LLMs", section 2.C
// "Kernel Fusion": the quantization runs on the CUDA cores of the GEMM kernel;
// section 2.A: the activation kept for the backward pass is stored in b bits).
//
//   Y[t][n] = bf16(fl32(sum_k X[t][k] * W[n][k]))     X [T][K], W [N][K], BF16
//   codes, scales = LAAQ b-bit quantization of Y (128-column blocks of each row)
//
// Blackwell design (sm_103a), persistent, one CTA per SM, 128 x 256 output
// tiles with both operands K-major:
//   warp 0      TMA producer: per 64-deep k-block, a 128 x 64 tile of X and a
//               256 x 64 tile of W, 128-byte swizzled, into a 4-stage ring;
//   warp 1      TMEM owner and MMA issuer: 4 x tcgen05.mma kind::f16 (M=128,
//               N=256, K=16, both operands K-major) per k-block into one of two
//               256-column accumulators, so the epilogue of a tile overlaps the
//               mainloop of the next;
//   warps 2-5   epilogue: one output row per thread (its TMEM lane quarter is
//               warp % 4); per 128-column block, a first pass reads the
//               accumulator (tcgen05.ld), rounds it to BF16, stores Y and takes
//               the block absmax; a second pass reads it again, forms the codes
//               (corrected-reciprocal quotient, as the LAAQ quantizer) and
//               stores the packed record and the scale.
// Every mbarrier wait is time-limited (status word, CTA abort flag, drains).
#include "agoq_device.cuh"
#include "agoq_launch.h"
#include "gemm_common.cuh"

namespace agoq {

// Device-side status word of this kernel (read with the GEMM's by
// agoq_device_status).
__device__ unsigned g_fwd_status;

namespace {

using namespace gemm;

constexpr int BM = 128, BN = 256, BK = 64, NS = 4;
constexpr int kThreads = 192;
constexpr int kTmaWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kEpiWarps = 4;
constexpr int kAStage = BM * BK * 2;                      // 16 KiB
constexpr int kBStage = BN * BK * 2;                      // 32 KiB
constexpr int kOffB = NS * kAStage;
constexpr int kOffBar = kOffB + NS * kBStage;
constexpr int kNumBars = 2 * NS + 4 + 1;                  // full/empty, tmem full/empty x2, drain
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
static_assert(kSmemBytes <= 232448, "shared memory budget");

#ifndef AGOQ_FWD_BAND
#define AGOQ_FWD_BAND 16
#endif
#ifndef AGOQ_FWD_STREAM_STORES
#define AGOQ_FWD_STREAM_STORES 1
#endif

// Tile order: bands of kBand consecutive N-panels; within a band the tiles run
// N-fastest, then M, so the CTAs working at the same time share a few W panels
// and X row blocks (a working set that stays in L2).
constexpr int kBand = AGOQ_FWD_BAND;

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &m0, int &n0) {
    const int band = tile / (kBand * num_m);
    const int nb = min(kBand, num_n - band * kBand);            // panels in this band
    const int r = tile - band * kBand * num_m;
    m0 = (r / nb) * BM;
    n0 = (band * kBand + r % nb) * BN;
}

__device__ __forceinline__ void st_stream16(void *p, uint4 v) {
#if AGOQ_FWD_STREAM_STORES
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
#else
    *static_cast<uint4 *>(p) = v;
#endif
}

// kind::f16, BF16 A and B, FP32 D, both K-major, M = 128, N = 256.
constexpr uint32_t kIdescK = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                             ((uint32_t)(BM >> 4) << 24);

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
    uint64_t *full = bars, *empty = bars + NS, *tfull = bars + 2 * NS, *tempty = tfull + 2,
             *drain = tempty + 2;
    uint32_t *tmem_addr = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    unsigned *status = &g_fwd_status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_m = T / BM, num_n = N / BN, num_tiles = num_m * num_n, kblocks = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_addr)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_addr;

    if (warp == kTmaWarp) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int m0, n0;
                tile_coords(tile, num_m, num_n, m0, n0);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % NS;
                    if (!wait_bar(&empty[s], ((it / NS) & 1u) ^ 1u, abort, status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&full[s], kAStage + kBStage);
                    tma_load_2d(sa + s * kAStage, &map_x, &full[s], kb * BK, m0);
                    tma_load_2d(sb + s * kBStage, &map_w, &full[s], kb * BK, n0);
                }
            }
            for (int d = 0; d < NS && d < (int)it; ++d) {
                const uint32_t last = it - 1 - d;
                wait_bar(&full[last % NS], (last / NS) & 1u, abort, status, true);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            uint32_t it = 0, t = 0;
            bool ok = true, issued = false;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++t) {
                const int buf = t & 1;
                if (!wait_bar(&tempty[buf], ((t >> 1) & 1u) ^ 1u, abort, status)) break;
                tc_fence_after();
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const int s = it % NS;
                    if (!wait_bar(&full[s], (it / NS) & 1u, abort, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sa + s * kAStage), b0 = smem_u32(sb + s * kBStage);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(tmem_base + buf * BN, sw128_kmajor_desc(a0 + 32 * kk),
                                  sw128_kmajor_desc(b0 + 32 * kk), kIdescK,
                                  (kb > 0 || kk > 0) ? 1u : 0u);
                    issued = true;
                    umma_commit(&empty[s]);
                }
                if (!ok) break;
                umma_commit(&tfull[buf]);
            }
            if (issued) {
                umma_commit(drain);
                wait_bar(drain, 0u, abort, status, true);
            }
        }
    } else {
        // epilogue: TMEM lane quarter q = warp % 4, one output row per thread
        constexpr int kQmax = (1 << (BITS - 1)) - 1;
        const int q = warp & 3;
        const int rec_per_row = N / kBlock;
        uint32_t t = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++t) {
            const int buf = t & 1;
            if (!warp_wait(&tfull[buf], (t >> 1) & 1u, abort, status)) break;
            tc_fence_after();
            int m0, n0;
            tile_coords(tile, num_m, num_n, m0, n0);
            const int row = m0 + 32 * q + lane;
            const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + buf * BN;
#pragma unroll 1
            for (int jb = 0; jb < BN / kBlock; ++jb) {
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
            if (lane == 0) mbar_arrive(&tempty[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
    }
}

template <int BITS>
cudaError_t launch_bits(const void *x, const void *w, int T, int N, int K, void *y, void *codes,
                        float *scales, cudaStream_t st) {
    CUtensorMap m_x, m_w;
    if (!encode_2d(&m_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)T,
                   (uint64_t)K * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&m_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, (uint64_t)K, (uint64_t)N,
                   (uint64_t)K * 2, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
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
    const int num_tiles = (T / BM) * (N / BN);
    const int grid = num_tiles < sm_count() ? num_tiles : sm_count();
    kernel<<<grid, kThreads, kSmemBytes, st>>>(m_x, m_w, T, N, K, static_cast<uint16_t *>(y),
                                               static_cast<uint32_t *>(codes), scales);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_gemm_quant(const void *x, const void *w, int T, int N, int K, int bits,
                                  void *y, void *codes, float *scales, cudaStream_t st) {
    switch (bits) {
        case 4: return launch_bits<4>(x, w, T, N, K, y, codes, scales, st);
        case 5: return launch_bits<5>(x, w, T, N, K, y, codes, scales, st);
        case 6: return launch_bits<6>(x, w, T, N, K, y, codes, scales, st);
        case 8: return launch_bits<8>(x, w, T, N, K, y, codes, scales, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_and_clear_fwd_status(unsigned *status) {
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

}  // namespace agoq
