"""ctypes front end of the CPU oracle (TEST INFRASTRUCTURE, not the product).

Only tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg import
this module.  It builds ``libagoq_oracle.so`` from ``agoq_oracle.c`` on first
use and exposes each oracle function over numpy arrays.  Arrays of BF16 values
are carried as ``numpy.uint16`` bit patterns and FP8 E4M3 values as
``numpy.uint8`` codes, so no library cast is involved on the oracle side.

What each function computes, and the section of "AGoQ: Activation and Gradient
Quantization for Memory-Efficient Distributed Training of LLMs" it restates, is
documented in ``agoq_oracle.c``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

BLOCK = 128

_libs = {}


def lib(parallel=False):
    """Load (building first if needed) the oracle shared library: the
    single-threaded build, or with ``parallel`` the all-core (OpenMP) build of
    the same source, which computes the same bits."""
    key = bool(parallel)
    if key not in _libs:
        path = _build.build()
        if parallel:
            path = _build.build_omp()
            if path is None:
                raise RuntimeError("the all-core oracle build is not available (no OpenMP)")
        L = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.or_quant_act.argtypes = [vp, i64, i32, vp, vp]
        L.or_dequant_act.argtypes = [vp, vp, i64, i32, vp]
        L.or_grad_accum_fp8.argtypes = [vp, vp, vp, i64]
        L.or_reduce_fp8_shards.argtypes = [vp, vp, i32, i64, vp, vp, vp]
        L.or_wgrad_gemm_int4_f64.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.or_wgrad_gemm_int4_f64_entries.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, i64, vp]
        L.or_grad_accum_fp8_f32.argtypes = [vp, vp, vp, i64]
        L.or_grad_accum_fp8_mid.argtypes = [vp, vp, vp, i64, i32]
        L.or_silu_backward.argtypes = [vp, vp, vp, i64, i32, vp, vp]
        L.or_fwd_gemm_quant.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
        L.or_rmsnorm_backward.argtypes = [vp, vp, vp, vp, i64, i64, i32, ctypes.c_double, vp, vp,
                                          vp]
        L.or_round_format_array.argtypes = [vp, vp, i64, i32, i32, i32]
        L.or_wgrad_accum_fp8.argtypes = [vp, vp, vp, i32, i32, i32, vp, i64, vp, vp]
        L.or_f32_to_bf16_array.argtypes = [vp, vp, i64]
        L.or_f32_to_e4m3_array.argtypes = [vp, vp, i64]
        L.or_e4m3_to_f32_array.argtypes = [vp, vp, i64]
        L.or_threads.argtypes = []
        for name in ("or_quant_act", "or_dequant_act", "or_grad_accum_fp8",
                     "or_reduce_fp8_shards", "or_wgrad_gemm_int4_f64",
                     "or_wgrad_gemm_int4_f64_entries", "or_grad_accum_fp8_f32",
                     "or_wgrad_accum_fp8", "or_grad_accum_fp8_mid", "or_silu_backward",
                     "or_rmsnorm_backward", "or_fwd_gemm_quant", "or_threads"):
            getattr(L, name).restype = ctypes.c_int
        for name in ("or_f32_to_bf16_array", "or_f32_to_e4m3_array", "or_e4m3_to_f32_array",
                     "or_round_format_array"):
            getattr(L, name).restype = None
        _libs[key] = L
    return _libs[key]


def parallel_available():
    """Whether the all-core build could be made."""
    return _build.build_omp() is not None


def threads(parallel=False):
    """Threads the oracle's loops use (1 for the single-threaded build)."""
    return int(lib(parallel).or_threads())


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _contig(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, a.dtype))
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError("oracle %s rejected its arguments (code %d)" % (what, rc))


def record_bytes(bits):
    """Bytes of one packed block record of 128 b-bit codes."""
    return 16 * bits


# --- codecs --------------------------------------------------------------
def f32_to_bf16(x):
    x = _contig(np.asarray(x, dtype=np.float32), np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().or_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f32(h):
    h = _contig(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def f32_to_e4m3(x):
    x = _contig(np.asarray(x, dtype=np.float32), np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().or_f32_to_e4m3_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_to_f32(c):
    c = _contig(c, np.uint8)
    out = np.empty(c.shape, np.float32)
    lib().or_e4m3_to_f32_array(_ptr(c), _ptr(out), c.size)
    return out


# --- the path ------------------------------------------------------------
def quant_act(x_bf16, bits, parallel=False):
    """LAAQ quantize: BF16 bit patterns [n] -> (codes uint8 [n/128*16*bits], scales f32 [n/128])."""
    x = _contig(x_bf16, np.uint16).reshape(-1)
    n = x.size
    codes = np.empty(n // BLOCK * record_bytes(bits), np.uint8)
    scales = np.empty(n // BLOCK, np.float32)
    _check(lib(parallel).or_quant_act(_ptr(x), n, bits, _ptr(codes), _ptr(scales)), "quant_act")
    return codes, scales


def dequant_act(codes, scales, n, bits, parallel=False):
    """LAAQ dequantize: packed codes + scales -> BF16 bit patterns [n]."""
    codes = _contig(codes, np.uint8).reshape(-1)
    scales = _contig(scales, np.float32).reshape(-1)
    if codes.size < n // BLOCK * record_bytes(bits) or scales.size < n // BLOCK:
        raise ValueError("codes/scales too short for n")
    y = np.empty(n, np.uint16)
    _check(lib(parallel).or_dequant_act(_ptr(codes), _ptr(scales), n, bits, _ptr(y)), "dequant_act")
    return y


def grad_accum_fp8(master, master_scales, grad_bf16, parallel=False, in_place=False):
    """QuanGrad local accumulation; returns new (master, scales), inputs untouched
    (with ``in_place`` the contiguous uint8/float32 arrays given are updated and
    returned)."""
    m = _contig(master, np.uint8).reshape(-1)
    s = _contig(master_scales, np.float32).reshape(-1)
    if not in_place:
        m, s = m.copy(), s.copy()
    g = _contig(grad_bf16, np.uint16).reshape(-1)
    if g.size != m.size or s.size != m.size // BLOCK:
        raise ValueError("shape mismatch")
    _check(lib(parallel).or_grad_accum_fp8(_ptr(m), _ptr(s), _ptr(g), m.size), "grad_accum_fp8")
    return m, s


def reduce_fp8_shards(shards, shard_scales, W, n, count_naive=True, parallel=False):
    """Local reduce over W shard-major shards; returns (codes, scales, naive_overflow or None)."""
    sh = _contig(shards, np.uint8).reshape(-1)
    ss = _contig(shard_scales, np.float32).reshape(-1)
    if sh.size != W * n or ss.size != W * (n // BLOCK):
        raise ValueError("shape mismatch")
    out = np.empty(n, np.uint8)
    outs = np.empty(n // BLOCK, np.float32)
    cnt = np.zeros(1, np.uint64)
    _check(lib(parallel).or_reduce_fp8_shards(_ptr(sh), _ptr(ss), W, n, _ptr(out), _ptr(outs),
                                       _ptr(cnt) if count_naive else None),
           "reduce_fp8_shards")
    return out, outs, (int(cnt[0]) if count_naive else None)


def wgrad_gemm_int4_f64(dY_bf16, x_codes, x_scales, M, N, K):
    """Binary64 dW [M][N] = dY^T Xhat for dY BF16 [K][M] and LAAQ INT4 X [K][N]."""
    dY = _contig(dY_bf16, np.uint16).reshape(-1)
    xc = _contig(x_codes, np.uint8).reshape(-1)
    xs = _contig(x_scales, np.float32).reshape(-1)
    if dY.size != K * M or xc.size != K * N // 2 or xs.size != K * N // BLOCK:
        raise ValueError("shape mismatch")
    out = np.empty((M, N), np.float64)
    _check(lib().or_wgrad_gemm_int4_f64(_ptr(dY), _ptr(xc), _ptr(xs), M, N, K, _ptr(out)),
           "wgrad_gemm_int4_f64")
    return out


def wgrad_gemm_int4_f64_matmul(dY_bf16, x_codes, x_scales, M, N, K, absolute=False):
    """The binary64 product dW = dY^T Xhat [M][N] for full-size shapes: Xhat is the
    oracle's own LAAQ 4-bit dequantization (dequant_act, BF16) of X, both operands
    are widened to binary64 and a library binary64 matrix product forms the sums
    (any summation order: the binary64 rounding error, about 1e-16 relative, is
    far below every tolerance it serves).  With ``absolute`` the product of the
    absolute values, sum_k |dY[k][i]| |Xhat[k][j]|, the scale of the binary32
    summation error bound."""
    dY = _contig(dY_bf16, np.uint16).reshape(K, M)
    xh = dequant_act(x_codes, x_scales, K * N, 4, parallel=parallel_available()).reshape(K, N)
    a = bf16_to_f32(dY).astype(np.float64)
    b = bf16_to_f32(xh).astype(np.float64)
    if absolute:
        np.abs(a, out=a)
        np.abs(b, out=b)
    return a.T @ b


def wgrad_gemm_int4_f64_entries(dY_bf16, x_codes, x_scales, M, N, K, rows, cols, parallel=False):
    """Binary64 entries dW[rows[e], cols[e]] of the same product."""
    dY = _contig(dY_bf16, np.uint16).reshape(-1)
    xc = _contig(x_codes, np.uint8).reshape(-1)
    xs = _contig(x_scales, np.float32).reshape(-1)
    r = _contig(np.asarray(rows, np.int32), np.int32)
    c = _contig(np.asarray(cols, np.int32), np.int32)
    out = np.empty(r.size, np.float64)
    _check(lib(parallel).or_wgrad_gemm_int4_f64_entries(_ptr(dY), _ptr(xc), _ptr(xs), M, N, K,
                                                _ptr(r), _ptr(c), r.size, _ptr(out)),
           "wgrad_gemm_int4_f64_entries")
    return out


def grad_accum_fp8_f32(master, master_scales, grad_f32):
    """QuanGrad accumulation of a binary32 gradient; returns new (master, scales)."""
    m = _contig(master, np.uint8).reshape(-1).copy()
    s = _contig(master_scales, np.float32).reshape(-1).copy()
    g = _contig(grad_f32, np.float32).reshape(-1)
    if g.size != m.size or s.size != m.size // BLOCK:
        raise ValueError("shape mismatch")
    _check(lib().or_grad_accum_fp8_f32(_ptr(m), _ptr(s), _ptr(g), m.size), "grad_accum_fp8_f32")
    return m, s


def wgrad_accum_fp8(dY_bf16, x_codes, x_scales, M, N, K, master, master_scales, blocks=None):
    """The product dY^T Xhat accumulated into an FP8 master [M][N]; returns new
    (master, scales).  With `blocks` (indices of 128-element blocks of the flat
    master) only those blocks are computed: master/master_scales then hold just
    them ([len(blocks)][128] and [len(blocks)])."""
    dY = _contig(dY_bf16, np.uint16).reshape(-1)
    xc = _contig(x_codes, np.uint8).reshape(-1)
    xs = _contig(x_scales, np.float32).reshape(-1)
    if dY.size != K * M or xc.size != K * N // 2 or xs.size != K * N // BLOCK:
        raise ValueError("shape mismatch")
    m = _contig(master, np.uint8).reshape(-1).copy()
    s = _contig(master_scales, np.float32).reshape(-1).copy()
    if blocks is None:
        b, count, nblk = None, 0, M * N // BLOCK
    else:
        b = _contig(np.asarray(blocks, np.int64), np.int64)
        count = nblk = b.size
    if m.size != nblk * BLOCK or s.size != nblk:
        raise ValueError("shape mismatch")
    _check(lib().or_wgrad_accum_fp8(_ptr(dY), _ptr(xc), _ptr(xs), M, N, K,
                                    _ptr(b) if b is not None else None, count, _ptr(m), _ptr(s)),
           "wgrad_accum_fp8")
    return m, s


MID_BF16, MID_FP16 = 1, 2
_FORMATS = {MID_BF16: (8, -126, 127), MID_FP16: (11, -14, 15)}


def round_format(x, mid):
    """Round binary64 values to BF16 (mid=1) or FP16 (mid=2), to nearest even; returns float64."""
    src = _contig(np.asarray(x, np.float64), np.float64).reshape(-1)
    dst = np.empty_like(src)
    p, emin, emax = _FORMATS[mid]
    lib().or_round_format_array(_ptr(src), _ptr(dst), src.size, p, emin, emax)
    return dst


def grad_accum_fp8_mid(master, master_scales, grad_bf16, mid):
    """QuanGrad accumulation with a BF16 (mid=1) or FP16 (mid=2) intermediate."""
    m = _contig(master, np.uint8).reshape(-1).copy()
    s = _contig(master_scales, np.float32).reshape(-1).copy()
    g = _contig(grad_bf16, np.uint16).reshape(-1)
    if g.size != m.size or s.size != m.size // BLOCK:
        raise ValueError("shape mismatch")
    _check(lib().or_grad_accum_fp8_mid(_ptr(m), _ptr(s), _ptr(g), m.size, mid), "grad_accum_fp8_mid")
    return m, s


def silu_backward(codes, scales, dy_bf16, n, bits, want_y=True):
    """SiLU backward recomputed from LAAQ codes: (dx, y) in binary64 (y None if not wanted)."""
    codes = _contig(codes, np.uint8).reshape(-1)
    scales = _contig(scales, np.float32).reshape(-1)
    dy = _contig(dy_bf16, np.uint16).reshape(-1)
    if codes.size < n // BLOCK * record_bytes(bits) or scales.size < n // BLOCK or dy.size != n:
        raise ValueError("shape mismatch")
    dx = np.empty(n, np.float64)
    y = np.empty(n, np.float64) if want_y else None
    _check(lib().or_silu_backward(_ptr(codes), _ptr(scales), _ptr(dy), n, bits, _ptr(dx),
                                  _ptr(y) if want_y else None), "silu_backward")
    return dx, y


def rmsnorm_backward(codes, scales, dy_bf16, w_bf16, T, H, bits, eps):
    """RMSNorm backward recomputed from LAAQ codes of x [T][H]: (dx [T][H], rstd [T],
    dw [H]) in binary64."""
    codes = _contig(codes, np.uint8).reshape(-1)
    scales = _contig(scales, np.float32).reshape(-1)
    dy = _contig(dy_bf16, np.uint16).reshape(-1)
    w = _contig(w_bf16, np.uint16).reshape(-1)
    n = T * H
    if (codes.size < n // BLOCK * record_bytes(bits) or scales.size < n // BLOCK or dy.size != n
            or w.size != H):
        raise ValueError("shape mismatch")
    dx = np.empty((T, H), np.float64)
    rstd = np.empty(T, np.float64)
    dw = np.empty(H, np.float64)
    _check(lib().or_rmsnorm_backward(_ptr(codes), _ptr(scales), _ptr(dy), _ptr(w), T, H, bits,
                                     float(eps), _ptr(dx), _ptr(rstd), _ptr(dw)),
           "rmsnorm_backward")
    return dx, rstd, dw


def fwd_gemm_quant(x_bf16, w_bf16, T, N, K, bits):
    """Forward product Y = bf16(fl32(X W^T)) (X [T][K], W [N][K], BF16 bits) and its
    LAAQ quantization: returns (Y bits [T][N], codes, scales)."""
    x = _contig(x_bf16, np.uint16).reshape(-1)
    w = _contig(w_bf16, np.uint16).reshape(-1)
    if x.size != T * K or w.size != N * K:
        raise ValueError("shape mismatch")
    y = np.empty(T * N, np.uint16)
    codes = np.empty(T * N // BLOCK * record_bytes(bits), np.uint8)
    scales = np.empty(T * N // BLOCK, np.float32)
    _check(lib().or_fwd_gemm_quant(_ptr(x), _ptr(w), T, N, K, bits, _ptr(y), _ptr(codes),
                                   _ptr(scales)), "fwd_gemm_quant")
    return y.reshape(T, N), codes, scales
