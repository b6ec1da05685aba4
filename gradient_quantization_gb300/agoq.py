"""Python binding of libagoq.so: argument marshalling only.

Every function has the name of the C entry point it calls (include/agoq.h) and
takes torch CUDA tensors; all arithmetic runs in the library's CUDA kernels.
Outputs that are not supplied are allocated with torch (device memory is the
caller's, as in the C ABI).  Calls are asynchronous on ``stream`` (default:
torch's current stream).  A non-zero status raises ``AgoqError``.

The library is built in-tree by ``python -m gradient_quantization_gb300.build``
(``__graft_entry__.build()`` does it too); importing a function without the
built library raises immediately -- there is no fallback implementation.
"""
import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libagoq.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "agoq.h")
BLOCK = 128

STATUS = {0: "AGOQ_OK", 1: "AGOQ_ERR_NULL", 2: "AGOQ_ERR_SHAPE", 3: "AGOQ_ERR_BITS",
          4: "AGOQ_ERR_ALIGN", 5: "AGOQ_ERR_ALIAS", 6: "AGOQ_ERR_CUDA", 7: "AGOQ_ERR_TIMEOUT",
          8: "AGOQ_ERR_FORMAT"}


class AgoqError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s" % (what, _lib_handle().agoq_status_string(status).decode()))


_L = None


def _lib_handle():
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libagoq.so is not built (%s); run "
                               "`python -m gradient_quantization_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.agoq_status_string.argtypes = [i32]
        L.agoq_status_string.restype = ctypes.c_char_p
        L.agoq_version.argtypes = []
        L.agoq_version.restype = i32
        L.agoq_quant_act.argtypes = [vp, i64, i32, vp, vp, vp]
        L.agoq_dequant_act.argtypes = [vp, vp, i64, i32, vp, vp]
        L.agoq_grad_accum_fp8.argtypes = [vp, vp, vp, i64, vp]
        L.agoq_silu_backward.argtypes = [vp, vp, vp, i64, i32, vp, vp, vp]
        L.agoq_rmsnorm_backward.argtypes = [vp, vp, vp, vp, i64, i64, i32, ctypes.c_float, vp,
                                            vp, vp, vp]
        L.agoq_rmsnorm_backward_ws.argtypes = [vp, vp, vp, vp, i64, i64, i32, ctypes.c_float, vp,
                                               vp, vp, vp, i64, vp]
        L.agoq_rmsnorm_backward_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i32, ctypes.c_float,
                                                    vp, vp, vp, vp]
        L.agoq_rmsnorm_backward_workspace_bytes.argtypes = [i64]
        L.agoq_rmsnorm_backward_workspace_bytes.restype = i64
        L.agoq_grad_accum_fp8_mid.argtypes = [vp, vp, vp, i64, i32, vp]
        L.agoq_reduce_fp8_shards.argtypes = [vp, vp, i32, i64, vp, vp, vp, vp]
        L.agoq_wgrad_gemm_int4.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        L.agoq_wgrad_gemm_int4_f32out.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        L.agoq_wgrad_gemm_int4_accum_fp8.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.agoq_device_status.argtypes = [vp]
        L.agoq_test_wait_timeout.argtypes = [i64, vp]
        L.agoq_dbca_pp_bits.argtypes = [i32, i32, i32, vp]
        L.agoq_fwd_gemm_quant.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
        for name in ("agoq_quant_act", "agoq_dequant_act", "agoq_grad_accum_fp8",
                     "agoq_reduce_fp8_shards", "agoq_wgrad_gemm_int4",
                     "agoq_wgrad_gemm_int4_f32out", "agoq_device_status",
                     "agoq_wgrad_gemm_int4_accum_fp8", "agoq_grad_accum_fp8_mid",
                     "agoq_silu_backward", "agoq_rmsnorm_backward", "agoq_rmsnorm_backward_ws",
                     "agoq_rmsnorm_backward_noalloc",
                     "agoq_dbca_pp_bits",
                     "agoq_fwd_gemm_quant", "agoq_test_wait_timeout"):
            getattr(L, name).restype = i32
        _L = L
    return _L


def lib():
    """The loaded ctypes library (raises if it is not built)."""
    return _lib_handle()


def declared_entry_points():
    """Names of the functions include/agoq.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:agoq_status|const char \*|int)\s*\*?\s*(agoq_\w+)\s*\(",
                                 text, flags=re.M)))


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, dtype, what):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % what)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (what, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)


def _check(rc, what):
    if rc != 0:
        raise AgoqError(rc, what)


def record_bytes(bits):
    """Bytes of one packed record of 128 codes of `bits` bits."""
    return 16 * bits


def agoq_quant_act(x, bits, codes=None, scales=None, stream=None):
    """LAAQ quantize BF16 `x` (any shape, numel % 128 == 0) -> (codes uint8, scales float32)."""
    _need(x, torch.bfloat16, "x")
    n = x.numel()
    if codes is None:
        codes = torch.empty(n // BLOCK * record_bytes(max(bits, 0)), dtype=torch.uint8,
                            device=x.device)
    if scales is None:
        scales = torch.empty(n // BLOCK, dtype=torch.float32, device=x.device)
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.float32, "scales")
    if bits in (4, 5, 6, 8) and (codes.numel() < n // BLOCK * record_bytes(bits)
                                 or scales.numel() < n // BLOCK):
        raise ValueError("codes/scales too small for %d elements at %d bits" % (n, bits))
    _check(lib().agoq_quant_act(_ptr(x), n, bits, _ptr(codes), _ptr(scales), _stream(stream)),
           "agoq_quant_act")
    return codes, scales


def agoq_dequant_act(codes, scales, n, bits, y=None, stream=None):
    """LAAQ dequantize -> BF16 tensor of n elements (or into `y`)."""
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.float32, "scales")
    if bits in (4, 5, 6, 8) and (codes.numel() < n // BLOCK * record_bytes(bits)
                                 or scales.numel() < n // BLOCK):
        raise ValueError("codes/scales too small for %d elements at %d bits" % (n, bits))
    if y is None:
        y = torch.empty(n, dtype=torch.bfloat16, device=codes.device)
    _need(y, torch.bfloat16, "y")
    if y.numel() < n:
        raise ValueError("y too small")
    _check(lib().agoq_dequant_act(_ptr(codes), _ptr(scales), n, bits, _ptr(y), _stream(stream)),
           "agoq_dequant_act")
    return y


def agoq_grad_accum_fp8(master, master_scales, grad, stream=None):
    """In-place QuanGrad accumulation of BF16 `grad` into the FP8 master (uint8 codes)."""
    _need(master, torch.uint8, "master")
    _need(master_scales, torch.float32, "master_scales")
    _need(grad, torch.bfloat16, "grad")
    n = grad.numel()
    if master.numel() != n or master_scales.numel() != n // BLOCK:
        raise ValueError("master/scales do not match the gradient size")
    _check(lib().agoq_grad_accum_fp8(_ptr(master), _ptr(master_scales), _ptr(grad), n,
                                     _stream(stream)), "agoq_grad_accum_fp8")
    return master, master_scales


def agoq_silu_backward(codes, scales, dy, n, bits, dx=None, y=None, want_y=False, stream=None):
    """SiLU backward recomputed from LAAQ codes: returns (dx, y) as BF16 tensors
    (y is None unless `y` is given or want_y is set)."""
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.float32, "scales")
    _need(dy, torch.bfloat16, "dy")
    if dx is None:
        dx = torch.empty(n, dtype=torch.bfloat16, device=dy.device)
    if y is None and want_y:
        y = torch.empty(n, dtype=torch.bfloat16, device=dy.device)
    _need(dx, torch.bfloat16, "dx")
    if y is not None:
        _need(y, torch.bfloat16, "y")
    _check(lib().agoq_silu_backward(_ptr(codes), _ptr(scales), _ptr(dy), n, bits, _ptr(dx),
                                    _ptr(y), _stream(stream)), "agoq_silu_backward")
    return dx, y


def agoq_rmsnorm_backward(codes, scales, dy, w, T, H, bits, eps, dx=None, rstd=None, dw=None,
                          want_dw=True, stream=None):
    """RMSNorm backward recomputed from LAAQ codes of x [T][H]: returns (dx BF16 [T][H],
    rstd FP32 [T], dw FP32 [H] or None)."""
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.float32, "scales")
    _need(dy, torch.bfloat16, "dy")
    _need(w, torch.bfloat16, "w")
    dev = dy.device
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if rstd is None:
        rstd = torch.empty(T, dtype=torch.float32, device=dev)
    if dw is None and want_dw:
        dw = torch.empty(H, dtype=torch.float32, device=dev)
    _check(lib().agoq_rmsnorm_backward(_ptr(codes), _ptr(scales), _ptr(dy), _ptr(w), T, H, bits,
                                       float(eps), _ptr(dx), _ptr(rstd), _ptr(dw),
                                       _stream(stream)), "agoq_rmsnorm_backward")
    return dx, rstd, dw


def agoq_rmsnorm_backward_workspace_bytes(H):
    """Bytes of scratch agoq_rmsnorm_backward_ws needs for rows of H elements."""
    return int(lib().agoq_rmsnorm_backward_workspace_bytes(int(H)))


def agoq_rmsnorm_backward_ws(codes, scales, dy, w, T, H, bits, eps, workspace, dx=None, rstd=None,
                             dw=None, stream=None):
    """The RMSNorm backward in one read of the input (H <= 4096), dw included; `workspace`
    is a CUDA tensor of at least agoq_rmsnorm_backward_workspace_bytes(H) bytes.
    Returns (dx, rstd, dw)."""
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.float32, "scales")
    _need(dy, torch.bfloat16, "dy")
    _need(w, torch.bfloat16, "w")
    dev = dy.device
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if rstd is None:
        rstd = torch.empty(T, dtype=torch.float32, device=dev)
    if dw is None:
        dw = torch.empty(H, dtype=torch.float32, device=dev)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().agoq_rmsnorm_backward_ws(_ptr(codes), _ptr(scales), _ptr(dy), _ptr(w), T, H, bits,
                                          float(eps), _ptr(dx), _ptr(rstd), _ptr(dw),
                                          _ptr(workspace), nbytes, _stream(stream)),
           "agoq_rmsnorm_backward_ws")
    return dx, rstd, dw


def agoq_rmsnorm_backward_noalloc(codes, scales, dy, w, T, H, bits, eps, dx, rstd, dw,
                                  stream=None):
    """agoq_rmsnorm_backward_ws with the library's own static scratch (H <= 4096), for
    callers that cannot allocate device memory at the call: every output is
    caller-provided and the call allocates nothing."""
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.float32, "scales")
    _need(dy, torch.bfloat16, "dy")
    _need(w, torch.bfloat16, "w")
    _check(lib().agoq_rmsnorm_backward_noalloc(_ptr(codes), _ptr(scales), _ptr(dy), _ptr(w), T, H,
                                               bits, float(eps), _ptr(dx), _ptr(rstd), _ptr(dw),
                                               _stream(stream)), "agoq_rmsnorm_backward_noalloc")
    return dx, rstd, dw


def agoq_dbca_pp_bits(stages, microbatches, base_bits=4):
    """DBCA-PP widths per pipeline stage (host-side): a list of `stages` ints."""
    out = (ctypes.c_int * max(int(stages), 1))()
    _check(lib().agoq_dbca_pp_bits(int(stages), int(microbatches), int(base_bits), out),
           "agoq_dbca_pp_bits")
    return list(out)[:stages]


def agoq_fwd_gemm_quant(x, w, T, N, K, bits, y=None, codes=None, scales=None, stream=None):
    """Forward GEMM Y = bf16(X W^T) (X [T][K], W [N][K], BF16) with the LAAQ
    quantization of Y fused: returns (Y [T][N], codes, scales)."""
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w")
    dev = x.device
    if y is None:
        y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    if codes is None:
        codes = torch.empty(T * N // BLOCK * record_bytes(bits), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(T * N // BLOCK, dtype=torch.float32, device=dev)
    _check(lib().agoq_fwd_gemm_quant(_ptr(x), _ptr(w), T, N, K, bits, _ptr(y), _ptr(codes),
                                     _ptr(scales), _stream(stream)), "agoq_fwd_gemm_quant")
    return y, codes, scales


MID_FP32, MID_BF16, MID_FP16 = 0, 1, 2


def agoq_grad_accum_fp8_mid(master, master_scales, grad, mid_format, stream=None):
    """In-place QuanGrad accumulation with the intermediate held in binary32
    (MID_FP32), BF16 (MID_BF16) or FP16 (MID_FP16)."""
    _need(master, torch.uint8, "master")
    _need(master_scales, torch.float32, "master_scales")
    _need(grad, torch.bfloat16, "grad")
    n = grad.numel()
    if master.numel() != n or master_scales.numel() != n // BLOCK:
        raise ValueError("master/scales do not match the gradient size")
    _check(lib().agoq_grad_accum_fp8_mid(_ptr(master), _ptr(master_scales), _ptr(grad), n,
                                         int(mid_format), _stream(stream)),
           "agoq_grad_accum_fp8_mid")
    return master, master_scales


def agoq_reduce_fp8_shards(shards, shard_scales, W, n, out=None, out_scales=None,
                           naive_overflow_count=None, stream=None):
    """Local reduce of W shard-major FP8 shards -> (codes, scales).  Pass a one-element
    int64 CUDA tensor as `naive_overflow_count` to receive the naive-sum overflow count."""
    _need(shards, torch.uint8, "shards")
    _need(shard_scales, torch.float32, "shard_scales")
    if shards.numel() != W * n or shard_scales.numel() != W * (n // BLOCK):
        raise ValueError("shards/shard_scales do not match W and n")
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=shards.device)
    if out_scales is None:
        out_scales = torch.empty(n // BLOCK, dtype=torch.float32, device=shards.device)
    _need(out, torch.uint8, "out")
    _need(out_scales, torch.float32, "out_scales")
    if naive_overflow_count is not None:
        _need(naive_overflow_count, torch.int64, "naive_overflow_count")
    _check(lib().agoq_reduce_fp8_shards(_ptr(shards), _ptr(shard_scales), W, n, _ptr(out),
                                        _ptr(out_scales), _ptr(naive_overflow_count),
                                        _stream(stream)), "agoq_reduce_fp8_shards")
    return out, out_scales


def agoq_wgrad_gemm_int4(dY, x_codes, x_scales, M, N, K, dW=None, stream=None):
    """dW[M][N] (BF16) = dY^T Xhat for dY BF16 [K][M] and LAAQ INT4 X (codes [K][N/2])."""
    _need(dY, torch.bfloat16, "dY")
    _need(x_codes, torch.uint8, "x_codes")
    _need(x_scales, torch.float32, "x_scales")
    if dW is None:
        dW = torch.empty((M, N), dtype=torch.bfloat16, device=dY.device)
    _need(dW, torch.bfloat16, "dW")
    _check(lib().agoq_wgrad_gemm_int4(_ptr(dY), _ptr(x_codes), _ptr(x_scales), M, N, K, _ptr(dW),
                                      _stream(stream)), "agoq_wgrad_gemm_int4")
    return dW


def agoq_wgrad_gemm_int4_f32out(dY, x_codes, x_scales, M, N, K, dW=None, stream=None):
    """The same GEMM with the FP32 accumulator as output."""
    _need(dY, torch.bfloat16, "dY")
    _need(x_codes, torch.uint8, "x_codes")
    _need(x_scales, torch.float32, "x_scales")
    if dW is None:
        dW = torch.empty((M, N), dtype=torch.float32, device=dY.device)
    _need(dW, torch.float32, "dW")
    _check(lib().agoq_wgrad_gemm_int4_f32out(_ptr(dY), _ptr(x_codes), _ptr(x_scales), M, N, K,
                                             _ptr(dW), _stream(stream)),
           "agoq_wgrad_gemm_int4_f32out")
    return dW


def agoq_wgrad_gemm_int4_accum_fp8(dY, x_codes, x_scales, M, N, K, master, master_scales,
                                   stream=None):
    """The GEMM with the QuanGrad accumulation as its epilogue: the product is
    added to the FP8 master [M][N] (uint8 E4M3 codes, float32 scales [M][N/128])
    in place.  Returns (master, master_scales)."""
    _need(dY, torch.bfloat16, "dY")
    _need(x_codes, torch.uint8, "x_codes")
    _need(x_scales, torch.float32, "x_scales")
    _need(master, torch.uint8, "master")
    _need(master_scales, torch.float32, "master_scales")
    _check(lib().agoq_wgrad_gemm_int4_accum_fp8(_ptr(dY), _ptr(x_codes), _ptr(x_scales), M, N, K,
                                                _ptr(master), _ptr(master_scales),
                                                _stream(stream)),
           "agoq_wgrad_gemm_int4_accum_fp8")
    return master, master_scales


def agoq_test_wait_timeout(limit_cycles, stream=None):
    """Launch the failure-path probe whose one pipeline wait gives up after
    `limit_cycles` SM cycles (test-only; see include/agoq.h)."""
    _check(lib().agoq_test_wait_timeout(int(limit_cycles), _stream(stream)),
           "agoq_test_wait_timeout")


def agoq_device_status(stream=None):
    """Synchronise and check the device status words (raises AgoqError if a pipeline wait timed out)."""
    _check(lib().agoq_device_status(_stream(stream)), "agoq_device_status")
