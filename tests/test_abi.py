"""The C-ABI library loads, exports every entry point include/agoq.h declares,
and rejects bad arguments on the host before any CUDA call (so these run
without a GPU: every call below fails validation and launches nothing)."""
import ctypes
import subprocess

import pytest

from gradient_quantization_gb300 import agoq

OK, NULL, SHAPE, BITS, ALIGN, ALIAS = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def L():
    return agoq.lib()


def test_every_declared_entry_point_is_exported(L):
    names = agoq.declared_entry_points()
    assert len(names) >= 9
    for name in names:
        assert hasattr(L, name), name


def test_exports_are_c_symbols():
    out = subprocess.run(["nm", "-D", "--defined-only", agoq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in agoq.declared_entry_points():
        assert name in syms, name


def test_status_strings(L):
    for code in range(9):
        s = L.agoq_status_string(code).decode()
        assert s.startswith(agoq.STATUS[code])
    assert L.agoq_status_string(99).decode() == "AGOQ_ERR_UNKNOWN"
    assert L.agoq_version() >= 100


P = ctypes.c_void_p
A = 0x10000000          # fake, 16-byte-aligned addresses: never dereferenced on these paths
B = 0x20000000
C = 0x30000000


def test_quant_act_validation(L):
    assert L.agoq_quant_act(P(A), 256, 7, P(B), P(C), None) == BITS
    assert L.agoq_quant_act(P(A), 100, 4, P(B), P(C), None) == SHAPE
    assert L.agoq_quant_act(P(A), -128, 4, P(B), P(C), None) == SHAPE
    assert L.agoq_quant_act(P(A), 0, 4, None, None, None) == OK          # empty: no-op
    assert L.agoq_quant_act(None, 256, 4, P(B), P(C), None) == NULL
    assert L.agoq_quant_act(P(A + 2), 256, 4, P(B), P(C), None) == ALIGN
    assert L.agoq_quant_act(P(A), 256, 4, P(B + 8), P(C), None) == ALIGN
    assert L.agoq_quant_act(P(A), 256, 4, P(B), P(C + 2), None) == ALIGN
    # codes overlapping the input
    assert L.agoq_quant_act(P(A), 256, 4, P(A + 256), P(C), None) == ALIAS
    # scales overlapping the codes (2 blocks * 64 bytes)
    assert L.agoq_quant_act(P(A), 256, 4, P(B), P(B + 64), None) == ALIAS


def test_dequant_act_validation(L):
    assert L.agoq_dequant_act(P(A), P(B), 256, 3, P(C), None) == BITS
    assert L.agoq_dequant_act(P(A), P(B), 130, 4, P(C), None) == SHAPE
    assert L.agoq_dequant_act(P(A), None, 256, 4, P(C), None) == NULL
    assert L.agoq_dequant_act(P(A), P(B), 256, 4, P(C + 4), None) == ALIGN
    assert L.agoq_dequant_act(P(A), P(B), 256, 4, P(A), None) == ALIAS
    assert L.agoq_dequant_act(P(A), P(B), 0, 8, P(C), None) == OK


def test_grad_accum_validation(L):
    assert L.agoq_grad_accum_fp8(P(A), P(B), P(C), 127, None) == SHAPE
    assert L.agoq_grad_accum_fp8(None, P(B), P(C), 128, None) == NULL
    assert L.agoq_grad_accum_fp8(P(A + 1), P(B), P(C), 128, None) == ALIGN
    assert L.agoq_grad_accum_fp8(P(A), P(B), P(A + 64), 128, None) == ALIAS
    assert L.agoq_grad_accum_fp8(P(A), P(B), P(C), 0, None) == OK


def test_silu_backward_validation(L):
    fn = L.agoq_silu_backward
    D = C + (1 << 20)
    assert fn(P(A), P(B), P(C), 256, 3, P(D), None, None) == BITS
    assert fn(P(A), P(B), P(C), 200, 4, P(D), None, None) == SHAPE
    assert fn(P(A), P(B), P(C), 0, 4, None, None, None) == OK
    assert fn(P(A), None, P(C), 256, 4, P(D), None, None) == NULL
    assert fn(P(A), P(B), P(C), 256, 4, None, None, None) == NULL
    assert fn(P(A), P(B), P(C + 2), 256, 4, P(D), None, None) == ALIGN
    assert fn(P(A), P(B), P(C), 256, 4, P(D), P(D + 8 + 4096), None) == ALIGN
    assert fn(P(A), P(B), P(C), 256, 4, P(C + 256), None, None) == ALIAS     # dx on dy
    assert fn(P(A), P(B), P(C), 256, 4, P(D), P(D + 256), None) == ALIAS     # y on dx
    assert fn(P(A), P(B), P(C), 256, 4, P(D), P(A), None) == ALIAS           # y on codes


def test_rmsnorm_backward_validation(L):
    fn = L.agoq_rmsnorm_backward
    f = ctypes.c_float
    D, E, F = C + (1 << 20), C + (1 << 22), C + (1 << 23)
    args = lambda T, H, bits, eps=1e-6: (P(A), P(B), P(C), P(C + (1 << 19)), T, H, bits, f(eps))
    assert fn(*args(4, 256, 7), P(D), P(E), P(F), None) == BITS
    assert fn(*args(4, 384, 4), P(D), P(E), P(F), None) == SHAPE       # H % 256
    assert fn(*args(4, 8448, 4), P(D), P(E), P(F), None) == SHAPE      # H > 8192
    assert fn(*args(4, 256, 4, -1.0), P(D), P(E), P(F), None) == SHAPE
    assert fn(*args(4, 256, 4, float("nan")), P(D), P(E), P(F), None) == SHAPE
    assert fn(*args(0, 256, 4), P(D), P(E), None, None) == OK
    assert fn(*args(4, 256, 4), None, P(E), P(F), None) == NULL
    assert fn(*args(4, 256, 4), P(D), None, P(F), None) == NULL
    assert fn(*args(4, 256, 4), P(D + 8), P(E), P(F), None) == ALIGN
    assert fn(*args(4, 256, 4), P(C), P(E), P(F), None) == ALIAS         # dx on dy
    assert fn(*args(4, 256, 4), P(D), P(D + 64), P(F), None) == ALIAS    # rstd inside dx
    assert fn(*args(4, 256, 4), P(D), P(E), P(A), None) == ALIAS         # dw on codes


def test_rmsnorm_workspace_bytes_and_ws_validation(L):
    """The single-read backward's scratch size and its argument checks, which
    return before any launch."""
    wb = L.agoq_rmsnorm_backward_workspace_bytes
    assert wb(4096) == 304 * 4096 * 4 and wb(256) == 304 * 256 * 4
    assert wb(4352) == 0 and wb(8192) == 0                    # H > 4096: the two-pass path
    assert wb(100) == -1 and wb(0) == -1 and wb(8448) == -1
    fn = L.agoq_rmsnorm_backward_ws
    f = ctypes.c_float
    D, E, F, W = C + (1 << 20), C + (1 << 22), C + (1 << 23), C + (1 << 26)
    need = wb(256)
    args = lambda T, H, bits, eps=1e-6: (P(A), P(B), P(C), P(C + (1 << 19)), T, H, bits, f(eps))
    assert fn(*args(4, 256, 7), P(D), P(E), P(F), P(W), need, None) == BITS
    assert fn(*args(4, 384, 4), P(D), P(E), P(F), P(W), need, None) == SHAPE   # H % 256
    assert fn(*args(4, 256, 4), P(D), P(E), P(F), P(W), need - 4, None) == SHAPE
    assert fn(*args(4, 256, 4), P(D), P(E), None, P(W), need, None) == NULL    # dw required
    assert fn(*args(4, 256, 4), P(D), P(E), P(F), None, need, None) == NULL
    assert fn(*args(4, 256, 4), P(D), P(E), P(F), P(W + 8), need, None) == ALIGN
    assert fn(*args(4, 256, 4), P(D), P(E), P(F), P(D), need, None) == ALIAS    # scratch on dx
    assert fn(*args(4, 256, 4), P(D), P(E), P(F), P(A), need, None) == ALIAS    # scratch on codes


def test_grad_accum_mid_validation(L):
    FORMAT = 8
    fn = L.agoq_grad_accum_fp8_mid
    assert fn(P(A), P(B), P(C), 128, 3, None) == FORMAT
    assert fn(P(A), P(B), P(C), 128, -1, None) == FORMAT
    assert fn(P(A), P(B), P(C), 127, 1, None) == SHAPE
    assert fn(None, P(B), P(C), 128, 2, None) == NULL
    assert fn(P(A + 1), P(B), P(C), 128, 1, None) == ALIGN
    assert fn(P(A), P(B), P(A + 64), 128, 2, None) == ALIAS
    for mid in (0, 1, 2):
        assert fn(P(A), P(B), P(C), 0, mid, None) == OK


def test_reduce_validation(L):
    assert L.agoq_reduce_fp8_shards(P(A), P(B), 0, 128, P(C), P(C + 4096), None, None) == SHAPE
    assert L.agoq_reduce_fp8_shards(P(A), P(B), 2, 200, P(C), P(C + 4096), None, None) == SHAPE
    assert L.agoq_reduce_fp8_shards(P(A), None, 2, 128, P(C), P(C + 4096), None, None) == NULL
    assert L.agoq_reduce_fp8_shards(P(A), P(B), 2, 128, P(C + 8), P(C + 4096), None, None) == ALIGN
    assert L.agoq_reduce_fp8_shards(P(A), P(B), 2, 128, P(C), P(C + 4096), P(C + 4100), None) == ALIGN
    # output inside the second shard
    assert L.agoq_reduce_fp8_shards(P(A), P(B), 2, 128, P(A + 128), P(C), None, None) == ALIAS
    # count overlapping the output scales
    assert L.agoq_reduce_fp8_shards(P(A), P(B), 2, 128, P(C), P(C + 4096), P(C + 4096), None) == ALIAS
    assert L.agoq_reduce_fp8_shards(P(A), P(B), 2, 0, P(C), P(C), None, None) == OK


def test_gemm_validation(L):
    for fn in (L.agoq_wgrad_gemm_int4, L.agoq_wgrad_gemm_int4_f32out):
        # M and N multiples of 128, K of 64
        assert fn(P(A), P(B), P(C), 100, 512, 64, P(C + (1 << 24)), None) == SHAPE
        assert fn(P(A), P(B), P(C), 256, 192, 64, P(C + (1 << 24)), None) == SHAPE
        assert fn(P(A), P(B), P(C), 256, 512, 32, P(C + (1 << 24)), None) == SHAPE
        assert fn(P(A), P(B), P(C), 0, 512, 64, P(C + (1 << 24)), None) == SHAPE
        assert fn(None, P(B), P(C), 256, 512, 64, P(C + (1 << 24)), None) == NULL
        # scales need 4-byte alignment, the other pointers 16
        assert fn(P(A), P(B), P(C + 2), 256, 512, 64, P(C + (1 << 24)), None) == ALIGN
        assert fn(P(A + 8), P(B), P(C), 256, 512, 64, P(C + (1 << 24)), None) == ALIGN
        assert fn(P(A), P(B), P(C), 256, 512, 64, P(A), None) == ALIAS


def test_gemm_accum_validation(L):
    fn = L.agoq_wgrad_gemm_int4_accum_fp8
    D = C + (1 << 24)
    E = C + (1 << 26)
    assert fn(P(A), P(B), P(C), 100, 512, 64, P(D), P(E), None) == SHAPE
    assert fn(P(A), P(B), P(C), 384, 320, 64, P(D), P(E), None) == SHAPE
    assert fn(P(A), P(B), P(C), 256, 512, 0, P(D), P(E), None) == SHAPE
    assert fn(P(A), P(B), P(C), 256, 512, 64, None, P(E), None) == NULL
    assert fn(P(A), P(B), P(C), 256, 512, 64, P(D), None, None) == NULL
    assert fn(P(A), P(B), P(C), 256, 512, 64, P(D + 8), P(E), None) == ALIGN
    assert fn(P(A), P(B), P(C), 256, 512, 64, P(D), P(E + 2), None) == ALIGN
    assert fn(P(A), P(B), P(C), 256, 512, 64, P(A), P(E), None) == ALIAS       # master on dY
    assert fn(P(A), P(B), P(C), 256, 512, 64, P(D), P(B), None) == ALIAS       # scales on codes
    assert fn(P(A), P(B), P(C), 256, 512, 64, P(D), P(D + 4096), None) == ALIAS


def test_fwd_gemm_quant_validation(L):
    fn = L.agoq_fwd_gemm_quant
    D, E, F = C + (1 << 24), C + (1 << 26), C + (1 << 27)
    assert fn(P(A), P(B), 128, 256, 64, 3, P(D), P(E), P(F), None) == BITS
    assert fn(P(A), P(B), 100, 256, 64, 4, P(D), P(E), P(F), None) == SHAPE
    assert fn(P(A), P(B), 128, 128, 64, 4, P(D), P(E), P(F), None) == SHAPE
    assert fn(P(A), P(B), 128, 256, 48, 4, P(D), P(E), P(F), None) == SHAPE
    assert fn(P(A), None, 128, 256, 64, 4, P(D), P(E), P(F), None) == NULL
    assert fn(P(A), P(B), 128, 256, 64, 4, P(D + 2), P(E), P(F), None) == ALIGN
    assert fn(P(A), P(B), 128, 256, 64, 4, P(A), P(E), P(F), None) == ALIAS      # y on x
    assert fn(P(A), P(B), 128, 256, 64, 4, P(D), P(D + 256), P(F), None) == ALIAS


def test_wait_timeout_probe_validation(L):
    fn = L.agoq_test_wait_timeout
    assert fn(0, None) == SHAPE
    assert fn(-5, None) == SHAPE
    assert fn(4000000001, None) == SHAPE


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(agoq, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(agoq, "_L", None)
    with pytest.raises(RuntimeError, match="not built"):
        agoq.lib()
