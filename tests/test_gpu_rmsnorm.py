"""GPU parity of the RMSNorm backward recomputed from LAAQ codes
(agoq_rmsnorm_backward) against the oracle's binary64 values.

Bounds (per element, from the binary32 operations the kernels perform):
r = rstd within dr = (H/2 + 8) * 2^-24 relative; dx within half a BF16 ulp plus
|r g|(dr + 2^-22) + |xh| r^3 (|c|(3 dr + 2^-21) + (H+1) 2^-24 S/H) + 2^-23 |dx|,
S = sum_j |g_j xh_j|, c = sum_j g_j xh_j / H; dw within
sum_t |dy xh r| (dr + (T/64 + 24) 2^-24).  At least 99% of dx must equal the
exact value rounded to BF16.  The outputs are deterministic.
"""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
MID_BF16 = 1
U = 2.0 ** -24


def _f64(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp_bf16(v):
    return 2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126))) - 7)


def _inputs(oracle, T, H, bits, seed):
    rng = np.random.default_rng(seed)
    x = synthetic.bf16_bits_from_f32(rng.standard_t(4, T * H).astype(np.float32))
    codes, scales = oracle.quant_act(x, bits)
    dy = synthetic.bf16_bits_from_f32(rng.standard_normal(T * H).astype(np.float32))
    w = synthetic.bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    return codes, scales, dy, w


def _check(oracle, codes, scales, dy, w, T, H, bits, eps, got):
    gdx, grstd, gdw = got
    ex_dx, ex_r, ex_dw = oracle.rmsnorm_backward(codes, scales, dy, w, T, H, bits, eps)
    xh = _f64(oracle.dequant_act(codes, scales, T * H, bits)).reshape(T, H)
    g = _f64(dy).reshape(T, H) * _f64(w)[None, :]
    dr = (H / 2 + 8) * U
    r = ex_r[:, None]
    S = np.abs(g * xh).sum(axis=1, keepdims=True)
    c = (g * xh).sum(axis=1, keepdims=True) / H
    assert np.all(np.abs(grstd - ex_r) <= dr * 1.01 * ex_r)
    got_dx = _f64(gdx).reshape(T, H)
    slack = (np.abs(r * g) * (dr + 4 * U) + np.abs(xh) * r ** 3 * (np.abs(c) * (3 * dr + 8 * U)
             + (H + 1) * U * S / H) + 2 * U * np.abs(ex_dx))
    tol = 0.5 * _ulp_bf16(np.maximum(np.abs(ex_dx), np.abs(got_dx))) + slack + 1e-38
    bad = np.argwhere(np.abs(got_dx - ex_dx) > tol)
    assert bad.size == 0, "dx out of bound at %s" % bad[:3].tolist()
    assert np.mean(got_dx == oracle.round_format(ex_dx, MID_BF16).reshape(T, H)) >= 0.99
    if gdw is not None:
        terms = np.abs(_f64(dy).reshape(T, H) * xh * r).sum(axis=0)
        assert np.all(np.abs(gdw - ex_dw) <= terms * (dr + (T / 64 + 24) * U) + 1e-38)


def _run(codes, scales, dy, w, T, H, bits, eps, want_dw=True):
    dx, rstd, dw = agoq.agoq_rmsnorm_backward(G.dev(codes), G.dev(scales), G.dev_bf16(dy),
                                              G.dev_bf16(w), T, H, bits, eps, want_dw=want_dw)
    torch.cuda.synchronize()
    return (G.host_bits_bf16(dx), rstd.cpu().numpy().astype(np.float64),
            None if dw is None else dw.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("T,H", [(1, 256), (7, 512), (33, 4096), (5, 5120), (70, 8192),
                                 (32, 4096), (64, 512), (96, 5120), (320, 8192)])
def test_rmsnorm_backward_parity(oracle, bits, T, H):
    """T a multiple of 32 with H a multiple of 512 takes the TMA-staged dw
    kernel (32 and 64 rows: some CTAs of a cluster get no tile); the other
    shapes the register-buffered one."""
    eps = 1e-6
    codes, scales, dy, w = _inputs(oracle, T, H, bits, seed=T * 10 + bits)
    got = _run(codes, scales, dy, w, T, H, bits, eps)
    _check(oracle, codes, scales, dy, w, T, H, bits, eps, got)


def test_rmsnorm_backward_edge_rows(oracle):
    """An all-zero row (rstd = 1/sqrt(eps)), a constant row, a row with one
    outlier, a row of tiny values dominated by eps."""
    H, T, eps = 512, 4, 1e-5
    rng = np.random.default_rng(9)
    x = np.zeros((T, H), np.float32)
    x[1] = 3.0
    x[2] = rng.standard_normal(H) * 1e-2
    x[2, 17] = 500.0
    x[3] = rng.standard_normal(H) * 1e-4
    codes, scales = oracle.quant_act(synthetic.bf16_bits_from_f32(x.reshape(-1)), 4)
    dy = synthetic.bf16_bits_from_f32(rng.standard_normal(T * H).astype(np.float32))
    w = synthetic.bf16_bits_from_f32(np.ones(H, np.float32))
    got = _run(codes, scales, dy, w, T, H, 4, eps)
    _check(oracle, codes, scales, dy, w, T, H, 4, eps, got)


def test_rmsnorm_backward_deterministic_and_dw_optional(oracle):
    T, H = 300, 4096
    codes, scales, dy, w = _inputs(oracle, T, H, 4, seed=12)
    a = _run(codes, scales, dy, w, T, H, 4, 1e-6)
    b = _run(codes, scales, dy, w, T, H, 4, 1e-6)
    c = _run(codes, scales, dy, w, T, H, 4, 1e-6, want_dw=False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1]) and c[2] is None


def test_rmsnorm_backward_full_size(oracle):
    """The DBCA-PP RMSNorm input (8192 x 4096, Student-t) at 4 bits, in the
    bench's launch configuration; every output against the oracle."""
    T, H, bits, eps = 8192, 4096, 4, 1e-6
    x = synthetic.dbca_activations_torch(seed=1)[0]
    codes, scales = agoq.agoq_quant_act(x, bits)
    c_np, s_np = codes.cpu().numpy(), scales.cpu().numpy()
    rng = np.random.default_rng(21)
    dy = synthetic.bf16_bits_from_f32(rng.standard_normal(T * H).astype(np.float32))
    w = synthetic.bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    got = _run(c_np, s_np, dy, w, T, H, bits, eps)
    _check(oracle, c_np, s_np, dy, w, T, H, bits, eps, got)


def test_rmsnorm_dw_tma_and_register_paths(oracle):
    """The same rows through both dw kernels: rstd on a 16-byte boundary takes
    the TMA-staged kernel, rstd 4 bytes off it the register-buffered one.  dx
    and rstd come from the same row kernel (equal bits); both dw are within the
    bound."""
    T, H, bits, eps = 256, 1024, 5, 1e-6
    codes, scales, dy, w = _inputs(oracle, T, H, bits, seed=44)
    outs = []
    for off in (0, 1):
        room = torch.zeros(T + 4, dtype=torch.float32, device="cuda")
        rstd = room[off:off + T]
        assert (rstd.data_ptr() % 16 == 0) == (off == 0)
        dx = torch.empty(T * H, dtype=torch.bfloat16, device="cuda")
        dw = torch.empty(H, dtype=torch.float32, device="cuda")
        agoq.agoq_rmsnorm_backward(G.dev(codes), G.dev(scales), G.dev_bf16(dy), G.dev_bf16(w), T,
                                   H, bits, eps, dx, rstd, dw)
        torch.cuda.synchronize()
        got = (G.host_bits_bf16(dx), rstd.cpu().numpy().astype(np.float64),
               dw.cpu().numpy().astype(np.float64))
        _check(oracle, codes, scales, dy, w, T, H, bits, eps, got)
        outs.append(got)
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    agoq.agoq_device_status()   # raises if a pipeline wait timed out


def test_rmsnorm_backward_guard_bands(oracle):
    T, H = 9, 768
    codes, scales, dy, w = _inputs(oracle, T, H, 6, seed=31)
    dxg = G.Guarded(2 * T * H, torch.bfloat16)
    rg = G.Guarded(4 * 12, torch.float32)
    wg = G.Guarded(4 * H, torch.float32)
    agoq.agoq_rmsnorm_backward(G.dev(codes), G.dev(scales), G.dev_bf16(dy), G.dev_bf16(w), T, H,
                               6, 1e-6, dxg.view, rg.view[:T], wg.view)
    assert dxg.intact() and rg.intact() and wg.intact()
