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


def _check(oracle, codes, scales, dy, w, T, H, bits, eps, got, dw_chain=None):
    """dw_chain: the longest chain of binary32 additions in a dw sum (default:
    the two-pass kernels' T/64 + 24)."""
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
        chain = T / 64 + 24 if dw_chain is None else dw_chain
        assert np.all(np.abs(gdw - ex_dw) <= terms * (dr + chain * U) + 1e-38)


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


# ---------------------------------------------------------------- single read
def _ws_chain(T):
    """Longest dw addition chain of the single-read path: ceil(T / 2G) rows per
    thread, the two row groups, ceil(G / 8) partial rows per range, the eight
    range sums; G <= min(304, ceil(T / 2)) partial rows (as many CTAs as fit at
    once), and the chain is longest for the largest G when T >= 2G."""
    worst = 0
    for G_ in range(1, min(304, (T + 1) // 2) + 1):
        worst = max(worst, -(-T // (2 * G_)) + 1 + -(-G_ // 8) + 8)
    return worst


def _run_ws(codes, scales, dy, w, T, H, bits, eps, ws=None):
    if ws is None:
        ws = torch.empty(max(agoq.agoq_rmsnorm_backward_workspace_bytes(H), 16), dtype=torch.uint8,
                         device="cuda")
    dx, rstd, dw = agoq.agoq_rmsnorm_backward_ws(G.dev(codes), G.dev(scales), G.dev_bf16(dy),
                                                 G.dev_bf16(w), T, H, bits, eps, ws)
    torch.cuda.synchronize()
    return (G.host_bits_bf16(dx), rstd.cpu().numpy().astype(np.float64),
            dw.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("T,H", [(1, 256), (7, 512), (33, 4096), (2, 1280), (64, 3072),
                                 (609, 1024), (1000, 4096), (5, 8192)])
def test_rmsnorm_backward_ws_parity(oracle, bits, T, H):
    """One read of the input: 1 to 4 chunks of 8 columns per thread (H up to
    4096), more rows than 2 x 304 (several rows per thread), odd T (a row group
    with no last row); H = 8192 takes the two-pass kernels."""
    eps = 1e-6
    codes, scales, dy, w = _inputs(oracle, T, H, bits, seed=T * 7 + bits + H)
    got = _run_ws(codes, scales, dy, w, T, H, bits, eps)
    chain = _ws_chain(T) if H <= 4096 else None
    _check(oracle, codes, scales, dy, w, T, H, bits, eps, got, dw_chain=chain)


def test_rmsnorm_backward_ws_deterministic_and_close_to_two_pass(oracle):
    """Repeatable bits; the row sums are added in another order than in the
    two-pass kernels, so rstd agrees to a few ulps and dx nearly everywhere; dw
    within the bound of its chain."""
    T, H = 1500, 4096
    codes, scales, dy, w = _inputs(oracle, T, H, 4, seed=77)
    a = _run_ws(codes, scales, dy, w, T, H, 4, 1e-6)
    b = _run_ws(codes, scales, dy, w, T, H, 4, 1e-6)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    c = _run(codes, scales, dy, w, T, H, 4, 1e-6)
    assert np.all(np.abs(a[1] - c[1]) <= 2 * (H / 2 + 8) * U * c[1])
    assert np.mean(a[0] == c[0]) >= 0.99
    _check(oracle, codes, scales, dy, w, T, H, 4, 1e-6, a, dw_chain=_ws_chain(T))


def test_rmsnorm_backward_ws_full_size(oracle):
    """The DBCA-PP RMSNorm input (8192 x 4096) at 4 bits, single read; every
    output against the oracle."""
    T, H, bits, eps = 8192, 4096, 4, 1e-6
    x = synthetic.dbca_activations_np(seed=1)[0].reshape(-1)
    codes, scales = oracle.quant_act(x, bits, parallel=oracle.parallel_available())
    rng = np.random.default_rng(21)
    dy = synthetic.bf16_bits_from_f32(rng.standard_normal(T * H).astype(np.float32))
    w = synthetic.bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    got = _run_ws(codes, scales, dy, w, T, H, bits, eps)
    _check(oracle, codes, scales, dy, w, T, H, bits, eps, got, dw_chain=_ws_chain(T))


def test_rmsnorm_backward_ws_guard_bands_and_arguments(oracle):
    T, H = 37, 1024
    codes, scales, dy, w = _inputs(oracle, T, H, 5, seed=38)
    need = agoq.agoq_rmsnorm_backward_workspace_bytes(H)
    assert need == 304 * H * 4
    dxg = G.Guarded(2 * T * H, torch.bfloat16)
    rg = G.Guarded(4 * 40, torch.float32)
    wg = G.Guarded(4 * H, torch.float32)
    ws = G.Guarded(need, torch.uint8)
    agoq.agoq_rmsnorm_backward_ws(G.dev(codes), G.dev(scales), G.dev_bf16(dy), G.dev_bf16(w), T, H,
                                  5, 1e-6, ws.view, dxg.view, rg.view[:T], wg.view)
    assert dxg.intact() and rg.intact() and wg.intact() and ws.intact()
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(agoq.AgoqError):
        agoq.agoq_rmsnorm_backward_ws(G.dev(codes), G.dev(scales), G.dev_bf16(dy), G.dev_bf16(w),
                                      T, H, 5, 1e-6, small)
