"""Pins of the oracle's RMSNorm backward recomputed from LAAQ codes.

The gradients are checked against torch autograd of the plain RMSNorm forward
in float64 (a library routine evaluating the same definition independently),
against central finite differences of the forward, and against closed forms;
the dequantization step is the separately pinned one.
"""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import synthetic


def _f64(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(oracle, T, H, bits, seed):
    rng = np.random.default_rng(seed)
    x = synthetic.bf16_bits_from_f32(rng.standard_t(4, T * H).astype(np.float32))
    codes, scales = oracle.quant_act(x, bits)
    dy = synthetic.bf16_bits_from_f32(rng.standard_normal(T * H).astype(np.float32))
    w = synthetic.bf16_bits_from_f32((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    return codes, scales, dy, w


def _forward(x, w, eps):
    return x * torch.rsqrt((x * x).mean(dim=1, keepdim=True) + eps) * w


@pytest.mark.parametrize("bits,T,H", [(4, 3, 256), (5, 5, 384), (8, 2, 1024)])
def test_rmsnorm_backward_matches_autograd(oracle, bits, T, H):
    eps = 1e-6
    codes, scales, dy, w = _case(oracle, T, H, bits, seed=bits * 10 + T)
    dx, rstd, dw = oracle.rmsnorm_backward(codes, scales, dy, w, T, H, bits, eps)
    xh = torch.from_numpy(_f64(oracle.dequant_act(codes, scales, T * H, bits)).reshape(T, H))
    xh.requires_grad_(True)
    wt = torch.from_numpy(_f64(w)).requires_grad_(True)
    y = _forward(xh, wt, eps)
    y.backward(torch.from_numpy(_f64(dy).reshape(T, H)))
    assert np.allclose(dx, xh.grad.numpy(), rtol=1e-12, atol=1e-12 * np.abs(dx).max())
    assert np.allclose(dw, wt.grad.numpy(), rtol=1e-12, atol=1e-12 * np.abs(dw).max())
    want_r = 1 / np.sqrt((xh.detach().numpy() ** 2).mean(axis=1) + eps)
    assert np.allclose(rstd, want_r, rtol=1e-14)


def test_rmsnorm_backward_matches_finite_differences(oracle):
    T, H, bits, eps = 2, 128, 6, 1e-5
    codes, scales, dy, w = _case(oracle, T, H, bits, seed=5)
    dx, _, dw = oracle.rmsnorm_backward(codes, scales, dy, w, T, H, bits, eps)
    x = _f64(oracle.dequant_act(codes, scales, T * H, bits)).reshape(T, H)
    wv, g = _f64(w), _f64(dy).reshape(T, H)
    def loss(xx, ww):
        r = 1 / np.sqrt((xx * xx).mean(axis=1, keepdims=True) + eps)
        return float((xx * r * ww * g).sum())
    h = 1e-6
    for (t, i) in [(0, 0), (1, 77), (0, 127)]:
        xp, xm = x.copy(), x.copy()
        xp[t, i] += h
        xm[t, i] -= h
        assert abs((loss(xp, wv) - loss(xm, wv)) / (2 * h) - dx[t, i]) < 1e-6 * (1 + abs(dx[t, i]))
    for i in (3, 100):
        wp, wm = wv.copy(), wv.copy()
        wp[i] += h
        wm[i] -= h
        assert abs((loss(x, wp) - loss(x, wm)) / (2 * h) - dw[i]) < 1e-6 * (1 + abs(dw[i]))


def test_rmsnorm_backward_closed_forms(oracle):
    """A constant row x = c (all codes +7 at scale c/7): r = 1/sqrt(c^2 + eps);
    with dy = 1 and w = 1 the input gradient is r - c^2 r^3 = eps * r^3."""
    H, eps = 256, 1e-3
    x = synthetic.bf16_bits_from_f32(np.full(H, 2.0, np.float32))
    codes, scales = oracle.quant_act(x, 4)
    one = synthetic.bf16_bits_from_f32(np.ones(H, np.float32))
    dx, rstd, dw = oracle.rmsnorm_backward(codes, scales, one, one, 1, H, 4, eps)
    r = 1 / np.sqrt(4.0 + eps)
    assert abs(rstd[0] - r) < 1e-15
    assert np.allclose(dx, eps * r ** 3, rtol=1e-9, atol=0)
    assert np.allclose(dw, 2.0 * r, rtol=1e-15)


def test_rmsnorm_backward_rejects_bad_shapes(oracle):
    with pytest.raises(ValueError):
        oracle.rmsnorm_backward(np.zeros(64, np.uint8), np.zeros(1, np.float32),
                                np.zeros(100, np.uint16), np.zeros(100, np.uint16), 1, 100, 4, 1e-6)
