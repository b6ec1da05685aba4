"""Pins of the oracle's SiLU backward recomputed from LAAQ codes.

The derivative is checked against sympy's symbolic derivative of x * sigma(x)
evaluated at the dequantized inputs, the recomputed forward value against
scipy's logistic function, and both against closed forms (x = 0 and the
saturated tails); the dequantization step is the separately pinned one.
"""
import numpy as np
import pytest

from gradient_quantization_gb300 import synthetic


def _bf16_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(oracle, n, bits, seed):
    x = synthetic.dbca_activations_np(seed=seed, tokens=1, hidden=n, ffn=128)[0].reshape(-1)
    codes, scales = oracle.quant_act(x, bits)
    rng = np.random.default_rng(seed)
    dy = synthetic.bf16_bits_from_f32(rng.standard_normal(n).astype(np.float32))
    return codes, scales, dy


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_silu_backward_matches_symbolic_derivative(oracle, bits):
    sympy = pytest.importorskip("sympy")
    n = 512
    codes, scales, dy = _case(oracle, n, bits, seed=70 + bits)
    dx, y = oracle.silu_backward(codes, scales, dy, n, bits)
    xh = _bf16_f64(oracle.dequant_act(codes, scales, n, bits))
    t = sympy.Symbol("t")
    dsilu = sympy.lambdify(t, sympy.diff(t / (1 + sympy.exp(-t)), t), "mpmath")
    want = np.array([float(dsilu(sympy.Float(v, 40))) for v in xh]) * _bf16_f64(dy)
    assert np.allclose(dx, want, rtol=1e-13, atol=1e-300)


@pytest.mark.parametrize("bits", [4, 8])
def test_silu_forward_recompute_matches_scipy_logistic(oracle, bits):
    special = pytest.importorskip("scipy.special")
    n = 1024
    codes, scales, dy = _case(oracle, n, bits, seed=80 + bits)
    _, y = oracle.silu_backward(codes, scales, dy, n, bits)
    xh = _bf16_f64(oracle.dequant_act(codes, scales, n, bits))
    assert np.allclose(y, xh * special.expit(xh), rtol=1e-14, atol=0)


def test_silu_backward_closed_forms(oracle):
    # one 4-bit block: codes 0, +-7 at scale 1 and at scale 40/7 (x = +-40)
    n = 128
    x = np.zeros(n, np.float32)
    x[0], x[1], x[2] = 40.0, -40.0, 0.0
    codes, scales = oracle.quant_act(synthetic.bf16_bits_from_f32(x), 4)
    dy = synthetic.bf16_bits_from_f32(np.full(n, 3.0, np.float32))
    dx, y = oracle.silu_backward(codes, scales, dy, n, 4)
    assert dx[2] == 1.5 and y[2] == 0.0                  # sigma(0) = 1/2: silu'(0) = 1/2
    assert abs(dx[0] - 3.0) < 3.0 * 41 * np.exp(-40)     # silu'(x) -> 1 for x >> 0
    assert abs(dx[1]) < 3.0 * 41 * np.exp(-40)           # silu'(x) -> 0 for x << 0
    assert abs(y[0] - 40.0) < 1e-15 and abs(y[1]) < 40 * np.exp(-39)


def test_silu_backward_without_forward_output(oracle):
    n = 256
    codes, scales, dy = _case(oracle, n, 5, seed=90)
    dx1, _ = oracle.silu_backward(codes, scales, dy, n, 5, want_y=False)
    dx2, _ = oracle.silu_backward(codes, scales, dy, n, 5)
    assert np.array_equal(dx1, dx2)
