"""Pins of the oracle's INT4-operand weight-gradient product dW = dY^T Xhat.

The contraction is checked against numpy's float64 matmul on the oracle's own
(separately pinned) 4-bit dequantization, against a one-hot selector that must
return dequantized rows exactly, and the sampled-entry form against the full form.
"""
import numpy as np
import pytest

from gradient_quantization_gb300 import synthetic


def _inputs(oracle, M, N, K, seed=4):
    dy, x = synthetic.wgrad_inputs_np(seed=seed, M=M, N=N, K=K)
    xc, xs = oracle.quant_act(x.reshape(-1), 4)
    return dy, xc, xs


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (96, 384, 200), (256, 128, 1)])
def test_product_matches_numpy_matmul_of_dequantized_operand(oracle, M, N, K):
    dy, xc, xs = _inputs(oracle, M, N, K)
    got = oracle.wgrad_gemm_int4_f64(dy, xc, xs, M, N, K)
    xhat = _f64(oracle.dequant_act(xc, xs, K * N, 4)).reshape(K, N)
    want = _f64(dy).reshape(K, M).T @ xhat
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_one_hot_selector_returns_dequantized_rows(oracle):
    M, N, K = 64, 256, 96
    _, xc, xs = _inputs(oracle, M, N, K)
    rng = np.random.default_rng(9)
    pick = rng.integers(0, K, M)
    dy = np.zeros((K, M), np.uint16)
    dy[pick, np.arange(M)] = 0x3F80            # BF16 1.0
    got = oracle.wgrad_gemm_int4_f64(dy, xc, xs, M, N, K)
    xhat = _f64(oracle.dequant_act(xc, xs, K * N, 4)).reshape(K, N)
    assert np.array_equal(got, xhat[pick])


def test_entries_match_full_product(oracle):
    M, N, K = 96, 256, 160
    dy, xc, xs = _inputs(oracle, M, N, K)
    full = oracle.wgrad_gemm_int4_f64(dy, xc, xs, M, N, K)
    rng = np.random.default_rng(3)
    rows = rng.integers(0, M, 300)
    cols = rng.integers(0, N, 300)
    got = oracle.wgrad_gemm_int4_f64_entries(dy, xc, xs, M, N, K, rows, cols)
    assert np.array_equal(got, full[rows, cols])


def test_rejects_bad_shapes(oracle):
    with pytest.raises(ValueError):
        oracle.wgrad_gemm_int4_f64(np.zeros(8, np.uint16), np.zeros(8, np.uint8),
                                   np.zeros(1, np.float32), 2, 100, 4)
