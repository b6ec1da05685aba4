"""Pins of the oracle's forward product with the fused LAAQ quantization of its
output: the product against numpy's float64 matmul of the BF16 operands
(rounded to binary32 then BF16 by torch's casts), exact-rational brute force on
a tiny case, and the quantization against the separately pinned quant_act."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import synthetic
from tests import exact


def _f64(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _operands(T, N, K, seed):
    rng = np.random.default_rng(seed)
    x = synthetic.bf16_bits_from_f32(rng.standard_normal(T * K).astype(np.float32))
    w = synthetic.bf16_bits_from_f32((rng.standard_normal(N * K) * 0.02).astype(np.float32))
    return x, w


@pytest.mark.parametrize("T,N,K,bits", [(8, 128, 64, 4), (5, 256, 96, 5), (3, 384, 40, 8)])
def test_product_and_quantization(oracle, T, N, K, bits):
    x, w = _operands(T, N, K, seed=T + N + K)
    y, codes, scales = oracle.fwd_gemm_quant(x, w, T, N, K, bits)
    prod = _f64(x).reshape(T, K) @ _f64(w).reshape(N, K).T
    want_y = torch.from_numpy(prod.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(y.reshape(-1), want_y.view(torch.int16).numpy().view(np.uint16).reshape(-1))
    wc, ws = oracle.quant_act(y.reshape(-1), bits)
    assert np.array_equal(codes, wc) and np.array_equal(scales.view(np.uint32), ws.view(np.uint32))


def test_product_exact_rational_tiny(oracle):
    T, N, K = 2, 128, 3
    x, w = _operands(T, N, K, seed=9)
    y, _, _ = oracle.fwd_gemm_quant(x, w, T, N, K, 4)
    xv, wv = _f64(x).reshape(T, K), _f64(w).reshape(N, K)
    for t in range(T):
        for n in range(N):
            acc = sum((Fraction(xv[t, k]) * Fraction(wv[n, k]) for k in range(K)), Fraction(0))
            f32 = exact.to_f32(acc)
            want = torch.tensor([f32], dtype=torch.float32).to(torch.bfloat16)
            assert int(y[t, n]) == int(want.view(torch.int16).numpy().view(np.uint16)[0])


def test_rejects_bad_shapes(oracle):
    x, w = _operands(2, 128, 4, seed=1)
    with pytest.raises(ValueError):
        oracle.fwd_gemm_quant(x, w, 2, 100, 4, 4)
