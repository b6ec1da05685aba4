"""Pins of the oracle's fused weight-gradient product + QuanGrad accumulation.

The accumulation of a binary32 gradient is checked against the separately
pinned BF16-gradient accumulation (on gradients that are BF16 values), against
an exact-rational brute force and against numpy binary32 arithmetic.  The
fused form is checked against an exact-rational brute force on a tiny product,
against numpy's float64 matmul followed by the numpy restatement, against a
one-hot selector (the gradient is then a dequantized row, exactly), and its
sampled-block form against the full form.
"""
from fractions import Fraction

import numpy as np
import pytest

from gradient_quantization_gb300 import synthetic
from tests import exact
from tests.test_oracle_quangrad import e4m3_f32, f32_e4m3, requant_restated


def _bf16_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _random_master(rng, n):
    codes = f32_e4m3(rng.uniform(-448, 448, n).astype(np.float32))
    scales = rng.uniform(1e-5, 1e-2, n // 128).astype(np.float32)
    return codes, scales


def _accum_f32_restated(master, scales, g):
    m = (e4m3_f32(master).reshape(-1, 128) * scales[:, None]).astype(np.float32)
    t = (m + g.reshape(-1, 128).astype(np.float32)).astype(np.float32)
    return requant_restated(t)


def _inputs(oracle, M, N, K, seed=4):
    dy, x = synthetic.wgrad_inputs_np(seed=seed, M=M, N=N, K=K)
    xc, xs = oracle.quant_act(x.reshape(-1), 4)
    return dy, xc, xs


# ------------------------------------------------------------ binary32 gradient
def test_f32_accum_equals_bf16_accum_on_bf16_gradients(oracle):
    rng = np.random.default_rng(21)
    n = 1 << 14
    master, scales = _random_master(rng, n)
    g = synthetic.bf16_bits_from_f32((rng.standard_normal(n) * 1e-2).astype(np.float32))
    want = oracle.grad_accum_fp8(master, scales, g)
    got = oracle.grad_accum_fp8_f32(master, scales, _bf16_f32(g))
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32))


def test_f32_accum_matches_numpy_restatement_over_steps(oracle):
    rng = np.random.default_rng(22)
    n = 1 << 15
    master = np.zeros(n, np.uint8)
    scales = np.zeros(n // 128, np.float32)
    for step in range(4):
        g = (rng.standard_normal(n) * 10.0 ** -(step + 1)).astype(np.float32)
        g[rng.random(n) < 1e-3] *= 1000
        want = _accum_f32_restated(master, scales, g)
        master, scales = oracle.grad_accum_fp8_f32(master, scales, g)
        assert np.array_equal(master, want[0])
        assert np.array_equal(scales.view(np.uint32), want[1].view(np.uint32))


def test_f32_accum_exact_rational_brute_force(oracle):
    """Gradients with full 24-bit significands (not BF16 values)."""
    rng = np.random.default_rng(23)
    n = 256
    master, scales = _random_master(rng, n)
    g = (rng.standard_normal(n) * 3e-3).astype(np.float32)
    m, s = oracle.grad_accum_fp8_f32(master, scales, g)
    for b in range(n // 128):
        sb = exact.frac(scales[b])
        t = []
        for i in range(128):
            k = b * 128 + i
            mv = exact.to_f32(exact.e4m3_value(int(master[k])) * sb)
            t.append(exact.to_f32(exact.frac(mv) + exact.frac(g[k])))
        amax = max(abs(exact.frac(v)) for v in t)
        s2 = exact.to_f32(amax / 448)
        assert exact.f32_bits(float(s[b])) == exact.f32_bits(s2)
        for i, tv in enumerate(t):
            q = exact.to_f32(exact.frac(tv) / exact.frac(s2))
            want = exact.to_e4m3_code(exact.frac(q), negative_zero=np.signbit(q))
            assert int(m[b * 128 + i]) == want


# ------------------------------------------------------- product + accumulation
def test_fused_exact_rational_brute_force_tiny(oracle):
    M, N, K = 2, 128, 3
    dy, xc, xs = _inputs(oracle, M, N, K, seed=31)
    rng = np.random.default_rng(32)
    master, scales = _random_master(rng, M * N)
    got_m, got_s = oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, master, scales)
    xhat = _bf16_f32(oracle.dequant_act(xc, xs, K * N, 4)).reshape(K, N)
    dyv = _bf16_f32(dy).reshape(K, M)
    for i in range(M):
        sb = exact.frac(scales[i])
        t = []
        for j in range(N):
            prod = sum((exact.frac(dyv[k, i]) * exact.frac(xhat[k, j]) for k in range(K)),
                       Fraction(0))
            g = exact.to_f32(prod)
            mv = exact.to_f32(exact.e4m3_value(int(master[i * N + j])) * sb)
            t.append(exact.to_f32(exact.frac(mv) + exact.frac(g)))
        amax = max(abs(exact.frac(v)) for v in t)
        s2 = exact.to_f32(amax / 448)
        assert exact.f32_bits(float(got_s[i])) == exact.f32_bits(s2)
        for j, tv in enumerate(t):
            q = exact.to_f32(exact.frac(tv) / exact.frac(s2))
            want = exact.to_e4m3_code(exact.frac(q), negative_zero=np.signbit(q))
            assert int(got_m[i * N + j]) == want


@pytest.mark.parametrize("M,N,K", [(64, 256, 96), (32, 512, 300)])
def test_fused_matches_numpy_matmul_then_restatement(oracle, M, N, K):
    dy, xc, xs = _inputs(oracle, M, N, K, seed=33)
    rng = np.random.default_rng(34)
    master, scales = _random_master(rng, M * N)
    got = oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, master, scales)
    xhat = _bf16_f32(oracle.dequant_act(xc, xs, K * N, 4)).astype(np.float64).reshape(K, N)
    g = (_bf16_f32(dy).astype(np.float64).reshape(K, M).T @ xhat).astype(np.float32)
    want = _accum_f32_restated(master, scales, g.reshape(-1))
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32))


def test_fused_one_hot_is_bf16_accumulation_of_dequantized_rows(oracle):
    M, N, K = 48, 384, 80
    _, xc, xs = _inputs(oracle, M, N, K, seed=35)
    rng = np.random.default_rng(36)
    pick = rng.integers(0, K, M)
    dy = np.zeros((K, M), np.uint16)
    dy[pick, np.arange(M)] = 0x3F80                     # BF16 1.0
    master, scales = _random_master(rng, M * N)
    got = oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, master, scales)
    rows = oracle.dequant_act(xc, xs, K * N, 4).reshape(K, N)[pick].reshape(-1)
    want = oracle.grad_accum_fp8(master, scales, rows)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32))


def test_fused_zero_master_is_requant_of_rounded_product(oracle):
    """From a zeroed master the result is the FP8 block quantization of the
    binary32-rounded product."""
    M, N, K = 16, 256, 64
    dy, xc, xs = _inputs(oracle, M, N, K, seed=37)
    got = oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, np.zeros(M * N, np.uint8),
                                 np.zeros(M * N // 128, np.float32))
    g = oracle.wgrad_gemm_int4_f64(dy, xc, xs, M, N, K).astype(np.float32)
    want = requant_restated(g.reshape(-1))
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32))


def test_fused_blocks_form_matches_full(oracle):
    M, N, K = 24, 512, 40
    dy, xc, xs = _inputs(oracle, M, N, K, seed=38)
    rng = np.random.default_rng(39)
    master, scales = _random_master(rng, M * N)
    full_m, full_s = oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, master, scales)
    blocks = np.array([0, 5, 17, M * N // 128 - 1], np.int64)
    sub_m, sub_s = oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K,
                                          master.reshape(-1, 128)[blocks], scales[blocks],
                                          blocks=blocks)
    assert np.array_equal(sub_m.reshape(-1, 128), full_m.reshape(-1, 128)[blocks])
    assert np.array_equal(sub_s, full_s[blocks])


def test_fused_rejects_bad_arguments(oracle):
    dy, xc, xs = _inputs(oracle, 2, 128, 4, seed=40)
    with pytest.raises(ValueError):
        oracle.wgrad_accum_fp8(dy, xc, xs, 2, 128, 4, np.zeros(10, np.uint8),
                               np.zeros(2, np.float32))
    with pytest.raises(ValueError, match="rejected"):         # block index out of range
        oracle.wgrad_accum_fp8(dy, xc, xs, 2, 128, 4, np.zeros(128, np.uint8),
                               np.zeros(1, np.float32), blocks=[2])
