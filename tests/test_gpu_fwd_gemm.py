"""GPU parity of the forward GEMM with the fused LAAQ quantization of its output
(agoq_fwd_gemm_quant) against the CPU oracle.

Operands on a power-of-two grid make the FP32 accumulation exact in any order:
Y, codes and scales are then compared bit for bit.  Gaussian operands: Y within
the binary32 summation bound of the binary64 product (and <= 1e-3 relative
Frobenius against its BF16 rounding), and codes/scales equal to the LAAQ
quantization of the returned Y restated with numpy binary32 arithmetic.
"""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _f64(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _exact_operands(T, N, K, seed):
    """X [T][K] = i * 2^-6 (i in -3..3), W [N][K] = c * 2^e blocks (c in -7..7)."""
    dy, x = synthetic.wgrad_exact_sum_inputs_np(seed=seed, M=T, N=N, K=K)
    return np.ascontiguousarray(dy.T), np.ascontiguousarray(x.T)


def _gauss_operands(T, N, K, seed):
    rng = np.random.default_rng(seed)
    x = synthetic.bf16_bits_from_f32(rng.standard_normal(T * K).astype(np.float32)).reshape(T, K)
    w = synthetic.bf16_bits_from_f32((rng.standard_normal(N * K) * 0.02).astype(np.float32))
    return x, w.reshape(N, K)


def _run(x, w, T, N, K, bits):
    y, c, s = agoq.agoq_fwd_gemm_quant(G.dev_bf16(x).view(T, K), G.dev_bf16(w).view(N, K), T, N,
                                       K, bits)
    agoq.agoq_device_status()
    return G.host_bits_bf16(y).reshape(T, N), c.cpu().numpy(), s.cpu().numpy()


def _unpack(codes, nblocks, bits):
    rec = codes.reshape(nblocks, 16 * bits)
    stream = np.unpackbits(rec, axis=1, bitorder="little").reshape(nblocks, 128, bits)
    v = (stream.astype(np.int64) << np.arange(bits)).sum(axis=2)
    return np.where(v >= 1 << (bits - 1), v - (1 << bits), v)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
# K a multiple of 128 runs the 128-deep instance, the other multiples of 64 the
# 64-deep one; T = 128 and 384 leave half of a 256-row pair tile empty.
@pytest.mark.parametrize("T,N,K", [(128, 256, 64), (256, 512, 192), (384, 768, 320),
                                   (128, 256, 128), (384, 768, 384), (512, 1024, 256)])
def test_exact_sums_bitwise(oracle, bits, T, N, K):
    x, w = _exact_operands(T, N, K, seed=T + N + K + bits)
    y, c, s = _run(x, w, T, N, K, bits)
    wy, wc, ws = oracle.fwd_gemm_quant(x, w, T, N, K, bits)
    assert np.array_equal(y, wy)
    assert np.array_equal(c, wc)
    assert np.array_equal(s.view(np.uint32), ws.view(np.uint32))


@pytest.mark.parametrize("K", [64, 128])
def test_exact_sums_many_tiles(oracle, K):
    """80 tiles of 256 x 256 on 76 CTA pairs (a second persistent round, both
    TMEM buffers), for both k-block depths."""
    T, N, bits = 1280, 4096, 4
    x, w = _exact_operands(T, N, K, seed=77)
    y, c, s = _run(x, w, T, N, K, bits)
    wy, wc, ws = oracle.fwd_gemm_quant(x, w, T, N, K, bits)
    assert np.array_equal(y, wy)
    assert np.array_equal(c, wc) and np.array_equal(s.view(np.uint32), ws.view(np.uint32))


def _check_codes_of_y(y, c, s, T, N, bits):
    """codes/scales are the LAAQ quantization of the returned Y (numpy binary32)."""
    qmax = np.float32((1 << (bits - 1)) - 1)
    yb = _f64(y).astype(np.float32).reshape(-1, 128)
    am = np.abs(yb).max(axis=1)
    want_s = (am / qmax).astype(np.float32)
    assert np.array_equal(s.view(np.uint32), want_s.view(np.uint32))
    safe = np.where(want_s > 0, want_s, np.float32(1))
    q = np.rint((yb / safe[:, None]).astype(np.float32)).astype(np.int64)
    q = np.where(want_s[:, None] > 0, np.clip(q, -qmax, qmax), 0)
    assert np.array_equal(_unpack(c, T * N // 128, bits), q)


@pytest.mark.parametrize("bits", [4, 6])
def test_gaussian_within_bounds(oracle, bits):
    T, N, K = 256, 512, 1024
    x, w = _gauss_operands(T, N, K, seed=5)
    y, c, s = _run(x, w, T, N, K, bits)
    prod = _f64(x).reshape(T, K) @ _f64(w).reshape(N, K).T
    bound = K * 2.0 ** -23 * (np.abs(_f64(x)).reshape(T, K) @ np.abs(_f64(w)).reshape(N, K).T)
    got = _f64(y)
    half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(prod), 2.0 ** -126))) - 8)
    assert np.all(np.abs(got - prod) <= bound + 2 * half_ulp)
    wy, _, _ = oracle.fwd_gemm_quant(x, w, T, N, K, bits)
    assert np.linalg.norm(got - _f64(wy)) / np.linalg.norm(_f64(wy)) <= 1e-3
    _check_codes_of_y(y, c, s, T, N, bits)


def test_full_size_sampled_rows(oracle):
    """The LLaMA-7B gate projection (8192 tokens x 4096 -> 11008) in the bench's
    launch configuration on exact-sum operands; 6 rows against the oracle bit
    for bit, every row's codes consistent with its Y."""
    T, N, K, bits = 8192, 11008, 4096, 4
    x, w = _exact_operands(T, N, K, seed=91)
    y, c, s = _run(x, w, T, N, K, bits)
    rows = np.array([0, 1, 4095, 5000, 8190, 8191])
    wy, wc, ws = oracle.fwd_gemm_quant(x[rows], w, rows.size, N, K, bits)
    assert np.array_equal(y[rows], wy)
    per_row = N // 128
    crow = c.reshape(T, per_row * 16 * bits)[rows].reshape(-1)
    assert np.array_equal(crow, wc)
    assert np.array_equal(s.reshape(T, per_row)[rows].reshape(-1).view(np.uint32), ws.view(np.uint32))
    _check_codes_of_y(y[:64], c[:64 * per_row * 16 * bits], s[:64 * per_row], 64, N, bits)


def test_guard_bands(oracle):
    T, N, K, bits = 128, 512, 128, 5
    x, w = _gauss_operands(T, N, K, seed=8)
    yg = G.Guarded(2 * T * N, torch.bfloat16)
    cg = G.Guarded(T * N // 128 * 16 * bits, torch.uint8)
    sg = G.Guarded(T * N // 128 * 4, torch.float32)
    agoq.agoq_fwd_gemm_quant(G.dev_bf16(x).view(T, K), G.dev_bf16(w).view(N, K), T, N, K, bits,
                             yg.view, cg.view, sg.view)
    agoq.agoq_device_status()
    assert yg.intact() and cg.intact() and sg.intact()
