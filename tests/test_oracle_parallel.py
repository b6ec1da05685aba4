"""The all-core (OpenMP) build of the oracle computes the same bits as the
single-threaded build, and the library-matmul form of the weight-gradient
product agrees with the plain k-ordered binary64 loop.

Both builds compile the same source; these checks guard the pragmas (a loop
variable or scratch array shared between threads would show up as a difference)
and the full-size product helper the GPU tests use."""
import numpy as np
import pytest

from gradient_quantization_gb300 import synthetic

pytestmark = pytest.mark.skipif(
    not __import__("oracle.oracle", fromlist=["x"]).parallel_available(),
    reason="no OpenMP toolchain for the all-core oracle build")


def test_threads_reported(oracle):
    assert oracle.threads(False) == 1
    assert oracle.threads(True) >= 1


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_quant_dequant_builds_agree(oracle, bits):
    x = synthetic.dbca_activations_np(seed=1, tokens=256, hidden=1024)[1].reshape(-1)
    c1, s1 = oracle.quant_act(x, bits)
    c2, s2 = oracle.quant_act(x, bits, parallel=True)
    assert np.array_equal(c1, c2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    y1 = oracle.dequant_act(c1, s1, x.size, bits)
    y2 = oracle.dequant_act(c1, s1, x.size, bits, parallel=True)
    assert np.array_equal(y1, y2)


def test_accum_builds_agree(oracle):
    n = 1 << 18
    m1, s1 = np.zeros(n, np.uint8), np.zeros(n // 128, np.float32)
    m2, s2 = m1.copy(), s1.copy()
    for g in synthetic.quangrad_grads_np(seed=2, n=n, steps=3):
        m1, s1 = oracle.grad_accum_fp8(m1, s1, g)
        oracle.grad_accum_fp8(m2, s2, g, parallel=True, in_place=True)
    assert np.array_equal(m1, m2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


@pytest.mark.parametrize("W", [2, 8, 13])
def test_reduce_builds_agree(oracle, W):
    n = 128 * 1000
    vals = synthetic.reduce_shard_values_np(seed=3, W=W, n=n)
    sh = np.empty((W, n), np.uint8)
    ss = np.empty((W, n // 128), np.float32)
    for r in range(W):
        sh[r], ss[r] = oracle.grad_accum_fp8(np.zeros(n, np.uint8), np.zeros(n // 128, np.float32),
                                             vals[r])
    a = oracle.reduce_fp8_shards(sh, ss, W, n)
    b = oracle.reduce_fp8_shards(sh, ss, W, n, parallel=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))
    assert a[2] == b[2] and a[2] > 0


def test_gemm_entries_builds_agree(oracle):
    M, N, K = 256, 512, 192
    dy, xg = synthetic.wgrad_inputs_np(seed=4, M=M, N=N, K=K)
    xc, xs = oracle.quant_act(xg.reshape(-1), 4)
    rng = np.random.default_rng(0)
    rows, cols = rng.integers(0, M, 500), rng.integers(0, N, 500)
    a = oracle.wgrad_gemm_int4_f64_entries(dy, xc, xs, M, N, K, rows, cols)
    b = oracle.wgrad_gemm_int4_f64_entries(dy, xc, xs, M, N, K, rows, cols, parallel=True)
    assert np.array_equal(a, b)


def test_matmul_product_matches_plain_loop(oracle):
    """Different summation orders in binary64: equal within a few binary64 ulps of
    the sum of |terms|; the absolute form is pinned by a numpy restatement."""
    M, N, K = 128, 256, 320
    dy, xg = synthetic.wgrad_inputs_np(seed=4, M=M, N=N, K=K)
    xc, xs = oracle.quant_act(xg.reshape(-1), 4)
    plain = oracle.wgrad_gemm_int4_f64(dy, xc, xs, M, N, K)
    fast = oracle.wgrad_gemm_int4_f64_matmul(dy, xc, xs, M, N, K)
    mag = oracle.wgrad_gemm_int4_f64_matmul(dy, xc, xs, M, N, K, absolute=True)
    assert np.all(np.abs(fast - plain) <= 4 * K * 2.0 ** -53 * mag)
    xh = oracle.bf16_to_f32(oracle.dequant_act(xc, xs, K * N, 4)).astype(np.float64).reshape(K, N)
    d = oracle.bf16_to_f32(dy).astype(np.float64).reshape(K, M)
    want = np.einsum("ki,kj->ij", np.abs(d), np.abs(xh))
    assert np.allclose(mag, want, rtol=1e-12, atol=0)
