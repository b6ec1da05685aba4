"""GPU checks of the weight-gradient GEMM with the QuanGrad FP8 accumulation as
its epilogue (agoq_wgrad_gemm_int4_accum_fp8) against the CPU oracle.

The tensor cores' FP32 summation order is not specified, so bit-exact parity
is asserted where that summation is exact in any order: operands on a
power-of-two grid (every partial sum a small multiple of 2^-10) and one-hot
selectors.  Seeded Gaussian operands are checked against the oracle within the
summation bound K * 2^-23 * sum|terms| carried through one E4M3 requantization.
"""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _bf16_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _exact_inputs(oracle, M, N, K, seed):
    dy, x = synthetic.wgrad_exact_sum_inputs_np(seed=seed, M=M, N=N, K=K)
    xc, xs = oracle.quant_act(x.reshape(-1), 4)
    return dy, xc, xs


def _gauss_inputs(oracle, M, N, K, seed):
    dy, x = synthetic.wgrad_inputs_np(seed=seed, M=M, N=N, K=K)
    xc, xs = oracle.quant_act(x.reshape(-1), 4)
    return dy, xc, xs


def _master(oracle, n, seed, sd):
    """An FP8 master made by the oracle's accumulation from zero of one seeded
    N(0, sd) BF16 gradient."""
    rng = np.random.default_rng(seed)
    g = synthetic.bf16_bits_from_f32((rng.standard_normal(n) * sd).astype(np.float32))
    return oracle.grad_accum_fp8(np.zeros(n, np.uint8), np.zeros(n // 128, np.float32), g)


def _run(dy, xc, xs, M, N, K, master, scales):
    mg = G.Guarded(M * N, torch.uint8)
    sg = G.Guarded(M * N // 128 * 4, torch.float32)
    mg.view.copy_(torch.from_numpy(master))
    sg.view.copy_(torch.from_numpy(scales))
    agoq.agoq_wgrad_gemm_int4_accum_fp8(G.dev_bf16(dy), G.dev(xc), G.dev(xs), M, N, K,
                                        mg.view, sg.view)
    agoq.agoq_device_status()
    assert mg.intact() and sg.intact()
    return mg.view.cpu().numpy(), sg.view.cpu().numpy()


def _assert_same(got, want):
    assert np.array_equal(got[0], want[0]), "codes differ at %s" % (
        np.flatnonzero(got[0] != want[0])[:8].tolist(),)
    assert np.array_equal(got[1].view(np.uint32), want[1].view(np.uint32)), "scales differ"


@pytest.mark.parametrize("M,N,K", [(256, 512, 64), (256, 512, 320), (512, 1024, 128),
                                   (768, 1536, 192), (768, 1536, 384),
                                   (128, 128, 64), (384, 640, 192), (640, 384, 128)])
def test_exact_sums_match_oracle_bitwise(oracle, M, N, K):
    dy, xc, xs = _exact_inputs(oracle, M, N, K, seed=50 + K)
    master, scales = _master(oracle, M * N, seed=60 + M, sd=2.0)
    got = _run(dy, xc, xs, M, N, K, master, scales)
    _assert_same(got, oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, master, scales))


@pytest.mark.parametrize("K", [64, 128])
def test_exact_sums_over_many_tiles_and_waves(oracle, K):
    """More tiles than SMs (several persistent waves); every block checked."""
    M, N = 2560, 4096
    dy, xc, xs = _exact_inputs(oracle, M, N, K, seed=70)
    master, scales = _master(oracle, M * N, seed=71, sd=0.5)
    got = _run(dy, xc, xs, M, N, K, master, scales)
    _assert_same(got, oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, master, scales))


def test_zeroed_master_and_chained_micro_batches(oracle):
    """A zeroed master (scales +0) takes three products in a row, as QuanGrad
    accumulates micro-batches; each step matches the oracle bit for bit."""
    M, N, K = 256, 1024, 192
    master = np.zeros(M * N, np.uint8)
    scales = np.zeros(M * N // 128, np.float32)
    mg = torch.from_numpy(master).cuda()
    sg = torch.from_numpy(scales).cuda()
    for step in range(3):
        dy, xc, xs = _exact_inputs(oracle, M, N, K, seed=80 + step)
        agoq.agoq_wgrad_gemm_int4_accum_fp8(G.dev_bf16(dy), G.dev(xc), G.dev(xs), M, N, K, mg, sg)
        agoq.agoq_device_status()
        master, scales = oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, master, scales)
        _assert_same((mg.cpu().numpy(), sg.cpu().numpy()), (master, scales))


def test_one_hot_selector_is_bf16_accumulation_of_rows(oracle):
    M, N, K = 512, 1024, 256
    _, xc, xs = _gauss_inputs(oracle, M, N, K, seed=90)
    rng = np.random.default_rng(91)
    pick = rng.integers(0, K, M)
    dy = np.zeros((K, M), np.uint16)
    dy[pick, np.arange(M)] = 0x3F80                     # 1.0
    master, scales = _master(oracle, M * N, seed=92, sd=1.0)
    got = _run(dy, xc, xs, M, N, K, master, scales)
    rows = oracle.dequant_act(xc, xs, K * N, 4).reshape(K, N)[pick].reshape(-1)
    _assert_same(got, oracle.grad_accum_fp8(master, scales, rows))


def _half_step(q):
    """Half the E4M3 spacing at |q| (code units)."""
    q = np.abs(q)
    e = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
    return np.where(q < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))


def _check_within_bound(oracle, dy, xc, xs, M, N, K, master, scales, got, blocks=None):
    """GPU result vs oracle: codes equal almost everywhere, and every dequantized
    value within the summation bound plus one requantization step of the oracle's."""
    want = oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, master, scales, blocks=blocks)
    gc, gs = got
    wc, ws = want
    ge = torch.from_numpy(gc).view(torch.float8_e4m3fn).double().numpy().reshape(-1, 128)
    we = torch.from_numpy(wc).view(torch.float8_e4m3fn).double().numpy().reshape(-1, 128)
    gd = ge * gs.astype(np.float64)[:, None]
    wd = we * ws.astype(np.float64)[:, None]
    # per-element summation bound sum_k |dY[k][m] Xhat[k][n]| for the checked blocks
    per_row = N // 128
    bidx = np.arange(M * per_row) if blocks is None else np.asarray(blocks)
    rows, cols0 = bidx // per_row, (bidx % per_row) * 128
    dyv = np.abs(_bf16_f64(dy)).reshape(K, M)
    xh = np.abs(_bf16_f64(oracle.dequant_act(xc, xs, K * N, 4))).reshape(K, N)
    terms = np.stack([dyv[:, r] @ xh[:, c0:c0 + 128] for r, c0 in zip(rows, cols0)])
    bound = K * 2.0 ** -23 * terms
    slack = (bound + 2.0 ** -22 * np.abs(wd)
             + _half_step(ge) * gs.astype(np.float64)[:, None]
             + _half_step(we) * ws.astype(np.float64)[:, None] + 1e-30)
    assert (np.abs(gd - wd) <= slack).all()
    assert np.mean(gc == wc) >= 0.99


@pytest.mark.parametrize("M,N,K", [(256, 512, 192), (512, 1024, 448)])
def test_gaussian_within_summation_and_requant_bound(oracle, M, N, K):
    dy, xc, xs = _gauss_inputs(oracle, M, N, K, seed=100 + K)
    master, scales = _master(oracle, M * N, seed=101, sd=0.2)
    got = _run(dy, xc, xs, M, N, K, master, scales)
    _check_within_bound(oracle, dy, xc, xs, M, N, K, master, scales, got)


def test_repeatable_across_calls(oracle):
    M, N, K = 512, 1024, 128
    dy, xc, xs = _gauss_inputs(oracle, M, N, K, seed=110)
    master, scales = _master(oracle, M * N, seed=111, sd=0.2)
    a = _run(dy, xc, xs, M, N, K, master, scales)
    b = _run(dy, xc, xs, M, N, K, master, scales)
    _assert_same(a, b)


def test_full_size_exact_sums_sampled_blocks(oracle):
    """11008 x 4096 x 8192 on the power-of-two grid, in the bench's launch
    configuration; 96 sampled blocks (first, last, random) bit for bit."""
    M, N, K = synthetic.WGRAD_M, synthetic.WGRAD_N, synthetic.WGRAD_K
    dy, xc, xs = _exact_inputs(oracle, M, N, K, seed=120)
    master, scales = _master(oracle, M * N, seed=121, sd=8.0)
    m, s = G.dev(master), G.dev(scales)
    blocks = G.sample_blocks(M * N // 128, 96, seed=122)
    m0, s0 = master.reshape(-1, 128)[blocks].reshape(-1), scales[blocks]
    agoq.agoq_wgrad_gemm_int4_accum_fp8(G.dev_bf16(dy), G.dev(xc), G.dev(xs), M, N, K, m, s)
    agoq.agoq_device_status()
    got = (G.gather_blocks(m, blocks, 128).numpy().reshape(-1),
           G.gather_blocks(s, blocks, 1).numpy().reshape(-1))
    _assert_same(got, oracle.wgrad_accum_fp8(dy, xc, xs, M, N, K, m0, s0, blocks=blocks))


def test_full_size_gaussian_sampled_blocks(oracle):
    """The bench's operands (dY ~ N(0, 1e-2), X Gaussian with outliers, 4-bit)
    at full size; 24 sampled blocks within the bound."""
    M, N, K = synthetic.WGRAD_M, synthetic.WGRAD_N, synthetic.WGRAD_K
    dy_t, x_t = synthetic.wgrad_inputs_torch(seed=4)
    x_np = G.host_bits_bf16(x_t)
    xc, xs = oracle.quant_act(x_np, 4)
    dy = G.host_bits_bf16(dy_t).reshape(K, M)
    master, scales = _master(oracle, M * N, seed=131, sd=0.05)
    m, s = G.dev(master), G.dev(scales)
    blocks = G.sample_blocks(M * N // 128, 24, seed=132)
    m0, s0 = master.reshape(-1, 128)[blocks].reshape(-1), scales[blocks]
    agoq.agoq_wgrad_gemm_int4_accum_fp8(dy_t, G.dev(xc), G.dev(xs), M, N, K, m, s)
    agoq.agoq_device_status()
    got = (G.gather_blocks(m, blocks, 128).numpy().reshape(-1),
           G.gather_blocks(s, blocks, 1).numpy().reshape(-1))
    _check_within_bound(oracle, dy, xc, xs, M, N, K, m0, s0, got, blocks=blocks)


def test_master_16_byte_aligned_takes_the_narrow_accesses(oracle):
    """Master codes 16 bytes off a 32-byte boundary are read and written with
    16-byte accesses instead of 32-byte ones: the same codes and scales."""
    M, N, K = 640, 384, 128
    dy, xc, xs = _gauss_inputs(oracle, M, N, K, seed=31)
    master, scales = _master(oracle, M * N, seed=32, sd=0.05)
    want = _run(dy, xc, xs, M, N, K, master, scales)
    room = torch.zeros(M * N + 64, dtype=torch.uint8, device="cuda")
    m_off = room[16:16 + M * N]
    assert m_off.data_ptr() % 32 == 16
    m_off.copy_(torch.from_numpy(master))
    s = torch.from_numpy(scales).cuda()
    agoq.agoq_wgrad_gemm_int4_accum_fp8(G.dev_bf16(dy), G.dev(xc), G.dev(xs), M, N, K, m_off, s)
    agoq.agoq_device_status()
    _assert_same((m_off.cpu().numpy(), s.cpu().numpy()), want)
    assert not room[:16].any() and not room[16 + M * N:].any()
