"""Full-size parity of the named workloads: every element of the GPU result
against the CPU oracle, on the seeded numpy inputs (seeds 1-4, the chunked
PCG64 recipe of gradient_quantization_gb300/synthetic.py) and in the launch
configurations the bench times.

  * DBCA-PP activations, RMSNorm input [8192 x 4096] and SiLU/gate input
    [8192 x 11008] (Student-t, seed 1): quantize and dequantize at 4, 5, 6 and
    8 bits; every code byte, scale and BF16 output bit-exact.
  * QuanGrad accumulation of 2^30 elements, 8 micro-batches from a zeroed
    master (seed 2): master codes and scales bit-exact after every step.
  * FP8 shard local reduce, W = 8 and W = 64 shards of 2^25 elements (seed 3,
    shards quantized by the oracle's E4M3 block rule): output codes, scales and
    the naive-overflow count bit-exact.
  * INT4-dequant-fused weight-gradient GEMM 11008 x 4096 x 8192 (seed 4):
    every entry of the BF16 output against bf16(binary64 product) (relative
    Frobenius <= 1e-3), and every entry of the FP32-output variant within the
    binary32 summation bound K * 2^-23 * sum|terms| of the binary64 product.

The oracle runs its all-core (OpenMP) build here when the toolchain has one;
it computes the same bits as the single-threaded build (tests/test_oracle_parallel.py).
"""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def par(oracle):
    return oracle.parallel_available()


def _u32(a):
    return np.ascontiguousarray(a).view(np.uint32)


def test_dbca_activations_every_block(oracle, par):
    rms, silu = synthetic.dbca_activations_np(seed=1)
    for x in (rms.reshape(-1), silu.reshape(-1)):
        n = x.size
        xd = G.dev_bf16(x)
        for bits in (4, 5, 6, 8):
            codes, scales = agoq.agoq_quant_act(xd, bits)
            y = agoq.agoq_dequant_act(codes, scales, n, bits)
            want_c, want_s = oracle.quant_act(x, bits, parallel=par)
            assert np.array_equal(codes.cpu().numpy(), want_c), "codes, %d bits" % bits
            assert np.array_equal(_u32(scales.cpu().numpy()), _u32(want_s)), "scales, %d bits" % bits
            want_y = oracle.dequant_act(want_c, want_s, n, bits, parallel=par)
            assert np.array_equal(G.host_bits_bf16(y), want_y), "dequantized, %d bits" % bits
            del codes, scales, y, want_c, want_s, want_y
        del xd


def test_quangrad_eight_steps_every_block(oracle, par):
    n = synthetic.QUANGRAD_N
    m = torch.zeros(n, dtype=torch.uint8, device="cuda")
    s = torch.zeros(n // 128, dtype=torch.float32, device="cuda")
    om = np.zeros(n, np.uint8)
    osc = np.zeros(n // 128, np.float32)
    for step in range(synthetic.QUANGRAD_STEPS):
        g = synthetic.quangrad_grad_np(seed=2, step=step)
        gd = G.dev_bf16(g)
        agoq.agoq_grad_accum_fp8(m, s, gd)
        oracle.grad_accum_fp8(om, osc, g, parallel=par, in_place=True)
        del g, gd
        assert np.array_equal(m.cpu().numpy(), om), "master codes, step %d" % step
        assert np.array_equal(_u32(s.cpu().numpy()), _u32(osc)), "master scales, step %d" % step
    assert not ((om & 0x7F) == 0x7F).any()          # no NaN codes after 8 steps


@pytest.mark.parametrize("W", synthetic.REDUCE_WS)
def test_reduce_every_block_and_count(oracle, par, W):
    n = synthetic.REDUCE_N
    vals = synthetic.reduce_shard_values_np(seed=3, W=W, n=n)
    sh = np.zeros((W, n), np.uint8)
    ss = np.zeros((W, n // 128), np.float32)
    for r in range(W):
        oracle.grad_accum_fp8(sh[r], ss[r], vals[r], parallel=par, in_place=True)
    del vals
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    out, outs = agoq.agoq_reduce_fp8_shards(G.dev(sh), G.dev(ss), W, n, naive_overflow_count=cnt)
    agoq.agoq_device_status()
    wc, ws, wcnt = oracle.reduce_fp8_shards(sh, ss, W, n, parallel=par)
    assert np.array_equal(out.cpu().numpy(), wc)
    assert np.array_equal(_u32(outs.cpu().numpy()), _u32(ws))
    assert int(cnt.item()) == wcnt and wcnt > 0


def test_wgrad_gemm_every_entry(oracle, par):
    M, N, K = synthetic.WGRAD_M, synthetic.WGRAD_N, synthetic.WGRAD_K
    dy, x = synthetic.wgrad_inputs_np(seed=4)
    xc, xs = oracle.quant_act(x.reshape(-1), 4, parallel=par)
    del x
    dyd, xcd, xsd = G.dev_bf16(dy), G.dev(xc), G.dev(xs)
    dw = agoq.agoq_wgrad_gemm_int4(dyd, xcd, xsd, M, N, K)
    f32 = agoq.agoq_wgrad_gemm_int4_f32out(dyd, xcd, xsd, M, N, K)
    agoq.agoq_device_status()
    got = dw.double().cpu().numpy()
    got32 = f32.double().cpu().numpy()
    del dyd, dw, f32
    ref = oracle.wgrad_gemm_int4_f64_matmul(dy, xc, xs, M, N, K)
    ref_b = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert np.linalg.norm(got - ref_b) / np.linalg.norm(ref_b) <= 1e-3
    assert np.linalg.norm(got32 - ref) / np.linalg.norm(ref) <= 1e-3
    del got, ref_b
    mag = oracle.wgrad_gemm_int4_f64_matmul(dy, xc, xs, M, N, K, absolute=True)
    assert (np.abs(got32 - ref) <= K * 2.0 ** -23 * mag + 1e-30).all()
