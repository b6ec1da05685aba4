"""GPU parity of the QuanGrad accumulation with a BF16 or FP16 intermediate
(agoq_grad_accum_fp8_mid) against the CPU oracle: bit-exact codes and scales."""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
MIDS = [agoq.MID_BF16, agoq.MID_FP16]


@pytest.mark.parametrize("mid", MIDS)
@pytest.mark.parametrize("nblocks", [1, 3, 33, 1031])
def test_mid_accum_parity_over_steps(oracle, mid, nblocks):
    n = nblocks * 128
    m_np = np.zeros(n, np.uint8)
    s_np = np.zeros(nblocks, np.float32)
    m = torch.zeros(n, dtype=torch.uint8, device="cuda")
    s = torch.zeros(nblocks, dtype=torch.float32, device="cuda")
    for g in synthetic.quangrad_grads_np(seed=2, n=n, steps=8):
        agoq.agoq_grad_accum_fp8_mid(m, s, G.dev_bf16(g), mid)
        m_np, s_np = oracle.grad_accum_fp8_mid(m_np, s_np, g, mid)
        assert np.array_equal(m.cpu().numpy(), m_np)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), s_np.view(np.uint32))


@pytest.mark.parametrize("mid", MIDS)
def test_mid_accum_edge_cases(oracle, mid):
    rng = np.random.default_rng(15)
    blocks = [np.zeros(128, np.uint16),                       # zero grad into zero master
              np.full(128, 0x8000, np.uint16)]                # -0 grads
    tiny = np.zeros(128, np.uint16); tiny[3] = 0x8001; tiny[9] = 0x3F80   # -tiny rounds to -0
    blocks.append(tiny)
    blocks.append(np.arange(1, 129, dtype=np.uint16))         # BF16 subnormals (FP16: zero)
    # magnitudes around the FP16 subnormal range and near its largest finite value
    blocks.append(synthetic.bf16_bits_from_f32(
        (rng.standard_normal(128) * 2.0 ** -20).astype(np.float32)))
    blocks.append(synthetic.bf16_bits_from_f32(
        rng.uniform(-30000, 30000, 128).astype(np.float32)))
    g0 = np.concatenate(blocks)
    n = g0.size
    master0 = np.zeros(n, np.uint8)
    scales0 = np.zeros(n // 128, np.float32)
    master1 = rng.integers(0, 0x7E, n).astype(np.uint8) | (rng.integers(0, 2, n) << 7).astype(np.uint8)
    scales1 = rng.uniform(1e-6, 60.0, n // 128).astype(np.float32)   # |m| <= 448 * 60 < 65504
    for mm, ss in ((master0, scales0), (master1, scales1)):
        m, s = G.dev(mm), G.dev(ss)
        agoq.agoq_grad_accum_fp8_mid(m, s, G.dev_bf16(g0), mid)
        wm, ws = oracle.grad_accum_fp8_mid(mm, ss, g0, mid)
        assert np.array_equal(m.cpu().numpy(), wm)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), ws.view(np.uint32))


def test_mid_fp32_is_the_plain_accumulation(oracle):
    n = 1 << 15
    g = next(synthetic.quangrad_grads_np(seed=4, n=n, steps=1))
    a = (torch.zeros(n, dtype=torch.uint8, device="cuda"), torch.zeros(n // 128, device="cuda"))
    b = (torch.zeros(n, dtype=torch.uint8, device="cuda"), torch.zeros(n // 128, device="cuda"))
    for _ in range(2):
        agoq.agoq_grad_accum_fp8(*a, G.dev_bf16(g))
        agoq.agoq_grad_accum_fp8_mid(*b, G.dev_bf16(g), agoq.MID_FP32)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("mid", MIDS)
def test_mid_accum_full_size_sampled_chain(oracle, mid):
    """2^30-element master, 8 micro-batches at full size; 1024 sampled blocks
    followed through all steps by the oracle; no NaN codes."""
    n = synthetic.QUANGRAD_N
    nb = n // 128
    blocks = G.sample_blocks(nb, 1024, seed=17)
    m = torch.zeros(n, dtype=torch.uint8, device="cuda")
    s = torch.zeros(nb, dtype=torch.float32, device="cuda")
    om = np.zeros(blocks.size * 128, np.uint8)
    osc = np.zeros(blocks.size, np.float32)
    for step in range(synthetic.QUANGRAD_STEPS):
        g = synthetic.quangrad_grad_torch(seed=2, step=step)
        agoq.agoq_grad_accum_fp8_mid(m, s, g, mid)
        gs = G.gather_blocks(g.view(torch.int16), blocks, 128).numpy().view(np.uint16).reshape(-1)
        om, osc = oracle.grad_accum_fp8_mid(om, osc, gs, mid)
        torch.cuda.synchronize()
        assert np.array_equal(G.gather_blocks(m, blocks, 128).numpy().reshape(-1), om), step
        assert np.array_equal(s.cpu().numpy()[blocks].view(np.uint32), osc.view(np.uint32)), step
        assert int(((m & 0x7F) == 0x7F).sum().item()) == 0
        del g


@pytest.mark.parametrize("mid", MIDS)
def test_mid_accum_guard_bands(oracle, mid):
    n = 4096
    mg = G.Guarded(n, torch.uint8)
    sg = G.Guarded(n // 128 * 4, torch.float32)
    mg.view.zero_()
    sg.view.zero_()
    g = next(synthetic.quangrad_grads_np(seed=2, n=n, steps=1))
    agoq.agoq_grad_accum_fp8_mid(mg.view, sg.view, G.dev_bf16(g), mid)
    assert mg.intact() and sg.intact()
