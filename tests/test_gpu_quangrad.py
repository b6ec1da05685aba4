"""GPU parity of the QuanGrad accumulation and the FP8 shard local reduce
against the CPU oracle: bit-exact codes, scales and naive-overflow counts."""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

# ---------------------------------------------------------------- accumulation
@pytest.mark.parametrize("nblocks", [1, 3, 33, 1031, 1 << 10])
def test_accum_parity_over_steps(oracle, nblocks):
    n = nblocks * 128
    m_np = np.zeros(n, np.uint8)
    s_np = np.zeros(nblocks, np.float32)
    m = torch.zeros(n, dtype=torch.uint8, device="cuda")
    s = torch.zeros(nblocks, dtype=torch.float32, device="cuda")
    for g in synthetic.quangrad_grads_np(seed=2, n=n, steps=8):
        agoq.agoq_grad_accum_fp8(m, s, G.dev_bf16(g))
        m_np, s_np = oracle.grad_accum_fp8(m_np, s_np, g)
        assert np.array_equal(m.cpu().numpy(), m_np)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), s_np.view(np.uint32))


@pytest.mark.parametrize("nblocks", [4, 600])
def test_accum_staged_and_register_kernels_agree(oracle, nblocks):
    """The same accumulation through both kernels: master scales on a 16-byte
    boundary take the staged kernel (bulk copies; 600 blocks leave a ragged
    last tile), the same scales 4 bytes off it the register kernel; both give
    the oracle's master bit for bit over three micro-batches."""
    n = nblocks * 128
    results = []
    for off in (0, 1):
        m = torch.zeros(n, dtype=torch.uint8, device="cuda")
        room = torch.zeros(nblocks + 4, dtype=torch.float32, device="cuda")
        ms = room[off:off + nblocks]
        assert (ms.data_ptr() % 16 == 0) == (off == 0)
        wm, ws = np.zeros(n, np.uint8), np.zeros(nblocks, np.float32)
        for g in synthetic.quangrad_grads_np(seed=30 + nblocks, n=n, steps=3):
            agoq.agoq_grad_accum_fp8(m, ms, G.dev_bf16(g))
            wm, ws = oracle.grad_accum_fp8(wm, ws, g)
        agoq.agoq_device_status()
        assert np.array_equal(m.cpu().numpy(), wm)
        assert np.array_equal(ms.cpu().numpy().view(np.uint32), ws.view(np.uint32))
        results.append(m.cpu().numpy())
    assert np.array_equal(results[0], results[1])


def test_accum_edge_cases(oracle):
    rng = np.random.default_rng(5)
    blocks = []
    blocks.append(np.zeros(128, np.uint16))                   # zero grad into zero master
    blocks.append(np.full(128, 0x8000, np.uint16))            # -0 grads
    tiny = np.zeros(128, np.uint16); tiny[3] = 0x8001; tiny[9] = 0x3F80   # -tiny rounds to -0
    blocks.append(tiny)
    blocks.append(np.arange(1, 129, dtype=np.uint16))         # BF16 subnormal grads
    blocks.append(synthetic.bf16_bits_from_f32(rng.standard_normal(128).astype(np.float32) * 1e30))
    g0 = np.concatenate(blocks)
    n = g0.size
    master0 = np.zeros(n, np.uint8)
    scales0 = np.zeros(n // 128, np.float32)
    # a second step on top of random non-zero masters
    master1 = rng.integers(0, 0x7E, n).astype(np.uint8) | (rng.integers(0, 2, n) << 7).astype(np.uint8)
    scales1 = rng.uniform(1e-6, 1.0, n // 128).astype(np.float32)
    for (mm, ss) in ((master0, scales0), (master1, scales1)):
        m = G.dev(mm)
        s = G.dev(ss)
        agoq.agoq_grad_accum_fp8(m, s, G.dev_bf16(g0))
        wm, ws = oracle.grad_accum_fp8(mm, ss, g0)
        assert np.array_equal(m.cpu().numpy(), wm)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), ws.view(np.uint32))


def test_accum_guard_bands(oracle):
    n = 4096
    mg = G.Guarded(n, torch.uint8)
    sg = G.Guarded(n // 128 * 4, torch.float32)
    mg.view.zero_()
    sg.view.zero_()
    g = next(synthetic.quangrad_grads_np(seed=2, n=n, steps=1))
    agoq.agoq_grad_accum_fp8(mg.view, sg.view, G.dev_bf16(g))
    assert mg.intact() and sg.intact()


# ---------------------------------------------------------------- local reduce
def _oracle_shards(oracle, W, n, seed=3):
    vals = synthetic.reduce_shard_values_np(seed=seed, W=W, n=n)
    codes = np.empty((W, n), np.uint8)
    scales = np.empty((W, n // 128), np.float32)
    for r in range(W):
        codes[r], scales[r] = oracle.grad_accum_fp8(np.zeros(n, np.uint8),
                                                    np.zeros(n // 128, np.float32), vals[r])
    return codes, scales


@pytest.mark.parametrize("W", [1, 2, 3, 8, 13, 64])
@pytest.mark.parametrize("nblocks", [1, 4, 5, 36, 37, 600, 1028])
def test_reduce_parity(oracle, W, nblocks):
    """Block counts that are multiples of 4 take the shared-memory staged kernel
    (36 and 1028: a ragged last tile), the others the register-staged one."""
    n = nblocks * 128
    sh, ss = _oracle_shards(oracle, W, n, seed=3 + W)
    og = G.Guarded(n, torch.uint8)
    osg = G.Guarded(n // 128 * 4, torch.float32)
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    agoq.agoq_reduce_fp8_shards(G.dev(sh), G.dev(ss), W, n, og.view, osg.view, cnt)
    wc, ws, wcnt = oracle.reduce_fp8_shards(sh, ss, W, n)
    assert np.array_equal(og.view.cpu().numpy(), wc)
    assert np.array_equal(osg.view.cpu().numpy().view(np.uint32), ws.view(np.uint32))
    assert int(cnt.item()) == wcnt
    assert og.intact() and osg.intact()
    # without the count: same codes
    o2, s2 = agoq.agoq_reduce_fp8_shards(G.dev(sh), G.dev(ss), W, n)
    assert np.array_equal(o2.cpu().numpy(), wc)


@pytest.mark.parametrize("W,nblocks", [(8, 600), (3, 36), (64, 100)])
def test_reduce_staged_and_register_kernels_agree(oracle, W, nblocks):
    """The same shards through both reduce kernels: scales on a 16-byte boundary
    take the staged kernel (bulk copies), the same scales 4 bytes off it the
    register-staged kernel; both equal the oracle, counts included."""
    n = nblocks * 128
    sh, ss = _oracle_shards(oracle, W, n, seed=40 + W)
    wc, ws, wcnt = oracle.reduce_fp8_shards(sh, ss, W, n)
    d_sh = G.dev(sh)
    room = torch.zeros(ss.size + 4, dtype=torch.float32, device="cuda")
    for off in (0, 1):
        ss_dev = room[off:off + ss.size]
        ss_dev.copy_(G.dev(ss))
        assert (ss_dev.data_ptr() % 16 == 0) == (off == 0)
        cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda")
        o, os_ = agoq.agoq_reduce_fp8_shards(d_sh, ss_dev, W, n, naive_overflow_count=cnt)
        assert np.array_equal(o.cpu().numpy(), wc)
        assert np.array_equal(os_.cpu().numpy().view(np.uint32), ws.view(np.uint32))
        assert int(cnt.item()) == wcnt
    agoq.agoq_device_status()   # raises if a pipeline wait timed out


def test_reduce_edge_cases(oracle):
    W, n = 4, 512
    rng = np.random.default_rng(8)
    sh = rng.integers(0, 256, (W, n)).astype(np.uint8)
    sh[(sh & 0x7F) == 0x7F] = 0x7E                       # no NaN codes
    sh[:, :128] = 0                                      # block 0: all zero
    sh[0, 128:256] = 0x80; sh[1:, 128:256] = 0           # block 1: -0 and +0
    ss = rng.uniform(1e-8, 1e3, (W, n // 128)).astype(np.float32)
    ss[:, 2] = 2.0 ** -140                               # block 2: subnormal shard scales
    # block 3: scale 2^-149, so codes below 1 in magnitude give products that
    # underflow to a signed zero (a negative one in shard 0 must still leave +0)
    ss[:, 3] = 2.0 ** -149
    sh[0, 384:448] = 0x80 | rng.integers(1, 0x38, 64)    # -(2^-9 .. <1)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    o, os_ = agoq.agoq_reduce_fp8_shards(G.dev(sh), G.dev(ss), W, n, naive_overflow_count=cnt)
    wc, ws, wcnt = oracle.reduce_fp8_shards(sh, ss, W, n)
    assert np.array_equal(o.cpu().numpy(), wc)
    assert np.array_equal(os_.cpu().numpy().view(np.uint32), ws.view(np.uint32))
    assert int(cnt.item()) == wcnt


def test_reduce_count_is_set_not_accumulated(oracle):
    W, n = 8, 128 * 64
    sh, ss = _oracle_shards(oracle, W, n)
    cnt = torch.full((1,), 12345, dtype=torch.int64, device="cuda")
    agoq.agoq_reduce_fp8_shards(G.dev(sh), G.dev(ss), W, n, naive_overflow_count=cnt)
    first = int(cnt.item())
    agoq.agoq_reduce_fp8_shards(G.dev(sh), G.dev(ss), W, n, naive_overflow_count=cnt)
    assert int(cnt.item()) == first == oracle.reduce_fp8_shards(sh, ss, W, n)[2]


# ---------------------------------------------------------------- checkpoint / resume
def test_accum_resume_from_saved_master_is_bit_identical(oracle, tmp_path):
    """The FP8 master (codes + scales) is the whole state of the accumulation:
    saving it to a file after 3 micro-batches, reloading it into fresh device
    buffers and continuing with 5 more gives the same bits as 8 uninterrupted
    micro-batches, and as the oracle."""
    nblocks = 1031
    n = nblocks * 128
    grads = list(synthetic.quangrad_grads_np(seed=9, n=n, steps=8))
    m = torch.zeros(n, dtype=torch.uint8, device="cuda")
    s = torch.zeros(nblocks, dtype=torch.float32, device="cuda")
    for g in grads:
        agoq.agoq_grad_accum_fp8(m, s, G.dev_bf16(g))
    m2 = torch.zeros(n, dtype=torch.uint8, device="cuda")
    s2 = torch.zeros(nblocks, dtype=torch.float32, device="cuda")
    for g in grads[:3]:
        agoq.agoq_grad_accum_fp8(m2, s2, G.dev_bf16(g))
    path = tmp_path / "master.npz"
    np.savez(path, codes=m2.cpu().numpy(), scales=s2.cpu().numpy())
    del m2, s2
    saved = np.load(path)
    m3 = torch.from_numpy(saved["codes"]).cuda()
    s3 = torch.from_numpy(saved["scales"]).cuda()
    for g in grads[3:]:
        agoq.agoq_grad_accum_fp8(m3, s3, G.dev_bf16(g))
    assert np.array_equal(m3.cpu().numpy(), m.cpu().numpy())
    assert np.array_equal(s3.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint32))
    m_np, s_np = np.zeros(n, np.uint8), np.zeros(nblocks, np.float32)
    for g in grads:
        m_np, s_np = oracle.grad_accum_fp8(m_np, s_np, g)
    assert np.array_equal(m.cpu().numpy(), m_np)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_np.view(np.uint32))
