"""GPU parity of the SiLU backward recomputed from LAAQ codes
(agoq_silu_backward) against the oracle's binary64 values.

Each BF16 output must lie within half a BF16 ulp plus the binary32 bound
2^-20 * |dy| * (1 + |xh|) (dx) or 2^-20 * |xh| (y) of the exact value, and at
least 99% of outputs must equal the exact value rounded to BF16.
"""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
MID_BF16 = 1


def _f64(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp_bf16(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def _check(oracle, got_bits, exact, slack):
    got = _f64(got_bits)
    tol = 0.5 * _ulp_bf16(np.maximum(np.abs(exact), np.abs(got))) + slack + 1e-40
    bad = np.flatnonzero(np.abs(got - exact) > tol)
    assert bad.size == 0, "first out of bound: %s got %r exact %r" % (bad[:3], got[bad[:3]], exact[bad[:3]])
    rounded = oracle.round_format(exact, MID_BF16)
    assert np.mean(got == rounded) >= 0.99


def _inputs(oracle, n, bits, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = synthetic.bf16_bits_from_f32((rng.standard_t(4, n) * scale).astype(np.float32))
    codes, scales = oracle.quant_act(x, bits)
    dy = synthetic.bf16_bits_from_f32(rng.standard_normal(n).astype(np.float32))
    return codes, scales, dy


def _run_and_check(oracle, codes, scales, dy, n, bits, with_y):
    dx, y = agoq.agoq_silu_backward(G.dev(codes), G.dev(scales), G.dev_bf16(dy), n, bits,
                                    want_y=with_y)
    ex_dx, ex_y = oracle.silu_backward(codes, scales, dy, n, bits)
    xh = _f64(oracle.dequant_act(codes, scales, n, bits))
    _check(oracle, G.host_bits_bf16(dx), ex_dx, 2.0 ** -20 * np.abs(_f64(dy)) * (1 + np.abs(xh)))
    if with_y:
        _check(oracle, G.host_bits_bf16(y), ex_y, 2.0 ** -20 * np.abs(xh))


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
@pytest.mark.parametrize("nblocks", [1, 37, 1031])
@pytest.mark.parametrize("with_y", [False, True])
def test_silu_backward_parity(oracle, bits, nblocks, with_y):
    n = nblocks * 128
    codes, scales, dy = _inputs(oracle, n, bits, seed=bits * 1000 + nblocks)
    _run_and_check(oracle, codes, scales, dy, n, bits, with_y)


@pytest.mark.parametrize("bits", [4, 8])
def test_silu_backward_edge_cases(oracle, bits):
    blocks = []
    rng = np.random.default_rng(3)
    for scale in (1e-30, 1e-3, 30.0, 1e4, 1e30):     # saturated and tiny sigmoid arguments
        blocks.append((rng.standard_normal(128) * scale).astype(np.float32))
    blocks.append(np.zeros(128, np.float32))           # all-zero block: xh = 0
    x = synthetic.bf16_bits_from_f32(np.concatenate(blocks))
    n = x.size
    codes, scales = oracle.quant_act(x, bits)
    dy = synthetic.bf16_bits_from_f32(rng.standard_normal(n).astype(np.float32))
    dy[::7] = 0x8000                                   # -0
    dy[1::11] = 0x0001                                 # BF16 subnormal
    _run_and_check(oracle, codes, scales, dy, n, bits, True)


def test_silu_backward_full_size_sampled(oracle):
    """The DBCA-PP SiLU input (8192 x 11008, Student-t) at 4 bits, in the bench's
    launch configuration; 4096 sampled blocks against the oracle."""
    x = synthetic.dbca_activations_torch(seed=1)[1]
    n = x.numel()
    bits = 4
    codes, scales = agoq.agoq_quant_act(x, bits)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    dy = torch.randn(n, generator=gen, device="cuda").to(torch.bfloat16)
    dx, y = agoq.agoq_silu_backward(codes, scales, dy, n, bits, want_y=True)
    blocks = G.sample_blocks(n // 128, 4096, seed=6)
    c_s = G.gather_blocks(codes, blocks, 64).numpy().reshape(-1)
    s_s = G.gather_blocks(scales, blocks, 1).numpy().reshape(-1)
    dy_s = G.gather_blocks(dy.view(torch.int16), blocks, 128).numpy().view(np.uint16).reshape(-1)
    m = blocks.size * 128
    ex_dx, ex_y = oracle.silu_backward(c_s, s_s, dy_s, m, bits)
    xh = _f64(oracle.dequant_act(c_s, s_s, m, bits))
    got_dx = G.gather_blocks(dx.view(torch.int16), blocks, 128).numpy().view(np.uint16).reshape(-1)
    got_y = G.gather_blocks(y.view(torch.int16), blocks, 128).numpy().view(np.uint16).reshape(-1)
    _check(oracle, got_dx, ex_dx, 2.0 ** -20 * np.abs(_f64(dy_s)) * (1 + np.abs(xh)))
    _check(oracle, got_y, ex_y, 2.0 ** -20 * np.abs(xh))


def test_silu_backward_guard_bands(oracle):
    n = 4096
    codes, scales, dy = _inputs(oracle, n, 5, seed=11)
    dxg = G.Guarded(2 * n, torch.bfloat16)
    yg = G.Guarded(2 * n, torch.bfloat16)
    agoq.agoq_silu_backward(G.dev(codes), G.dev(scales), G.dev_bf16(dy), n, 5, dxg.view, yg.view)
    assert dxg.intact() and yg.intact()
