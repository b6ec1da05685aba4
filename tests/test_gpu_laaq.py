"""GPU parity of the LAAQ / DBCA-PP quantize and dequantize kernels against the
CPU oracle: bit-exact codes, packed bytes, scales and BF16 outputs."""
import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import agoq, synthetic
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
WIDTHS = (4, 5, 6, 8)


def _parity(oracle, xbits, bits):
    """Quantize and dequantize on the GPU; compare with the oracle bit for bit."""
    n = xbits.size
    x = G.dev_bf16(xbits)
    cg = G.Guarded(n // 128 * 16 * bits, torch.uint8)
    sg = G.Guarded(n // 128 * 4, torch.float32)
    agoq.agoq_quant_act(x, bits, cg.view, sg.view)
    want_c, want_s = oracle.quant_act(xbits.reshape(-1), bits)
    got_c = cg.view.cpu().numpy()
    got_s = sg.view.cpu().numpy()
    assert cg.intact() and sg.intact()
    assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), "scales differ"
    bad = np.flatnonzero(got_c != want_c)
    assert bad.size == 0, "codes differ at bytes %s" % bad[:10]
    # dequantize the oracle's codes on the GPU
    yg = G.Guarded(2 * n, torch.bfloat16)
    agoq.agoq_dequant_act(G.dev(want_c), G.dev(want_s), n, bits, yg.view)
    want_y = oracle.dequant_act(want_c, want_s, n, bits)
    assert yg.intact()
    assert np.array_equal(G.host_bits_bf16(yg.view), want_y)


@pytest.mark.parametrize("bits", WIDTHS)
@pytest.mark.parametrize("nblocks", [1, 2, 3, 5, 31, 33, 65, 1031])
def test_small_ragged_sizes(oracle, bits, nblocks):
    rng = np.random.default_rng(nblocks * 10 + bits)
    x = synthetic.outlier_normal_np(rng, nblocks * 128)
    _parity(oracle, synthetic.bf16_bits_from_f32(x), bits)


@pytest.mark.parametrize("bits", WIDTHS)
def test_int4_activation_workload_full(oracle, bits):
    """The 2048 x 4096 outlier-normal activation, every block checked."""
    _parity(oracle, synthetic.laaq_activation_np(seed=0), bits)


@pytest.mark.parametrize("bits", WIDTHS)
def test_dbca_student_t_reduced(oracle, bits):
    a, b = synthetic.dbca_activations_np(seed=1, tokens=128)
    _parity(oracle, a, bits)
    _parity(oracle, b, bits)


def _edge_blocks():
    blocks = []
    z = np.zeros(128, np.uint16)
    blocks.append(z)                                    # all +0
    blocks.append(np.full(128, 0x8000, np.uint16))      # all -0
    one = z.copy(); one[77] = 0xC2C8                    # single nonzero (-100)
    blocks.append(one)
    blocks.append(np.full(128, 0x3F80, np.uint16))      # all equal (1.0)
    blocks.append(np.arange(1, 129, dtype=np.uint16))   # BF16 subnormals: subnormal scale
    tiny = np.arange(128, dtype=np.uint16) % 7 | 0x0080 # smallest normals
    blocks.append(tiny)
    big = np.full(128, 0x7F7F, np.uint16); big[::3] = 0xFF7F   # +-BF16 max
    blocks.append(big)
    alt = np.where(np.arange(128) % 2 == 0, 0x4000, 0xC000).astype(np.uint16)  # +-2
    blocks.append(alt)
    return np.concatenate(blocks)


def _midpoint_blocks(bits, count, seed):
    """Blocks whose elements sit on or one BF16 step beside (k + 1/2) * scale."""
    rng = np.random.default_rng(seed)
    qmax = (1 << (bits - 1)) - 1
    out = []
    for _ in range(count):
        amax = np.float32(rng.uniform(0.25, 64.0))
        amax_b = synthetic.bf16_bits_from_f32(np.array([amax], np.float32))
        s = (torch.tensor(amax_b.view(np.int16)).view(torch.bfloat16).float() / qmax).item()
        ks = rng.integers(-qmax, qmax, 127)
        xs = synthetic.bf16_bits_from_f32(((ks + 0.5) * s).astype(np.float32)).astype(np.int32)
        xs += rng.integers(-1, 2, 127)
        out.append(np.concatenate([amax_b, xs.astype(np.uint16)]))
    return np.concatenate(out)


@pytest.mark.parametrize("bits", WIDTHS)
def test_edge_and_midpoint_blocks(oracle, bits):
    x = np.concatenate([_edge_blocks(), _midpoint_blocks(bits, 512, 40 + bits)])
    _parity(oracle, x, bits)


def test_repeatable_and_stream_ordered(oracle):
    x = G.dev_bf16(synthetic.laaq_activation_np(seed=2, tokens=64))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c1, s1 = agoq.agoq_quant_act(x, 5, stream=s)
        c2, s2 = agoq.agoq_quant_act(x, 5, stream=s)
    s.synchronize()
    assert torch.equal(c1, c2) and torch.equal(s1, s2)


def test_widths_on_two_streams_match_the_oracle(oracle):
    """The bench's step layout: widths {4, 6} on one side stream and {5, 8} on
    another, each quantizing then dequantizing its own buffers, forked from and
    joined to the main stream; every output equals the oracle's."""
    xbits = synthetic.laaq_activation_np(seed=5, tokens=96)
    n = xbits.size
    x = G.dev_bf16(xbits)
    main = torch.cuda.current_stream()
    side = [torch.cuda.Stream(), torch.cuda.Stream()]
    out = {}
    fork = torch.cuda.Event()
    fork.record(main)
    for st, widths in zip(side, ((4, 6), (5, 8))):
        st.wait_event(fork)
        with torch.cuda.stream(st):
            for b in widths:
                out[b] = agoq.agoq_quant_act(x, b)
            for b in widths:
                out[b] = out[b] + (agoq.agoq_dequant_act(out[b][0], out[b][1], n, b),)
    for st in side:
        join = torch.cuda.Event()
        join.record(st)
        main.wait_event(join)
    torch.cuda.synchronize()
    for b in WIDTHS:
        want_c, want_s = oracle.quant_act(xbits.reshape(-1), b)
        assert np.array_equal(out[b][0].cpu().numpy(), want_c)
        assert np.array_equal(out[b][1].cpu().numpy().view(np.uint32), want_s.view(np.uint32))
        assert np.array_equal(G.host_bits_bf16(out[b][2]), oracle.dequant_act(want_c, want_s, n, b))


def test_errors_raise_and_touch_nothing():
    x = torch.zeros(200, dtype=torch.bfloat16, device="cuda")
    c = torch.full((64,), 7, dtype=torch.uint8, device="cuda")
    with pytest.raises(agoq.AgoqError):
        agoq.agoq_quant_act(x, 4, c, torch.zeros(2, device="cuda"))
    with pytest.raises(agoq.AgoqError):
        agoq.agoq_quant_act(x[:128], 7, c, torch.zeros(1, device="cuda"))
    torch.cuda.synchronize()
    assert bool((c == 7).all())
    # empty input is a no-op
    agoq.agoq_quant_act(torch.zeros(0, dtype=torch.bfloat16, device="cuda"), 4)
