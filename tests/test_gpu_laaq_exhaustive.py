"""Exhaustive check of LAAQ quantization over the whole BF16 input domain.

Every positive finite BF16 value a (0x0001 .. 0x7F7F) is made a block absmax,
and every BF16 x with |x| <= a (both signs) appears in one of a's blocks, so
each (x, absmax) pair -- about 1.07e9 -- is quantized at 4, 5, 6 and 8 bits
through agoq_quant_act.  The expected codes are the definition restated with
torch on the GPU: scale = fl32(absmax / qmax), code = round-half-even of the
IEEE binary32 quotient fl32(x / scale), clamped; codes and scales must match
bit for bit.  This pins the kernel's fast quotient paths (reciprocal with a
correction step, bracketing) for every input they can see, not a sample.
"""
import pytest
import torch

from gradient_quantization_gb300 import agoq

pytestmark = pytest.mark.gpu

AMAX_LAST = 0x7F7F          # largest finite positive BF16 bit pattern


def _unpack(codes, nblocks, bits):
    """Signed b-bit fields of the dense little-endian stream, on the GPU."""
    rec = codes.view(nblocks, 16 * bits)
    shifts = torch.arange(8, device=codes.device, dtype=torch.uint8)
    stream = (rec.unsqueeze(-1) >> shifts) & 1                      # [nb, 16b, 8]
    fields = stream.reshape(nblocks, 128, bits).to(torch.int32)
    weights = (1 << torch.arange(bits, device=codes.device, dtype=torch.int32))
    v = (fields * weights).sum(-1)
    return torch.where(v >= (1 << (bits - 1)), v - (1 << bits), v)


def _blocks_for(a_lo, a_hi, device):
    """BF16 bit patterns [nb, 128] covering absmax values a in [a_lo, a_hi): element 0
    of each block is +-a, elements 1..127 run through 0..a and -0..-a (padded with +0)."""
    a = torch.arange(a_lo, a_hi, device=device, dtype=torch.int64)
    count = 2 * (a + 1)                                  # |x| <= a, both signs
    nblk = (count + 126) // 127
    a_of_block = torch.repeat_interleave(a, nblk)
    first = torch.cumsum(nblk, 0) - nblk
    idx_in_a = torch.arange(a_of_block.numel(), device=device) - torch.repeat_interleave(first, nblk)
    k = idx_in_a[:, None] * 127 + torch.arange(127, device=device)[None, :]
    aa = a_of_block[:, None]
    pos = k <= aa
    x = torch.where(pos, k, (k - aa - 1) | 0x8000)
    x = torch.where(k < 2 * (aa + 1), x, torch.zeros_like(x))
    head = torch.where((idx_in_a % 2) == 0, a_of_block, a_of_block | 0x8000)[:, None]
    bits16 = torch.cat([head, x], dim=1).to(torch.int32)
    return bits16.to(torch.int16).view(torch.bfloat16)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_every_bf16_pair(bits):
    dev = torch.device("cuda")
    qmax = (1 << (bits - 1)) - 1
    checked = 0
    step = 2048                                          # absmax values per chunk
    for a_lo in range(1, AMAX_LAST + 1, step):
        a_hi = min(a_lo + step, AMAX_LAST + 1)
        x = _blocks_for(a_lo, a_hi, dev)
        nb = x.shape[0]
        codes, scales = agoq.agoq_quant_act(x, bits)
        xf = x.float()
        am = xf.abs().amax(dim=1)
        # a tensor divisor: torch turns division by a Python scalar into a multiply
        # by its reciprocal, which is not the IEEE quotient the definition needs
        s = am / torch.full_like(am, float(qmax))
        want = torch.round(xf / s[:, None]).clamp_(-qmax, qmax).to(torch.int32)
        assert torch.equal(scales.view(torch.int32), s.view(torch.int32)), "scales, chunk %d" % a_lo
        got = _unpack(codes, nb, bits)
        bad = (got != want).nonzero()
        assert bad.numel() == 0, "bits %d: first mismatch block %s" % (bits, bad[:1].tolist())
        checked += nb * 128
        del x, codes, scales, xf, got, want
    assert checked > 1.0e9
