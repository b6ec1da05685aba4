"""Every pair of BF16 values (t, absmax) with |t| <= absmax through the
requantization of BF16-valued sums.

The QuanGrad accumulation forms the new codes e4m3_rne(fl(t/s)), s =
fl(absmax/448), in two ways: a reciprocal product bracketed on both sides with
IEEE division where the bracket straddles an E4M3 rounding boundary (binary32
sums), and Markstein's corrected quotient without a bracket when every t is a
BF16 value (the BF16 intermediate, and a binary32 sum onto an all-zero master
block, where t = 0 + g).  The second is exact only if the corrected quotient
equals the IEEE quotient, which is checked here for every pair: the gradient
blocks hold absmax at element 0 and every BF16 value of magnitude <= absmax,
both signs, in the other 127 slots, for every positive finite BF16 absmax.
The same gradient is accumulated onto a zero master (corrected quotient, both
for binary32 and for the BF16 intermediate) and onto a master with zero codes
and scale 1 (the products are +0, so t = g again, but the block takes the
bracketed path, which the parity tests pin to the oracle); codes and scales
must agree bit for bit.  A sum onto a zero master is never -0 (+0 + -0 = +0),
so the BF16 intermediate also runs onto a master of -0 codes (0x80) and scale
1, where t = -0 + g keeps a -0 gradient, against the bracketed binary32 path
on the same master.  The FP16 intermediate takes the corrected quotient onto a
zero master, where t = fp16(g), a value with at most 8 significant bits; it is
compared with the same FP16 sums onto a master of zero codes and scale 1 (the
bracketed path), for every absmax within the FP16 range (an FP16 overflow is
outside the contract).
"""
import pytest
import torch

from gradient_quantization_gb300 import agoq

pytestmark = pytest.mark.gpu

SLOTS = 127   # t values per block besides the absmax element
FP16_TOP = 0x4780   # BF16 patterns below this are at most 65280, within the FP16 range


def _blocks(a_lo, a_hi, device="cuda"):
    """BF16 gradient bit patterns (int16) for absmax patterns a_lo .. a_hi - 1."""
    a = torch.arange(a_lo, a_hi, dtype=torch.int64, device=device)
    count = 2 * (a + 1)                           # magnitudes 0 .. a, both signs
    nblk = (count + SLOTS - 1) // SLOTS
    start = torch.cumsum(nblk, 0) - nblk
    nb = int(nblk.sum())
    b = torch.arange(nb, dtype=torch.int64, device=device)
    ai = torch.searchsorted(start, b, right=True) - 1
    j = b - start[ai]
    k = j[:, None] * SLOTS + torch.arange(SLOTS, dtype=torch.int64, device=device)[None, :]
    valid = k < count[ai][:, None]
    mag = torch.where(valid, k // 2, torch.zeros_like(k))
    sign = torch.where(valid, k % 2, torch.zeros_like(k))
    t = (sign << 15) | mag
    blocks = torch.cat([a[ai][:, None], t], dim=1)   # element 0: the absmax
    return blocks.reshape(-1).to(torch.int32).to(torch.int16).view(torch.bfloat16)


def _accum(g, scale, mid=None, code=0):
    n = g.numel()
    m = torch.full((n,), code, dtype=torch.uint8, device="cuda")
    s = torch.full((n // 128,), scale, dtype=torch.float32, device="cuda")
    if mid is None:
        agoq.agoq_grad_accum_fp8(m, s, g)
    else:
        agoq.agoq_grad_accum_fp8_mid(m, s, g, mid)
    return m, s


def test_corrected_quotient_equals_bracketed_path_for_every_bf16_pair():
    top = 0x7F80                                   # patterns 1 .. 0x7F7F: positive finite
    edges = [1, 0x3000, 0x3C00, 0x4400, FP16_TOP, 0x4C00, 0x5400, 0x6000, 0x6C00, top]
    total = 0
    for lo, hi in zip(edges[:-1], edges[1:]):
        g = _blocks(lo, hi)
        total += g.numel()
        want_m, want_s = _accum(g, 1.0)              # bracketed requantization
        neg_m, neg_s = _accum(g, 1.0, code=0x80)     # bracketed, t = -0 + g
        cases = [(None, 0, (want_m, want_s)), (agoq.MID_BF16, 0, (want_m, want_s)),
                 (agoq.MID_BF16, 0x80, (neg_m, neg_s))]
        if hi <= FP16_TOP:
            cases.append((agoq.MID_FP16, 0, _accum(g, 1.0, agoq.MID_FP16)))   # bracketed FP16 sums
        for mid, code, ref in cases:
            m, s = _accum(g, 0.0 if code == 0 else 1.0, mid, code)   # corrected quotient
            assert torch.equal(s.view(torch.int32), ref[1].view(torch.int32)), (lo, hi, mid, code)
            bad = (m != ref[0]).nonzero()
            assert bad.numel() == 0, (lo, hi, mid, code, bad[:4].flatten().tolist())
            del m, s
        del g, want_m, want_s, neg_m, neg_s, cases
    agoq.agoq_device_status()
    assert total > 1_000_000_000                     # every pair was there
