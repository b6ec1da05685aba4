"""Pins of the oracle's LAAQ / DBCA-PP block quantizer and dequantizer.

Checks that do not go through the oracle's own arithmetic: exact rational
brute force of the division and rounding, a bit-stream reader written with
numpy, closed forms, hand-worked fixtures and invariants of the block rule.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import synthetic
from tests import exact, golden_io

WIDTHS = (4, 5, 6, 8)


def unpack_fields(codes, n, bits):
    """Signed b-bit fields of the dense little-endian stream, via numpy.unpackbits."""
    recs = codes.reshape(n // 128, 16 * bits)
    stream = np.unpackbits(recs, axis=1, bitorder="little").reshape(n // 128, 128, bits)
    weights = (1 << np.arange(bits)).astype(np.int64)
    field = (stream.astype(np.int64) * weights).sum(axis=2)
    field = np.where(field >= (1 << (bits - 1)), field - (1 << bits), field)
    return field.reshape(-1)


def bf16_vals(bits16):
    return synthetic.bf16_tensor_from_bits(bits16).to(torch.float32).numpy()


def _brute_block(xbits, bits):
    """Codes and scale of one block by exact rational arithmetic."""
    qmax = (1 << (bits - 1)) - 1
    xs = [exact.frac(v) for v in bf16_vals(xbits)]
    absmax = max(abs(v) for v in xs)
    s = exact.to_f32(absmax / qmax)
    if absmax == 0:
        return [0] * 128, 0.0
    codes = []
    for v in xs:
        q = exact.to_f32(v / exact.frac(s))             # IEEE binary32 quotient
        c = exact.round_half_even(exact.frac(q))        # then to the nearest integer
        codes.append(max(-qmax, min(qmax, c)))
    return codes, s


def _adversarial_block(rng, bits):
    """A block whose quotients sit on or next to half-integers: x = (k + 1/2) * s
    and its BF16 neighbours, with s fixed by a planted absmax."""
    qmax = (1 << (bits - 1)) - 1
    amax = np.float32(rng.uniform(0.5, 4.0))
    s = np.float32(amax / np.float32(qmax))
    ks = rng.integers(-qmax, qmax, 127)
    target = ((ks + 0.5) * s.astype(np.float64)).astype(np.float32)
    xb = synthetic.bf16_bits_from_f32(target).astype(np.int32)
    xb = xb + rng.integers(-1, 2, 127)                  # step one BF16 ulp either way
    xb = np.concatenate([[synthetic.bf16_bits_from_f32(np.array([amax]))[0]], xb])
    return xb.astype(np.uint16)


@pytest.mark.parametrize("bits", WIDTHS)
def test_quant_matches_exact_rational_brute_force(oracle, bits):
    rng = np.random.default_rng(100 + bits)
    blocks = [synthetic.bf16_bits_from_f32(rng.standard_normal(128).astype(np.float32)),
              synthetic.bf16_bits_from_f32((rng.standard_t(4, 128) * 1e-3).astype(np.float32)),
              _adversarial_block(rng, bits), _adversarial_block(rng, bits),
              np.zeros(128, np.uint16)]
    x = np.concatenate(blocks)
    codes, scales = oracle.quant_act(x, bits)
    fields = unpack_fields(codes, x.size, bits)
    for b, xb in enumerate(blocks):
        want_codes, want_s = _brute_block(xb, bits)
        assert exact.f32_bits(float(scales[b])) == exact.f32_bits(want_s)
        assert list(fields[b * 128:(b + 1) * 128]) == want_codes


def test_rounding_reads_binary32_quotient_not_exact_quotient(oracle):
    """x/s is rounded to binary32 before the integer rounding.  Search a case
    where the exact quotient is just below k+1/2 but its binary32 rounding is the
    tie, and check that the oracle follows the binary32 quotient."""
    rng = np.random.default_rng(7)
    found = 0
    for _ in range(20000):
        amax = np.float32(rng.uniform(1, 2))
        amax = np.float32(bf16_vals(synthetic.bf16_bits_from_f32(np.array([amax])))[0])
        s = exact.to_f32(exact.frac(amax) / 7)
        k = int(rng.integers(0, 7))
        xq = exact.to_f32((k + Fraction(1, 2)) * exact.frac(s))
        xbits = synthetic.bf16_bits_from_f32(np.array([xq], np.float32))[0]
        xv = exact.frac(bf16_vals(np.array([xbits], np.uint16))[0])
        q_exact = xv / exact.frac(s)
        q32 = exact.frac(exact.to_f32(q_exact))
        if q32.denominator == 2 and q_exact != q32:
            blk = np.zeros(128, np.uint16)
            blk[0] = synthetic.bf16_bits_from_f32(np.array([amax]))[0]
            blk[1] = xbits
            codes, _ = oracle.quant_act(blk, 4)
            got = unpack_fields(codes, 128, 4)[1]
            assert got == exact.round_half_even(q32)
            found += 1
            if found >= 3:
                break
    assert found >= 1


@pytest.mark.parametrize("bits", WIDTHS)
def test_block_rule_invariants(oracle, bits):
    x = synthetic.laaq_activation_np(seed=0, tokens=64, hidden=4096).reshape(-1)
    n = x.size
    qmax = (1 << (bits - 1)) - 1
    codes, scales = oracle.quant_act(x, bits)
    assert codes.size == n // 128 * 16 * bits and scales.size == n // 128
    c = unpack_fields(codes, n, bits).reshape(-1, 128)
    xv = bf16_vals(x).astype(np.float64).reshape(-1, 128)
    s = scales.astype(np.float64)[:, None]
    # codes in range; -2^(b-1) never produced
    assert c.min() >= -qmax and c.max() <= qmax
    # the block's absmax element codes to +-qmax with its sign
    idx = np.abs(xv).argmax(axis=1)
    rows = np.arange(c.shape[0])
    assert np.array_equal(c[rows, idx], (np.sign(xv[rows, idx]) * qmax).astype(np.int64))
    # scale = fl32(absmax / qmax)
    amax = np.abs(xv).max(axis=1).astype(np.float32)
    assert np.array_equal(scales, (amax / np.float32(qmax)).astype(np.float32))
    # per-element error <= scale/2, plus the binary32 rounding of the quotient
    # (at most qmax * 2^-24 in code units, doubled for the scale's own rounding)
    err = np.abs(xv - c * s)
    assert (err <= s * (0.5 + qmax * 2.0 ** -23)).all()


@pytest.mark.parametrize("bits", WIDTHS)
def test_sign_symmetry_and_power_of_two_scaling(oracle, bits):
    x = synthetic.laaq_activation_np(seed=3, tokens=8, hidden=4096).reshape(-1)
    c0, s0 = oracle.quant_act(x, bits)
    neg = x ^ np.uint16(0x8000)
    c1, s1 = oracle.quant_act(neg, bits)
    assert np.array_equal(s0, s1)
    assert np.array_equal(unpack_fields(c1, x.size, bits), -unpack_fields(c0, x.size, bits))
    for k in (-3, 5):
        xs = synthetic.bf16_bits_from_f32(bf16_vals(x) * np.float32(2.0 ** k))
        c2, s2 = oracle.quant_act(xs, bits)
        assert np.array_equal(c2, c0)
        assert np.array_equal(s2, s0 * np.float32(2.0 ** k))


def test_int4_is_low_nibble_first(oracle):
    x = synthetic.laaq_activation_np(seed=5, tokens=4, hidden=4096).reshape(-1)
    codes, _ = oracle.quant_act(x, 4)
    lo = (codes & 0x0F).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    nib = np.stack([lo, hi], axis=1).reshape(-1)
    nib = np.where(nib >= 8, nib - 16, nib)
    assert np.array_equal(nib, unpack_fields(codes, x.size, 4))


def test_int8_is_one_int8_per_byte(oracle):
    x = synthetic.laaq_activation_np(seed=6, tokens=4, hidden=4096).reshape(-1)
    codes, _ = oracle.quant_act(x, 8)
    assert np.array_equal(codes.view(np.int8).astype(np.int64), unpack_fields(codes, x.size, 8))


@pytest.mark.parametrize("bits", WIDTHS)
def test_zero_and_signed_zero_blocks(oracle, bits):
    x = np.zeros(256, np.uint16)
    x[128:] = 0x8000                           # a block of -0
    codes, scales = oracle.quant_act(x, bits)
    assert (codes == 0).all()
    assert scales.view(np.uint32).tolist() == [0, 0]   # +0 scales
    y = oracle.dequant_act(codes, scales, 256, bits)
    assert (y == 0).all()                      # +0 outputs


@pytest.mark.parametrize("bits", WIDTHS)
def test_dequant_against_numpy_binary32_product(oracle, bits):
    """y = bf16(fl32(c * s)) restated with numpy binary32 products and torch's BF16 cast."""
    x = synthetic.laaq_activation_np(seed=8, tokens=16, hidden=4096).reshape(-1)
    codes, scales = oracle.quant_act(x, bits)
    y = oracle.dequant_act(codes, scales, x.size, bits)
    c = unpack_fields(codes, x.size, bits).astype(np.float32).reshape(-1, 128)
    prod = (c * scales[:, None]).astype(np.float32)
    assert np.array_equal(y, synthetic.bf16_bits_from_f32(prod.reshape(-1)))
    # round trip error: scale/2 from the code plus half a BF16 ulp of the output
    xv = bf16_vals(x).astype(np.float64).reshape(-1, 128)
    yv = bf16_vals(y).astype(np.float64).reshape(-1, 128)
    qmax = (1 << (bits - 1)) - 1
    bound = scales[:, None].astype(np.float64) * (0.5 + qmax * 2.0 ** -23) + np.abs(yv) * 2.0 ** -8
    assert (np.abs(xv - yv) <= bound).all()


@pytest.mark.parametrize("name", ["laaq_int4_block.txt", "laaq_int6_block.txt"])
def test_hand_worked_block(oracle, name):
    g = golden_io.read(name)
    bits = int(g["bits"][0])
    vals = np.zeros(128, np.float32)
    xs = golden_io.floats(g["x"])
    vals[:len(xs)] = xs
    x = synthetic.bf16_bits_from_f32(vals)
    codes, scales = oracle.quant_act(x, bits)
    want = np.zeros(16 * bits, np.uint8)
    wb = golden_io.hexbytes(g["bytes"])
    want[:len(wb)] = wb
    assert np.array_equal(codes, want)
    assert scales[0] == float(g["scale"][0])
    y = bf16_vals(oracle.dequant_act(codes, scales, 128, bits))
    dq = golden_io.floats(g["dequant"])
    assert list(y[:len(dq)]) == dq and not y[len(dq):].any()


def test_rejects_bad_arguments(oracle):
    with pytest.raises(ValueError):
        oracle.quant_act(np.zeros(128, np.uint16), 7)
    with pytest.raises(ValueError):
        oracle.quant_act(np.zeros(100, np.uint16), 4)
