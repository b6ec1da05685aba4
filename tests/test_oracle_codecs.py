"""Pins of the oracle's own BF16 and FP8 E4M3 codecs.

The oracle writes both codecs from the format definitions; here they are
checked against independent library casts (torch, ml_dtypes) where those
define the same mapping, and against closed-form values of the formats.
"""
import numpy as np
import pytest
import torch


def _f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def _torch_bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _sample_f32_patterns(seed=0, n_random=1 << 20):
    """All 2^16 upper halves with the lower halves that decide BF16 rounding
    (zero, one, just below/at/above the half-way point, all ones), plus random patterns."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    pats = (hi[:, None] | lows[None, :]).reshape(-1)
    rnd = np.random.default_rng(seed).integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([pats, rnd])


def test_bf16_encode_matches_torch_cast(oracle):
    pats = _sample_f32_patterns()
    x = _f32(pats)
    finite = np.isfinite(x)
    ours = oracle.f32_to_bf16(x[finite])
    ref = _torch_bf16_bits(x[finite])
    assert np.array_equal(ours, ref)
    # NaN stays NaN, infinities stay infinities.
    nonfin = x[~finite]
    back = oracle.bf16_to_f32(oracle.f32_to_bf16(nonfin))
    assert np.array_equal(np.isnan(back), np.isnan(nonfin))
    assert np.array_equal(back[np.isinf(nonfin)], nonfin[np.isinf(nonfin)])


def test_bf16_encode_closed_forms(oracle):
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2.0 ** -8: 0x3F80,            # exact tie, even (down)
        one + 3 * 2.0 ** -8: 0x3F82,        # exact tie, even (up)
        one + 2.0 ** -8 + 2.0 ** -20: 0x3F81,  # just above the tie
        -2.5: 0xC020,
        3.3895313892515355e38: 0x7F7F,      # largest BF16 stays
        -0.0: 0x8000,
        2.0 ** -133: 0x0001,                # smallest BF16 subnormal
    }
    xs = np.array(list(cases.keys()), np.float32)
    got = oracle.f32_to_bf16(xs)
    assert [int(v) for v in got] == list(cases.values())


def test_bf16_decode_exhaustive(oracle):
    h = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_decode_all_codes_against_torch(oracle):
    c = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(c)
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}


def test_e4m3_decode_all_codes_against_ml_dtypes(oracle):
    ml_dtypes = pytest.importorskip("ml_dtypes")
    c = np.arange(256, dtype=np.uint8)
    ref = c.view(ml_dtypes.float8_e4m3fn).astype(np.float32)
    ours = oracle.e4m3_to_f32(c)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_decode_closed_forms(oracle):
    v = oracle.e4m3_to_f32(np.array([0x7E, 0x01, 0x07, 0x08, 0x38, 0x80, 0xFE, 0x40], np.uint8))
    assert v[0] == 448.0                       # largest finite
    assert v[1] == 2.0 ** -9                   # smallest subnormal
    assert v[2] == 7 * 2.0 ** -9               # largest subnormal
    assert v[3] == 2.0 ** -6                   # smallest normal
    assert v[4] == 1.0
    assert v[5] == 0.0 and np.signbit(v[5])    # negative zero
    assert v[6] == -448.0
    assert v[7] == 2.0                         # exponent field 8 -> 2^(8-7)


def _e4m3_probe_values():
    """Stratified float32 values over the E4M3 range: every binade from the
    binary32 subnormals up to 2^8, 2^10 leading fraction patterns each with a few
    low patterns, both signs; plus every E4M3 midpoint and its binary32 neighbours."""
    vals = []
    lows = np.array([0, 1, 0x1FFF, 0x2000, 0x2001], np.uint32)
    for e in range(0, 127 + 9):                 # biased exponents up to 2^8
        lead = np.arange(1 << 10, dtype=np.uint32) << 13
        pats = (np.uint32(e) << 23) | (lead[:, None] | lows[None, :]).reshape(-1)
        vals.append(_f32(pats))
    mags = np.array(sorted({float(abs(v)) for v in
                            torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn)
                            .to(torch.float32).tolist()}), np.float64)
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    vals.append(mids)
    vals.append(np.nextafter(mids, np.float32(np.inf)))
    vals.append(np.nextafter(mids, np.float32(0)))
    v = np.concatenate(vals).astype(np.float32)
    v = v[np.abs(v) <= 448.0]
    return np.concatenate([v, -v])


def test_e4m3_encode_matches_torch_cast_in_range(oracle):
    v = _e4m3_probe_values()
    ours = oracle.f32_to_e4m3(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_matches_ml_dtypes_in_range(oracle):
    ml_dtypes = pytest.importorskip("ml_dtypes")
    v = _e4m3_probe_values()
    rng = np.random.default_rng(5)
    v = np.concatenate([v, rng.uniform(-448, 448, 1 << 20).astype(np.float32),
                        (rng.standard_normal(1 << 20) * 1e-2).astype(np.float32)])
    ours = oracle.f32_to_e4m3(v)
    ref = v.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_ties_and_saturation(oracle):
    m9 = 2.0 ** -9
    cases = [
        (0.5 * m9, 0x00),          # tie between 0 and 2^-9: even (0)
        (1.5 * m9, 0x02),          # tie between 1 and 2 subnormal steps: even (2)
        (7.5 * m9, 0x08),          # tie across the subnormal/normal boundary: 0x08 is even
        (432.0, 0x7E),             # tie between 416 (odd fraction) and 448 (even)
        (400.0, 0x7C),             # tie between 384 (even) and 416: 384 = 0x7C
        (448.0, 0x7E),
        (448.0 * (1 + 2.0 ** -23), 0x7E),   # saturate
        (464.0, 0x7E),
        (1e30, 0x7E),
        (3.4028234663852886e38, 0x7E),
        (-1e30, 0xFE),
        (-0.0, 0x80),
        (-1e-12, 0x80),            # negative value rounding to zero keeps its sign
        (1e-12, 0x00),
    ]
    xs = np.array([c[0] for c in cases], np.float32)
    got = oracle.f32_to_e4m3(xs)
    assert [int(g) for g in got] == [c[1] for c in cases]
