"""Pins of the oracle's QuanGrad accumulation with a BF16 or FP16 intermediate
and of its rounding to those formats.

The rounding is checked against numpy's float16 casts (from binary32 and
binary64), torch's bfloat16 cast and exact-rational rounding at and next to
every kind of midpoint; the accumulation against an exact-rational brute force
and a numpy/torch restatement in the formats' own arithmetic.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import synthetic
from tests import exact
from tests.test_oracle_quangrad import e4m3_f32, f32_e4m3, requant_restated

MID_BF16, MID_FP16 = 1, 2


def _stratified_f32(rng, lo_exp, hi_exp, n):
    """Random finite binary32 values spread over binades 2^lo_exp .. 2^hi_exp
    (exponent -127 gives binary32 subnormals), both signs."""
    assert -127 <= lo_exp < hi_exp <= 128
    e = rng.integers(lo_exp, hi_exp, n)
    m = rng.integers(0, 1 << 23, n)
    bits = ((e + 127).astype(np.uint32) << 23) | m.astype(np.uint32)
    v = bits.view(np.float32).copy()
    v[rng.random(n) < 0.5] *= -1
    return v


def test_fp16_rounding_of_binary32_matches_numpy(oracle):
    rng = np.random.default_rng(41)
    v = np.concatenate([_stratified_f32(rng, -30, 17, 1 << 18),
                        np.array([65504, 65519.996, 65520, 2 ** -24, 2 ** -25, 3 * 2 ** -26,
                                  2 ** -14, 2 ** -14 - 2 ** -25, 0.0, -0.0], np.float32)])
    got = oracle.round_format(v.astype(np.float64), MID_FP16)
    with np.errstate(over="ignore"):                 # values beyond 65504 become inf
        want = v.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, want)


def test_fp16_rounding_of_binary64_near_midpoints_matches_numpy(oracle):
    """Binary64 values a hair off FP16 midpoints: rounding through binary32 first
    would land on the midpoint and tie the wrong way."""
    rng = np.random.default_rng(42)
    h = rng.integers(0, 0x7BFF, 4096).astype(np.uint16)            # finite positive halves
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    v = np.concatenate([mid, mid * (1 + 2.0 ** -40), mid * (1 - 2.0 ** -40), -mid])
    got = oracle.round_format(v, MID_FP16)
    assert np.array_equal(got, v.astype(np.float16).astype(np.float64))


def test_bf16_rounding_of_binary32_matches_torch(oracle):
    rng = np.random.default_rng(43)
    v = _stratified_f32(rng, -127, 128, 1 << 18)
    got = oracle.round_format(v.astype(np.float64), MID_BF16)
    want = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, want)


def test_rounding_exact_rational_near_midpoints(oracle):
    rng = np.random.default_rng(44)
    for fmt, mid in ((exact.BF16_FORMAT, MID_BF16), (exact.FP16_FORMAT, MID_FP16)):
        p, emin, emax = fmt
        vals = []
        for _ in range(300):
            e = int(rng.integers(emin - p + 1, emax + 1))
            k = int(rng.integers(1 << (p - 1), 1 << p))
            q = Fraction(2 * k + 1, 2) * Fraction(2) ** (max(e, emin) - (p - 1))   # a midpoint
            for d in (Fraction(0), Fraction(1, 1 << 45), -Fraction(1, 1 << 45)):
                vals.append(q * (1 + d))
        got = oracle.round_format([float(x) for x in vals], mid)
        for x, g in zip(vals, got):
            want = exact.round_format(Fraction(float(x)), p, emin, emax)
            assert (g == float(want)) if not np.isinf(g) else want == np.inf, (float(x), g, want)


def _bf16_bits(rng, n, sd):
    return synthetic.bf16_bits_from_f32((rng.standard_normal(n) * sd).astype(np.float32))


def _random_master(rng, n):
    return (f32_e4m3(rng.uniform(-448, 448, n).astype(np.float32)),
            rng.uniform(1e-5, 1e-2, n // 128).astype(np.float32))


@pytest.mark.parametrize("mid,fmt", [(MID_BF16, exact.BF16_FORMAT), (MID_FP16, exact.FP16_FORMAT)])
def test_mid_accum_exact_rational_brute_force(oracle, mid, fmt):
    rng = np.random.default_rng(45 + mid)
    n = 256
    master, scales = _random_master(rng, n)
    g = _bf16_bits(rng, n, 2e-2)
    m, s = oracle.grad_accum_fp8_mid(master, scales, g, mid)
    gv = (g.astype(np.uint32) << 16).view(np.float32)
    for b in range(n // 128):
        sb = exact.frac(scales[b])
        t = []
        for i in range(128):
            k = b * 128 + i
            m32 = exact.to_f32(exact.e4m3_value(int(master[k])) * sb)
            mm = exact.round_format(exact.frac(m32), *fmt)
            gg = exact.round_format(exact.frac(gv[k]), *fmt)
            t.append(float(exact.round_format(mm + gg, *fmt)))
        amax = max(abs(exact.frac(v)) for v in t)
        s2 = exact.to_f32(amax / 448)
        assert exact.f32_bits(float(s[b])) == exact.f32_bits(s2)
        for i, tv in enumerate(t):
            q = exact.to_f32(exact.frac(tv) / exact.frac(s2))
            want = exact.to_e4m3_code(exact.frac(q), negative_zero=np.signbit(q))
            assert int(m[b * 128 + i]) == want


def _mid_restated(master, scales, g, mid):
    """numpy float16 / torch bfloat16 element-wise arithmetic: each of these
    libraries rounds the binary32 sum of two format values, which for such
    operands equals the rounding of the exact sum."""
    m32 = (e4m3_f32(master).reshape(-1, 128) * scales[:, None]).astype(np.float32).reshape(-1)
    g32 = (g.astype(np.uint32) << 16).view(np.float32)
    if mid == MID_FP16:
        t = (m32.astype(np.float16) + g32.astype(np.float16)).astype(np.float32)
    else:
        tb = torch.from_numpy(m32).to(torch.bfloat16) + torch.from_numpy(g32).to(torch.bfloat16)
        t = tb.float().numpy()
    return requant_restated(t)


@pytest.mark.parametrize("mid", [MID_BF16, MID_FP16])
def test_mid_accum_matches_format_arithmetic_over_steps(oracle, mid):
    rng = np.random.default_rng(50 + mid)
    n = 1 << 15
    master = np.zeros(n, np.uint8)
    scales = np.zeros(n // 128, np.float32)
    for step in range(4):
        g = _bf16_bits(rng, n, 1e-3)
        want = _mid_restated(master, scales, g, mid)
        master, scales = oracle.grad_accum_fp8_mid(master, scales, g, mid)
        assert np.array_equal(master, want[0])
        assert np.array_equal(scales.view(np.uint32), want[1].view(np.uint32))


def test_mid_accum_differs_from_fp32_intermediate_but_stays_close(oracle):
    """The BF16 intermediate loses bits the FP32 one keeps: results differ
    somewhere, and every dequantized value stays within one BF16 rounding of the
    master plus one of the sum plus one E4M3 step of the FP32 result."""
    rng = np.random.default_rng(60)
    n = 1 << 14
    master, scales = _random_master(rng, n)
    g = _bf16_bits(rng, n, 1e-3)
    a = oracle.grad_accum_fp8(master, scales, g)
    b = oracle.grad_accum_fp8_mid(master, scales, g, MID_BF16)
    assert not np.array_equal(a[0], b[0])
    da = e4m3_f32(a[0]).reshape(-1, 128).astype(np.float64) * a[1][:, None]
    db = e4m3_f32(b[0]).reshape(-1, 128).astype(np.float64) * b[1][:, None]
    step = np.maximum(a[1], b[1])[:, None] * 32.0          # one E4M3 step at the top binade
    assert (np.abs(da - db) <= step + 2.0 ** -7 * np.abs(da)).all()


def test_mid_rejects_unknown_format(oracle):
    with pytest.raises(ValueError):
        oracle.grad_accum_fp8_mid(np.zeros(128, np.uint8), np.zeros(1, np.float32),
                                  np.zeros(128, np.uint16), 3)
