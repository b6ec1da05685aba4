"""Pins of the oracle's QuanGrad accumulation and precision-preserved local reduce.

The second restatement here uses numpy binary32 element-wise arithmetic (each
operation IEEE round-to-nearest, no fused multiply-add) and torch's E4M3 cast;
the exact-rational brute force uses tests/exact.py.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from gradient_quantization_gb300 import synthetic
from tests import exact, golden_io

E4M3 = torch.float8_e4m3fn


def e4m3_f32(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(E4M3).to(torch.float32).numpy()


def f32_e4m3(v):
    """Saturating RNE E4M3 via torch's cast: clipping to +-448 first reproduces
    saturation (values in (448, 464) round to 448 either way)."""
    v = np.clip(np.asarray(v, np.float32), -448.0, 448.0)
    return torch.from_numpy(np.ascontiguousarray(v)).to(E4M3).view(torch.uint8).numpy()


def bf16_f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def requant_restated(t):
    t = t.reshape(-1, 128).astype(np.float32)
    amax = np.abs(t).max(axis=1)
    s = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(amax == 0, np.float32(1), s).astype(np.float32)
    q = (t / safe[:, None]).astype(np.float32)
    codes = f32_e4m3(q)
    codes[amax == 0] = 0
    return codes.reshape(-1), s


def accum_restated(master, scales, g):
    m = (e4m3_f32(master).reshape(-1, 128) * scales[:, None]).astype(np.float32)
    t = (m + bf16_f32(g).reshape(-1, 128)).astype(np.float32)
    return requant_restated(t)


def reduce_restated(shards, shard_scales, W, n):
    acc = np.zeros((n // 128, 128), np.float32)
    for r in range(W):
        v = (e4m3_f32(shards[r]).reshape(-1, 128) * shard_scales[r][:, None]).astype(np.float32)
        acc = (acc + v).astype(np.float32)
    return requant_restated(acc)


def make_shards(oracle, W, n, seed=3):
    """Shards quantized from seeded BF16 values with the accumulation's requant rule."""
    vals = synthetic.reduce_shard_values_np(seed=seed, W=W, n=n)
    codes = np.empty((W, n), np.uint8)
    scales = np.empty((W, n // 128), np.float32)
    for r in range(W):
        codes[r], scales[r] = oracle.grad_accum_fp8(np.zeros(n, np.uint8),
                                                    np.zeros(n // 128, np.float32), vals[r])
    return codes, scales


# ------------------------------------------------------------------ accumulation
def test_accum_matches_numpy_restatement_over_steps(oracle):
    n = 1 << 16
    master = np.zeros(n, np.uint8)
    scales = np.zeros(n // 128, np.float32)
    for g in synthetic.quangrad_grads_np(seed=2, n=n, steps=8):
        want = accum_restated(master, scales, g)
        master, scales = oracle.grad_accum_fp8(master, scales, g)
        assert np.array_equal(master, want[0])
        assert np.array_equal(scales.view(np.uint32), want[1].view(np.uint32))


def test_accum_hand_worked_block(oracle):
    gold = golden_io.read("quangrad_e4m3_block.txt")
    vals = np.zeros(128, np.float32)
    gv = golden_io.floats(gold["grad"])
    vals[:len(gv)] = gv
    g = synthetic.bf16_bits_from_f32(vals)
    m, s = oracle.grad_accum_fp8(np.zeros(128, np.uint8), np.zeros(1, np.float32), g)
    want = np.zeros(128, np.uint8)
    wc = golden_io.hexbytes(gold["codes"])
    want[:len(wc)] = wc
    assert np.array_equal(m, want)
    assert s[0] == float(gold["scale"][0])


def test_accum_exact_rational_brute_force(oracle):
    rng = np.random.default_rng(11)
    n = 256
    master0 = f32_e4m3(rng.uniform(-448, 448, n).astype(np.float32))
    scales0 = rng.uniform(1e-6, 1e-3, n // 128).astype(np.float32)
    g = synthetic.bf16_bits_from_f32((rng.standard_normal(n) * 1e-2).astype(np.float32))
    m, s = oracle.grad_accum_fp8(master0, scales0, g)
    for b in range(n // 128):
        sb = exact.frac(scales0[b])
        t = []
        for i in range(128):
            k = b * 128 + i
            mv = exact.to_f32(exact.e4m3_value(int(master0[k])) * sb)
            t.append(exact.to_f32(exact.frac(mv) + exact.frac(bf16_f32(g[k:k + 1])[0])))
        amax = max(abs(exact.frac(v)) for v in t)
        s2 = exact.to_f32(amax / 448)
        assert exact.f32_bits(float(s[b])) == exact.f32_bits(s2)
        for i, tv in enumerate(t):
            q = exact.to_f32(exact.frac(tv) / exact.frac(s2))
            want = exact.to_e4m3_code(exact.frac(q), negative_zero=np.signbit(q))
            assert int(m[b * 128 + i]) == want


def _half_e4m3_step(q):
    """Half the E4M3 spacing at |q| (q in code units, |q| <= 448)."""
    q = np.abs(q)
    e = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
    return np.where(q < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))


def test_accum_never_overflows_where_naive_fp8_does(oracle):
    """8 micro-batches with 0.01% x1000 outliers: QuanGrad codes stay finite and
    each step lands within half an E4M3 step of (previous master + gradient); a
    naive FP8 master that keeps the first step's block scale and adds in the FP8
    code domain overflows."""
    n = 1 << 18
    master = np.zeros(n, np.uint8)
    scales = np.zeros(n // 128, np.float32)
    exact_sum = np.zeros(n, np.float64)
    naive = None
    naive_scale = None
    naive_overflow = np.zeros(n, bool)
    for g in synthetic.quangrad_grads_np(seed=2, n=n, steps=8):
        gf = bf16_f32(g)
        exact_sum += gf
        prev = (e4m3_f32(master).reshape(-1, 128) * scales[:, None]).reshape(-1).astype(np.float64)
        master, scales = oracle.grad_accum_fp8(master, scales, g)
        assert not np.isin(master, [0x7F, 0xFF]).any()
        t = prev + gf
        s = np.repeat(scales.astype(np.float64), 128)
        deq = (e4m3_f32(master).reshape(-1, 128) * scales[:, None]).reshape(-1).astype(np.float64)
        q = np.divide(np.abs(t), s, out=np.zeros_like(t), where=s > 0)
        bound = _half_e4m3_step(q) * s * (1 + 2.0 ** -20) + np.abs(t) * 2.0 ** -22
        assert (np.abs(deq - t) <= bound).all()
        if naive is None:
            amax = np.abs(gf.reshape(-1, 128)).max(axis=1)
            naive_scale = np.where(amax == 0, 1, amax / 448.0).astype(np.float32)
            naive = e4m3_f32(f32_e4m3(gf.reshape(-1, 128) / naive_scale[:, None])).reshape(-1)
            continue
        tn = naive + (gf.reshape(-1, 128) / naive_scale[:, None]).reshape(-1)
        naive_overflow |= np.abs(tn) > 448
        naive = e4m3_f32(f32_e4m3(tn))
    assert naive_overflow.sum() > 0
    deq = (e4m3_f32(master).reshape(-1, 128) * scales[:, None]).reshape(-1).astype(np.float64)
    rel = np.linalg.norm(deq - exact_sum) / np.linalg.norm(exact_sum)
    assert rel < 0.05


def test_accum_zero_grad_requantizes_within_one_step(oracle):
    rng = np.random.default_rng(12)
    n = 1 << 14
    master = f32_e4m3(rng.uniform(-448, 448, n).astype(np.float32))
    master[np.isin(master, [0x7F, 0xFF])] = 0
    scales = rng.uniform(1e-5, 1e-2, n // 128).astype(np.float32)
    m2, s2 = oracle.grad_accum_fp8(master, scales, np.zeros(n, np.uint16))
    before = (e4m3_f32(master).reshape(-1, 128) * scales[:, None]).astype(np.float64)
    after = (e4m3_f32(m2).reshape(-1, 128) * s2[:, None]).astype(np.float64)
    q = np.abs(before / s2[:, None].astype(np.float64))
    ulp = np.where(q < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(q, 2.0 ** -6))) - 3))
    assert (np.abs(after - before) <= (0.5 * ulp + q * 2.0 ** -21) * s2[:, None]).all()


# ------------------------------------------------------------------ local reduce
@pytest.mark.parametrize("W", [1, 2, 8, 13])
def test_reduce_matches_numpy_restatement(oracle, W):
    n = 1 << 14
    shards, ss = make_shards(oracle, W, n)
    out, outs, _ = oracle.reduce_fp8_shards(shards, ss, W, n)
    want = reduce_restated(shards, ss, W, n)
    assert np.array_equal(out, want[0])
    assert np.array_equal(outs.view(np.uint32), want[1].view(np.uint32))


def test_reduce_single_shard_is_requant_of_that_shard(oracle):
    n = 1 << 13
    shards, ss = make_shards(oracle, 1, n)
    out, outs, cnt = oracle.reduce_fp8_shards(shards, ss, 1, n)
    m, s = oracle.grad_accum_fp8(shards[0], ss[0], np.zeros(n, np.uint16))
    assert np.array_equal(out, m) and np.array_equal(outs, s) and cnt == 0


def test_reduce_within_one_requantization_step_of_exact_sum(oracle):
    W, n = 8, 1 << 14
    shards, ss = make_shards(oracle, W, n)
    out, outs, _ = oracle.reduce_fp8_shards(shards, ss, W, n)
    vals = np.stack([(e4m3_f32(shards[r]).reshape(-1, 128) * ss[r][:, None]).astype(np.float64)
                     for r in range(W)])
    exact_sum = vals.sum(axis=0)
    sum_abs = np.abs(vals).sum(axis=0)
    s = outs.astype(np.float64)[:, None]
    deq = e4m3_f32(out).reshape(-1, 128) * s
    q = np.abs(exact_sum) / s
    ulp = np.where(q < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(q, 2.0 ** -6))) - 3))
    bound = 0.5 * ulp * s + W * 2.0 ** -24 * sum_abs * 2 + q * s * 2.0 ** -20
    assert (np.abs(deq - exact_sum) <= bound).all()


def test_reduce_rank_order_is_honoured(oracle):
    """Binary32 addition is not associative: reversing the shard order changes
    some output, so the oracle must be summing in the stated rank order."""
    W, n = 8, 1 << 14
    shards, ss = make_shards(oracle, W, n)
    a = oracle.reduce_fp8_shards(shards, ss, W, n)
    b = oracle.reduce_fp8_shards(shards[::-1].copy(), ss[::-1].copy(), W, n)
    assert not (np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]))
    want = reduce_restated(shards, ss, W, n)
    assert np.array_equal(a[0], want[0])


def test_reduce_naive_overflow_exact_brute_force(oracle):
    W, n = 8, 256
    shards, ss = make_shards(oracle, W, n, seed=21)
    _, _, cnt = oracle.reduce_fp8_shards(shards, ss, W, n)
    want = 0
    for i in range(n):
        acc = exact.e4m3_value(int(shards[0, i]))
        for r in range(1, W):
            t = acc + exact.e4m3_value(int(shards[r, i]))
            if abs(t) > 448:
                want += 1
                break
            acc = exact.e4m3_value(exact.to_e4m3_code(t))
    assert cnt == want and want > 0


def test_reduce_naive_overflow_is_common_on_shard_workload(oracle):
    W, n = 8, 1 << 16
    shards, ss = make_shards(oracle, W, n)
    _, _, cnt = oracle.reduce_fp8_shards(shards, ss, W, n)
    assert 0.2 * n < cnt < 0.8 * n


def test_reduce_hand_worked(oracle):
    gold = golden_io.read("reduce_two_shards.txt")
    sh = np.zeros((2, 128), np.uint8)
    c0 = golden_io.hexbytes(gold["shard0_codes"])
    c1 = golden_io.hexbytes(gold["shard1_codes"])
    sh[0, :len(c0)] = c0
    sh[1, :len(c1)] = c1
    ss = np.array(golden_io.floats(gold["shard_scales"]), np.float32).reshape(2, 1)
    out, outs, cnt = oracle.reduce_fp8_shards(sh, ss, 2, 128)
    want = np.zeros(128, np.uint8)
    oc = golden_io.hexbytes(gold["out_codes"])
    want[:len(oc)] = oc
    assert np.array_equal(out, want)
    assert outs[0] == float(gold["out_scale"][0])
    assert cnt == int(gold["naive_overflow"][0])
