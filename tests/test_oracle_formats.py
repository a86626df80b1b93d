"""Pins for the oracle's number formats and its fixed exp/SiLU sequence.

The references here are other than the oracle: torch's float8_e4m3fn and
bfloat16 casts (library routines), the OCP E4M3/E8M0 definitions written as
exact rational arithmetic, and fp64 ``math.exp``.
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch


def f32(x):
    return float(np.float32(x))


def f32_ulp(x):
    x = abs(f32(x))
    if x == 0:
        return 2.0 ** -149
    e = math.frexp(x)[1] - 1
    return 2.0 ** max(e - 23, -149)


def test_e4m3_decode_all_256_vs_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def _e4m3_grid():
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return np.unique(vals[~np.isnan(vals)])


def test_e4m3_encode_in_range_vs_torch(orc):
    g = np.random.default_rng(11)
    grid = _e4m3_grid()
    pos = grid[grid >= 0]
    mids = (pos[1:] + pos[:-1]) / 2            # exact ties: RNE decides
    xs = np.concatenate([
        grid, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
        g.standard_normal(4000) * 50, g.standard_normal(2000) * 0.01,
        g.uniform(-2.0 ** -6, 2.0 ** -6, 2000), [0.0, -0.0, 2.0 ** -10, -(2.0 ** -10), 463.9, -463.9],
    ]).astype(np.float32)
    xs = xs[np.abs(xs) < 464.0]                # torch maps values rounding past 448 to NaN
    ours = orc.e4m3_from_f32(xs)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, (xs[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_saturates_and_keeps_sign_of_zero(orc):
    # OCP E4M3: largest finite magnitude 448 = S.1111.110; saturating conversion
    big = np.array([448.0, 464.0, 480.0, 1e6, 3.0e38, np.inf], dtype=np.float32)
    assert np.all(orc.e4m3_from_f32(big) == 0x7E)
    assert np.all(orc.e4m3_from_f32(-big) == 0xFE)
    assert orc.e4m3_from_f32([-0.0])[0] == 0x80
    assert orc.e4m3_from_f32([-(2.0 ** -12)])[0] == 0x80     # underflows to -0
    assert orc.e4m3_from_f32([2.0 ** -10])[0] == 0x00        # tie at half the smallest subnormal -> even (0)
    assert orc.e4m3_from_f32([3 * 2.0 ** -10])[0] == 0x02    # 1.5 * 2^-9 -> tie -> even (2)
    assert orc.e4m3_from_f32([5 * 2.0 ** -10])[0] == 0x02    # 2.5 * 2^-9 -> tie -> even (2)
    assert orc.e4m3_from_f32([3 * 2.0 ** -11])[0] == 0x01    # 0.75 * 2^-9 -> 1


def test_bf16_encode_vs_torch(orc):
    g = np.random.default_rng(3)
    xs = np.concatenate([g.standard_normal(3000) * 10, g.standard_normal(1000) * 1e-30,
                         [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 0.0, 3.0e38]]).astype(np.float32)
    ours = orc.bf16_from_f32(xs)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = orc.bf16_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(xs).to(torch.bfloat16).float().numpy())


def test_bf16_encode_exhaustive_vs_torch(orc):
    """Every non-NaN fp32: the oracle's bf16 encoding (round to nearest even)
    equals torch's bfloat16 cast."""
    import multiprocessing as mp
    import os

    from tests.exhaustive_util import bf16_chunk_mismatches
    ch = 1 << 24
    jobs = [(s, s + ch) for s in range(0, 1 << 32, ch)]
    with mp.get_context("spawn").Pool(min(8, os.cpu_count() or 1)) as pool:
        bad = [b for r in pool.map(bf16_chunk_mismatches, jobs, chunksize=4) for b in r]
    assert not bad, [hex(b) for b in bad[:8]]


def test_e8m0_decode(orc):
    codes = np.arange(256, dtype=np.uint8)
    v = orc.e8m0_to_f64(codes)
    assert np.isnan(v[255])
    for b in (0, 1, 126, 127, 128, 254):
        assert v[b] == math.ldexp(1.0, b - 127)


def _mx_exp_bruteforce(a):
    a = Fraction(float(a))
    if a == 0:
        return 0
    e = -400
    while Fraction(448) * Fraction(2) ** e < a:
        e += 1
    return max(-127, min(127, e))


def test_mx_scale_exponent_vs_search(orc):
    g = np.random.default_rng(5)
    vals = list(np.abs(g.standard_normal(300) * 10.0 ** g.integers(-30, 30, 300)).astype(np.float32))
    vals += [448.0, 448.0 * 2, 448.0 * 0.5, 1.75, 1.75 * 1.0000001, 1.0, 0.0, 2.0 ** -149, 3.4e38,
             np.nextafter(np.float32(448.0), np.float32(0)), np.nextafter(np.float32(448.0), np.float32(1e9))]
    for a in vals:
        assert orc.mx_scale_exponent(float(np.float32(a))) == _mx_exp_bruteforce(np.float32(a)), a


def test_mx_scale_exponent_exhaustive(orc):
    """Every non-negative finite fp32 a (about 2.1e9 values): the oracle's MX
    block exponent is the smallest integer e with 448 * 2^e >= a, clamped to
    [-127, 127], and 0 for a = 0 -- settled by exact comparisons in float64."""
    import multiprocessing as mp
    import os

    from tests.exhaustive_util import mx_exponent_chunk_mismatches
    ch = 1 << 22
    end = 0x7F800000  # +inf
    jobs = [(s, min(s + ch, end)) for s in range(0, end, ch)]
    with mp.get_context("spawn").Pool(min(8, os.cpu_count() or 1)) as pool:
        bad = [b for r in pool.map(mx_exponent_chunk_mismatches, jobs, chunksize=16) for b in r]
    assert not bad, [hex(b) for b in bad[:8]]


def test_exp_within_2ulp_of_fp64(orc):
    g = np.random.default_rng(9)
    xs = np.concatenate([np.linspace(-87.0, 88.0, 20001), g.uniform(-87, 88, 20000),
                         g.uniform(-1, 1, 5000)]).astype(np.float32)
    ys = orc.exp_f32(xs)
    worst = 0.0
    for x, y in zip(xs, ys):
        ref = math.exp(float(x))
        worst = max(worst, abs(float(y) - ref) / f32_ulp(ref))
    assert worst <= 2.0, worst


def test_e4m3_encode_exhaustive_vs_torch(orc):
    """Every non-NaN fp32: the oracle's e4m3 code equals torch's float8_e4m3fn
    cast wherever that cast is finite.  Where torch overflows to NaN (|x| past
    the rounding midpoint between 448 and the NaN encoding, and infinities),
    the oracle saturates to +-448 (0x7E / 0xFE), as satfinite prescribes."""
    import multiprocessing as mp
    import os

    from tests.exhaustive_util import e4m3_chunk_mismatches
    ch = 1 << 24
    jobs = [(s, s + ch) for s in range(0, 1 << 32, ch)]
    with mp.get_context("spawn").Pool(min(8, os.cpu_count() or 1)) as pool:
        bad = [b for r in pool.map(e4m3_chunk_mismatches, jobs, chunksize=4) for b in r]
    assert not bad, [hex(b) for b in bad[:8]]


def test_exp_faithful_exhaustive(orc):
    """Every fp32 x in [-87, 88] (about 2.2e9 values, exp(x) a normal fp32):
    the oracle's exp is within one ulp of fp64 exp, i.e. faithfully rounded."""
    import multiprocessing as mp
    import os

    from tests.exhaustive_util import exp_chunk_worst_ulp
    spans = [(0, int(np.float32(88.0).view(np.uint32)) + 1),
             (0x80000000, int(np.float32(-87.0).view(np.uint32)) + 1)]
    ch = 1 << 22
    jobs = [(s, min(s + ch, hi)) for lo, hi in spans for s in range(lo, hi, ch)]
    with mp.get_context("spawn").Pool(min(8, os.cpu_count() or 1)) as pool:
        res = pool.map(exp_chunk_worst_ulp, jobs, chunksize=8)
    worst, at = max(res)
    assert worst < 1.0, (worst, at)


def test_silu_accuracy_exhaustive(orc):
    """Every fp32 g in [-87.3, 89], where sigma = 1/(1 + exp(-g)) is a normal
    fp32: the oracle's silu(g) is within 3 ulp of fp64 g / (1 + exp(-g))
    (within half of 2^-149 where the result is subnormal).  Below, exp(-g)
    overflows from g < -88.72 on and the sequence gives -0 (|true value| <
    2.7e-37)."""
    import multiprocessing as mp
    import os

    from tests.exhaustive_util import silu_chunk_worst
    spans = [(0, int(np.float32(89.0).view(np.uint32)) + 1),
             (0x80000000, int(np.float32(-87.3).view(np.uint32)) + 1)]
    ch = 1 << 22
    jobs = [(s, min(s + ch, hi)) for lo, hi in spans for s in range(lo, hi, ch)]
    with mp.get_context("spawn").Pool(min(8, os.cpu_count() or 1)) as pool:
        res = pool.map(silu_chunk_worst, jobs, chunksize=8)
    worst_n = max(r[0] for r in res)
    worst_s = max(r[1] for r in res)
    assert worst_n[0] <= 3.0, worst_n
    assert worst_s[0] <= 0.5, worst_s
    low = np.array([-88.73, -89.0, -95.5, -103.9, -104.0, -1e4], dtype=np.float32)
    h = orc.silu_mul_f32_array(low, np.ones_like(low))
    assert np.all(h == 0.0) and np.all(np.signbit(h))


def test_exp_special_values(orc):
    assert orc.exp_f32([0.0])[0] == 1.0
    assert np.isinf(orc.exp_f32([89.0])[0]) and np.isinf(orc.exp_f32([1000.0])[0])
    assert orc.exp_f32([-104.0])[0] == 0.0 and orc.exp_f32([-1e9])[0] == 0.0
    assert orc.exp_f32([88.0])[0] == np.float32(math.exp(88.0)) or \
        abs(float(orc.exp_f32([88.0])[0]) - math.exp(88.0)) <= 2 * f32_ulp(math.exp(88.0))
    sub = float(orc.exp_f32([-100.0])[0])                  # subnormal range: absolute bound
    assert abs(sub - math.exp(-100.0)) <= 2.0 ** -149


def test_silu_mul_vs_fp64(orc):
    g = np.random.default_rng(13)
    gs = np.concatenate([g.standard_normal(4000) * 4, [0.0, -0.0, 50.0, -50.0, 120.0, -120.0]]).astype(np.float32)
    us = g.standard_normal(gs.size).astype(np.float32)
    hs = orc.silu_mul_f32(gs, us)
    for a, b, h in zip(gs, us, hs):
        ref = float(a) / (1.0 + math.exp(-float(a))) * float(b) if float(a) > -700 else 0.0
        assert abs(float(h) - ref) <= 6 * f32_ulp(ref) + 2.0 ** -140, (a, b, h, ref)


def test_array_forms_match_scalar_forms(orc):
    g = np.random.default_rng(17)
    x = (g.standard_normal(5000) * 30).astype(np.float32)
    u = g.standard_normal(5000).astype(np.float32)
    assert np.array_equal(orc.e4m3_from_f32_array(x), orc.e4m3_from_f32(x))
    assert np.array_equal(orc.exp_f32_array(x / 4), orc.exp_f32(x / 4))
    assert np.array_equal(orc.silu_mul_f32_array(x / 8, u), orc.silu_mul_f32(x / 8, u))
