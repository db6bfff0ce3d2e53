"""Exact host check of the quantisers' division-free element quotient.

The quantisation rule (Jet-RL digest "Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8
强化学习", 前置知识 › FP8 量化 (E4M3 格式)) codes x as E4M3(RN32(x / S)).  The kernels
form RN32(x/S) without a division: per group y = RN32(1/S) (an IEEE reciprocal),
per element two Markstein corrections (P. Markstein, "Computation of elementary
functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990)
of q0 = RN32(x·y), run on −x and −y so that the sign of a zero survives:

    q1 = RN32(q0 + (−x − q0·S)·(−y))      (the residual by one FMA, then one FMA)
    q2 = RN32(q1 + (−x − q1·S)·(−y))

Groups whose maximum is below 2^-80 run the same sequence on x·2^96 and S·2^96
(exact scalings that leave every quotient unchanged).  The tests evaluate each
FMA exactly (the product in FP64 is exact, the sum by TwoSum, then one rounding
to FP32 with the midpoint decided by the sign of the error term) and compare q2
with the correctly rounded quotient, for every bf16 element of groups whose
maxima step through the bf16 range, and for FP32 elements next to E4M3 rounding
boundaries across the scale range.  Quotients below 2^-11 (which round to a
zero code) are only required to stay below 2^-10 with the sign of x.
"""
from fractions import Fraction

import numpy as np

from tests.test_scale_division_free import _rn32_exact, _rn32_of_sum


def _rn32_div_exact(num: np.ndarray, den: np.ndarray) -> np.ndarray:
    """RN32(num/den) for FP32 arrays: the FP64 quotient rounds right unless it
    lands on an FP32 midpoint, which exact rationals then settle."""
    d = num.astype(np.float64) / den.astype(np.float64)
    out = d.astype(np.float32)
    lo = np.where(out.astype(np.float64) > d, np.nextafter(out, np.float32(-np.inf)), out)
    hi = np.nextafter(lo, np.float32(np.inf))
    mid = (lo.astype(np.float64) + hi.astype(np.float64)) / 2
    for i in np.nonzero((d == mid) & (d != 0))[0]:
        q = Fraction(float(num[i])) / Fraction(float(den[i]))
        v = _rn32_exact(abs(q))
        out[i] = -v if q < 0 else v
    return out


def _fma32(a, b, c):
    """RN32(a·b + c) evaluated exactly (a, b, c FP32; a·b is exact in FP64)."""
    p = a.astype(np.float64) * b.astype(np.float64)
    c64 = c.astype(np.float64)
    s = p + c64
    bb = s - p
    err = (p - (s - bb)) + (c64 - bb)
    out = _rn32_of_sum(s, err)
    # an exact zero sum is +0 unless both addends are −0
    zero = (s == 0) & (err == 0)
    neg = np.signbit(p) & (p == 0) & np.signbit(c) & (c == 0)
    return np.where(zero, np.where(neg, np.float32(-0.0), np.float32(0.0)), out).astype(np.float32)


def division_free_quotient(x, S):
    """The kernels' sequence for elements x of a group with scale S (FP32)."""
    y = _rn32_div_exact(np.ones_like(S), S)
    nx, ny = (-x).astype(np.float32), (-y).astype(np.float32)
    q0 = (nx.astype(np.float64) * ny.astype(np.float64)).astype(np.float32)
    q1 = _fma32(_fma32(q0, S, nx), ny, q0)
    return _fma32(_fma32(q1, S, nx), ny, q1)


def _check(x, S):
    got = division_free_quotient(x, S)
    want = _rn32_div_exact(x, S)
    big = np.abs(want.astype(np.float64)) >= 2.0 ** -11
    bad = big & (got.view(np.uint32) != want.view(np.uint32))
    small_bad = (~big) & ((np.abs(got) >= 2.0 ** -10) | (np.signbit(got) != np.signbit(x)))
    assert not bad.any(), f"x={x[bad][0]!r} S={S[bad][0]!r}: {got[bad][0]!r} vs {want[bad][0]!r}"
    assert not small_bad.any(), f"x={x[small_bad][0]!r}: {got[small_bad][0]!r}"
    return x.size


def _bf16_magnitudes():
    return (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)   # +0 .. max finite


def test_every_bf16_element_under_stepped_group_maxima():
    """Groups with maxima every 32nd bf16 value from 2^-80 up (and the largest):
    every bf16 element of magnitude up to the maximum, both signs, S = RN32(amax/448)."""
    mags = _bf16_magnitudes()
    maxima = mags[mags >= np.float32(2.0 ** -80)]
    maxima = np.concatenate([maxima[::32], maxima[-1:]])
    n = 0
    for amax in maxima:
        m = mags[mags <= amax]
        x = np.concatenate([m, -m]).astype(np.float32)
        S = np.full(x.shape, np.float32(amax) / np.float32(448.0), np.float32)
        n += _check(x, S)
    assert n > 3_000_000


def test_tiny_groups_on_scaled_operands():
    """Maxima below 2^-80: the sequence on x·2^96 and S·2^96 gives RN32(x/S)."""
    mags = _bf16_magnitudes()
    maxima = mags[(mags > 0) & (mags < np.float32(2.0 ** -80))][::7]
    two96 = np.float32(2.0 ** 96)
    for amax in maxima:
        m = mags[mags <= amax]
        x = np.concatenate([m, -m]).astype(np.float32)
        S = np.full(x.shape, np.float32(amax) / np.float32(448.0), np.float32)
        xs, Ss = (x * two96).astype(np.float32), (S * two96).astype(np.float32)
        assert np.array_equal(xs.astype(np.float64), x.astype(np.float64) * 2.0 ** 96)   # exact scaling
        got = division_free_quotient(xs, Ss)
        want = _rn32_div_exact(x, S)
        big = np.abs(want.astype(np.float64)) >= 2.0 ** -11
        assert np.array_equal(got[big].view(np.uint32), want[big].view(np.uint32)), amax


def test_fp32_elements_next_to_e4m3_boundaries():
    """FP32 elements (as the requantiser's dequantised values are) whose
    quotients sit on or one ulp beside E4M3 midpoints, across scales 2^-88..2^118."""
    rng = np.random.default_rng(5)
    ulp9 = 2.0 ** -9
    mids = np.array([ulp9 * (k + 0.5) for k in range(1, 8)] + [12.5, 13.5, 17.0, 19.0, 104.0, 240.0, 416.0, 448.0])
    for e in range(-88, 119, 5):
        s = np.ldexp(rng.uniform(1, 2, 64), e).astype(np.float32)
        S = np.repeat(s, 1024)
        x = (rng.uniform(-1, 1, S.size) * 448.0 * S.astype(np.float64)).astype(np.float32)
        q = S.size // 4
        xm = (mids[rng.integers(0, len(mids), q)] * S[:q].astype(np.float64)).astype(np.float32)
        toward = np.where(rng.random(q) < 0.5, np.float32(np.inf), np.float32(-np.inf))
        x[:q] = np.nextafter(xm, toward)
        x[q:2 * q] = xm
        x[2 * q:3 * q] = -xm
        _check(x, S)


def test_hand_cases():
    """Quotients with known answers: exact multiples of S and exact E4M3 values."""
    S = np.full(6, np.float32(3.0) / np.float32(448.0), np.float32)
    x = (S.astype(np.float64) * np.array([448.0, -448.0, 1.0, 0.0, -0.0, 2.0 ** -9])).astype(np.float32)
    got = division_free_quotient(x, S)
    assert np.array_equal(got.view(np.uint32), _rn32_div_exact(x, S).view(np.uint32))
    assert np.signbit(got[4]) and not np.signbit(got[3]) and got[3] == 0


def test_fp4_block_scales():
    """The FP4 variant's quantiser runs the same sequence with d = RN(s_b·g)
    (an E4M3 block scale times an FP32 row scale) for d >= 2^-90: bf16 elements
    of every magnitude up to 8·d, both signs, under block scales of every E4M3
    exponent and random row scales."""
    rng = np.random.default_rng(11)
    mags = _bf16_magnitudes()
    e4m3 = np.array([(1 + m / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)], np.float64)
    n = 0
    for sb in e4m3[::3]:
        for g in np.ldexp(rng.uniform(1, 2, 3), rng.integers(-60, 20, 3)).astype(np.float32):
            d = np.float32(np.float32(sb) * g)
            if d < np.float32(2.0 ** -90):
                continue
            m = mags[mags <= np.float32(8) * d]
            x = np.concatenate([m, -m]).astype(np.float32)
            n += _check(x, np.full(x.shape, d, np.float32))
    assert n > 1_000_000
