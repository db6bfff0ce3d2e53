"""Exhaustive host check of the quantisers' division-free scale.

The quantisation rule (Jet-RL digest "Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8
强化学习", 前置知识 › FP8 量化 (E4M3 格式)) takes S = max|x| / 448 as the correctly
rounded FP32 quotient.  The kernels form it without a division:

    c  = RN32(1/448)
    q0 = RN32(a·c)
    r  = a − 448·q0          (one FMA; exact)
    S  = RN32(q0 + r·c)      (one FMA)

This is Markstein's correction of a quotient (P. Markstein, "Computation of
elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
Dev. 34(1), 1990; also in Muller et al., Handbook of Floating-Point
Arithmetic, on division by Newton-Raphson iteration): with y within half an ulp of 1/b and
q within one ulp of a/b, RN(q + (a − bq)·y) = RN(a/b).  The tests below do
not rely on the theorem: they evaluate the sequence in exact arithmetic
(FP64 where it is exact, an exact sum otherwise) and compare it with the
correctly rounded quotient, for every positive finite bf16 value (every
exponent, the extremes included) and for all 2^23 FP32 significands of one
binade (the sequence commutes with scaling by powers of two while every
intermediate is normal, i.e. for a ≥ 2^-100, the kernels' threshold for the
division fallback).
"""
from fractions import Fraction

import numpy as np

C32 = np.float32(1.0) / np.float32(448.0)          # RN32(1/448)


def _rn32_exact(x: Fraction) -> np.float32:
    """Round a positive rational to the nearest FP32 (ties to even), normal range."""
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    ulp = Fraction(2) ** (e - 23)
    m, rem = divmod(x, ulp)
    m = int(m)
    if rem > ulp / 2 or (rem == ulp / 2 and m % 2 == 1):
        m += 1
    return np.float32(float(m * ulp))


def _rn32_of_sum(hi: np.ndarray, lo: np.ndarray) -> np.ndarray:
    """RN32 of the exact value hi + lo (hi = fl64(hi + lo), |lo| tiny): FP64 →
    FP32 rounding is right unless hi sits exactly on an FP32 midpoint, where
    the sign of lo decides (lo == 0: a true tie, to even)."""
    r = hi.astype(np.float32)
    exact = r.astype(np.float64) == hi
    lo32 = np.where(r.astype(np.float64) > hi, np.nextafter(r, np.float32(-np.inf)), r)
    hi32 = np.nextafter(lo32, np.float32(np.inf))
    mid = (lo32.astype(np.float64) + hi32.astype(np.float64)) / 2
    on_mid = (~exact) & (hi == mid)
    up = on_mid & (lo > 0)
    down = on_mid & (lo < 0)
    r = np.where(up, hi32, np.where(down, lo32, r))
    return r


def division_free_scale(a: np.ndarray) -> np.ndarray:
    """The kernels' sequence, evaluated exactly (a: positive FP32, ≥ 2^-100)."""
    a64 = a.astype(np.float64)
    q0 = (a64 * np.float64(C32)).astype(np.float32)                # product exact in FP64
    r64 = a64 - 448.0 * q0.astype(np.float64)                      # exact (Sterbenz range)
    r = r64.astype(np.float32)
    assert np.array_equal(r.astype(np.float64), r64), "the FMA residual must be exact"
    rc = r.astype(np.float64) * np.float64(C32)                    # exact (24 × 24 bits)
    s = q0.astype(np.float64) + rc
    bb = s - q0.astype(np.float64)
    err = (q0.astype(np.float64) - (s - bb)) + (rc - bb)           # TwoSum: s + err = q0 + rc
    return _rn32_of_sum(s, err)


def correct_quotient(a: np.ndarray) -> np.ndarray:
    """RN32(a/448), exactly: a/448 is never an FP32 midpoint (that would need
    448·(2Q+1)/2 with a 25-bit odd factor inside a 24-bit significand), so the
    FP64 quotient, within 2^-53 of it, rounds to the same FP32 value unless it
    lands exactly on a midpoint, which is then resolved with exact rationals."""
    d = a.astype(np.float64) / 448.0
    out = d.astype(np.float32)
    lo32 = np.where(out.astype(np.float64) > d, np.nextafter(out, np.float32(-np.inf)), out)
    hi32 = np.nextafter(lo32, np.float32(np.inf))
    mid = (lo32.astype(np.float64) + hi32.astype(np.float64)) / 2
    for i in np.nonzero(d == mid)[0]:
        out[i] = _rn32_exact(Fraction(float(a[i])) / 448)
    return out


def _all_positive_finite_bf16() -> np.ndarray:
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16            # 0x0001 .. 0x7F7F
    return bits.view(np.float32)


def test_every_bf16_amax_from_the_division_threshold_up():
    a = _all_positive_finite_bf16()
    a = a[a >= np.float32(2.0 ** -100)]
    assert a.size > 28000 and a.max() == np.float32(3.3895314e38)
    got = division_free_scale(a)
    want = correct_quotient(a)
    bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
    assert bad.size == 0, f"{bad.size} bf16 maxima differ, first {a[bad[0]]!r}"


def test_every_fp32_significand_of_one_binade():
    a = (np.arange(1 << 23, dtype=np.uint32) | np.uint32(127 << 23)).view(np.float32)   # [1, 2)
    got = division_free_scale(a)
    want = correct_quotient(a)
    bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
    assert bad.size == 0, f"{bad.size} significands differ, first {a[bad[0]]!r}"


def test_extreme_exponents_and_exact_rationals():
    """Random significands at the threshold's binade and at the top of the FP32
    range, against quotients rounded with exact rationals."""
    rng = np.random.default_rng(7)
    for e in (-100, -99, -60, 0, 100, 126, 127):
        sig = rng.integers(0, 1 << 23, size=400, dtype=np.uint32)
        a = (sig | np.uint32((e + 127) << 23)).view(np.float32)
        got = division_free_scale(a)
        for v, gv in zip(a[:60], got[:60]):
            assert gv == _rn32_exact(Fraction(float(v)) / 448), (e, float(v))
        assert np.array_equal(got.view(np.uint32), correct_quotient(a).view(np.uint32))


def test_exact_quotients_and_the_tie_helper():
    """Cases with a known answer: multiples of 448 give exact quotients, and
    the exact rounding helper breaks ties to even."""
    a = np.float32(448.0) * np.array([1, 2, 3, 0.5, 1.25, 2.0 ** 20, 2.0 ** -90], np.float32)
    assert np.array_equal(division_free_scale(a), (a.astype(np.float64) / 448).astype(np.float32))
    one = Fraction(1)
    assert _rn32_exact(one + Fraction(1, 2 ** 24)) == np.float32(1.0)                  # tie, even stays
    assert _rn32_exact(one + Fraction(3, 2 ** 24)) == np.float32(1.0) + np.float32(2.0 ** -22)

