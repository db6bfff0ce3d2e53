"""Pins of the oracle's E4M3 decode/encode and bf16 rounding against things
other than itself: the format's defining constants, hand-worked encodings,
torch's independent float8_e4m3fn / bfloat16 casts, and a brute-force
nearest-code search."""
import math

import numpy as np
import pytest
import torch

from oracle import jetfp8_oracle as O


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_format_constants():
    d = O.e4m3_decode(np.arange(256))
    assert d[0x7E] == 448.0 == O.E4M3_MAX          # Δmax of the E4M3 section
    assert d[0x08] == 2.0 ** -6                     # smallest normal
    assert d[0x01] == 2.0 ** -9                     # smallest subnormal
    assert d[0x38] == 1.0
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.isfinite(d).sum() == 254
    pos = d[:0x7F]
    assert np.all(np.diff(pos) > 0)                 # monotone over 0x00..0x7E
    assert math.copysign(1.0, d[0x80]) == -1.0 and d[0x80] == 0.0
    assert np.array_equal(d[0x80:0xFF], -d[0x00:0x7F])


def test_decode_matches_torch_for_all_codes():
    d = O.e4m3_decode(np.arange(256))
    t = _torch_decode_all()
    both_nan = np.isnan(d) & np.isnan(t)
    assert np.array_equal(np.isnan(d), np.isnan(t))
    assert np.array_equal(d[~both_nan], t[~both_nan])


def test_encode_roundtrip_all_finite_codes():
    d = O.e4m3_decode(np.arange(256))
    finite = np.where(np.isfinite(d))[0]
    enc = O.e4m3_encode(d[finite].astype(np.float32))
    assert np.array_equal(enc, finite.astype(np.uint8))


def test_encode_hand_cases(golden):
    for val, code, *_ in golden("e4m3_hand_cases.txt"):
        got = int(O.e4m3_encode(np.array([float(val)], dtype=np.float32))[0])
        assert got == int(code, 16), (val, hex(got), code)


def _brute_force_encode(v: float) -> int:
    """Independent encoder: nearest finite code by exhaustive search, ties to
    the code with an even mantissa LSB, saturating at ±448, sign kept."""
    table = [O._decode_one(c) for c in range(0x7F)]   # non-negative finite codes
    a = min(abs(v), 448.0)
    best, bestd = None, None
    for c, m in enumerate(table):
        dist = abs(m - a)
        if bestd is None or dist < bestd or (dist == bestd and (c & 1) == 0):
            best, bestd = c, dist
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    return best | sign


def test_encode_matches_brute_force_including_midpoints():
    d = O.e4m3_decode(np.arange(0x7F))
    mids = (d[:-1] + d[1:]) / 2                          # every tie point
    eps = np.array([0.0, 1e-7, -1e-7])
    vals = [m * (1 + e) for m in mids for e in eps] + list(d) + [450.0, 463.9, 464.0, 1e4]
    vals = np.array(vals + [-v for v in vals], dtype=np.float32)
    enc = O.e4m3_encode(vals)
    for v, c in zip(vals, enc):
        assert int(c) == _brute_force_encode(float(v)), (float(v), hex(int(c)))


def test_encode_matches_torch_in_range():
    g = np.random.default_rng(1)
    v = np.concatenate([g.standard_normal(200000) * 40, g.uniform(-448, 448, 100000),
                        g.standard_normal(50000) * 1e-2]).astype(np.float32)
    ours = O.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_rne_matches_torch_from_float32():
    g = np.random.default_rng(2)
    v = np.concatenate([g.standard_normal(100000), g.standard_normal(1000) * 1e4]).astype(np.float32)
    ours = O.bf16_rne(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    # ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even -> 1
    assert O.bf16_rne(np.array([1 + 2 ** -8]))[0] == 1.0
    assert O.bf16_rne(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
