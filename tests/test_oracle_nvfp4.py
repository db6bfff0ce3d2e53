"""Pins of the FP4 (NVFP4-style) oracle against things other than itself: the
E2M1 format's closed form, hand-worked encodings and a hand-quantised row
(tests/golden/), brute force on small inputs, invariants of the quantiser,
and exact integer GEMMs."""
import os

import numpy as np
import pytest

from oracle import jetfp8_oracle as O8
from oracle import nvfp4_oracle as O4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_decode_every_code():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    v = O4.e2m1_decode(np.arange(16))
    assert list(v[:8]) == mags and list(v[8:]) == [-m for m in mags]
    assert np.signbit(v[8]) and not np.signbit(v[0])
    # closed form: e = 0 subnormal m·2^-1, else (1 + m/2)·2^(e-1); the largest is 6
    assert O4.E2M1_MAX == v.max() == 6.0 and np.all(np.diff(v[:8]) > 0)


def test_e2m1_encode_hand_cases():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_hand_cases.txt")) if l.strip() and l[0] != "#"]
    v = np.array([float(r[0]) for r in rows])
    want = np.array([int(r[1]) for r in rows])
    assert np.array_equal(O4.e2m1_encode(v), want)


def test_e2m1_encode_round_trip_and_brute_force():
    codes = np.arange(16)
    assert np.array_equal(O4.e2m1_encode(O4.e2m1_decode(codes)), codes)
    rng = np.random.default_rng(3)
    mags = O4.e2m1_decode(np.arange(8))
    mids = (mags[1:] + mags[:-1]) / 2
    v = np.concatenate([rng.uniform(-8, 8, 20000), mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 9)])
    got = O4.e2m1_encode(v)
    for x, c in zip(v, got):
        a = min(abs(x), 6.0)
        d = np.abs(mags - a)
        best = np.flatnonzero(d == d.min())
        k = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert c == (k | (8 if np.signbit(x) else 0)), (x, c)


def _golden_row():
    kv = {}
    for l in open(os.path.join(GOLDEN, "nvfp4_hand_cases.txt")):
        if l.strip() and l[0] != "#":
            k, *vals = l.split()
            kv[k] = vals
    return kv


def test_quantiser_hand_worked_row():
    kv = _golden_row()
    x = np.array([float(t) for t in kv["x"]], np.float32)[None, :]
    q, s, g = O4.quant_nvfp4_rows(x)
    assert np.array_equal(q[0], [int(t) for t in kv["codes"]])
    assert list(s[0]) == [int(t, 16) for t in kv["block_scales"]]
    assert g[0] == np.float32(float(kv["row_scale"][0]))


def _explicit_loops(x):
    """The rule written out element by element with numpy float32 scalars."""
    R, K = x.shape
    f = np.float32
    codes = np.zeros((R, K), np.int64)
    scales = np.zeros((R, K // 16), np.int64)
    gs = np.zeros(R, np.float32)
    for r in range(R):
        amax = f(0)
        for k in range(K):
            amax = max(amax, abs(f(x[r, k])))
        g = f(amax / f(2688)) if amax > 0 else f(1)
        h = f(f(6) * g)
        gs[r] = g
        for b in range(K // 16):
            blk = [f(x[r, 16 * b + i]) for i in range(16)]
            ab = max(abs(v) for v in blk)
            s = int(O8.e4m3_encode(np.array([f(ab / h)]))[0])
            scales[r, b] = s
            d = f(f(O8.e4m3_decode(np.array([s]))[0]) * g)
            for i, v in enumerate(blk):
                if d == 0:
                    codes[r, 16 * b + i] = 8 if np.signbit(v) else 0
                else:
                    codes[r, 16 * b + i] = int(O4.e2m1_encode(np.array([f(v / d)]))[0])
    return codes, scales, gs


def test_quantiser_equals_explicit_loops():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((6, 64)) * np.exp(rng.uniform(-20, 20, (6, 1)))).astype(np.float32)
    x[2, 16:32] = 0.0                  # an all-zero block
    x[3] = 0.0                         # an all-zero row (g = 1)
    x[4, 5] = -0.0
    x[5] *= np.float32(1e-30)          # tiny values: block scales underflow E4M3
    q, s, g = O4.quant_nvfp4_rows(x)
    eq, es, eg = _explicit_loops(x)
    assert np.array_equal(q, eq) and np.array_equal(s, es) and np.array_equal(g, eg)
    assert g[3] == 1.0 and np.all(q[3] == 0) and q[4, 5] == 8


def test_quantiser_invariants_and_batch_independence():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((40, 256)) * 3).astype(np.float32)
    q, s, g = O4.quant_nvfp4_rows(x)
    d = O8.e4m3_decode(s).astype(np.float32) * g[:, None]
    # each element within half an E2M1 spacing (at most 1 in units of d, 2 above 4) of its block's grid
    err = np.abs(O4.dequant_nvfp4_rows(q, s, g).reshape(40, 16, 16) - x.reshape(40, 16, 16))
    assert np.all(err <= np.repeat(d, 1).reshape(40, 16, 1) * 1.0 + 1e-12)
    # a block's maximum lands within 2^-4 of 6·d (the E4M3 block scale rounds by at
    # most that much), so it takes the largest code, 6
    mag = (q.reshape(40, 16, 16) & 7).max(axis=2)
    assert np.all(mag == 7)
    # a row's codes do not depend on the other rows quantised with it
    q1, s1, g1 = O4.quant_nvfp4_rows(x[7:8])
    assert np.array_equal(q1[0], q[7]) and np.array_equal(s1[0], s[7]) and g1[0] == g[7]


def test_gemm_unit_scales_exact_and_explicit_loops():
    rng = np.random.default_rng(7)
    M, N, K = 3, 4, 48
    xq = rng.integers(0, 16, (M, K)).astype(np.int8)
    wq = rng.integers(0, 16, (N, K)).astype(np.int8)
    one = np.full((M, K // 16), 0x38, np.uint8)         # E4M3 1.0
    onew = np.full((N, K // 16), 0x38, np.uint8)
    y = O4.gemm_fprop_nvfp4(xq, one, np.ones(M, np.float32), wq, onew, np.ones(N, np.float32))
    # exact: in units of 1/4, integer dot products
    xi = np.rint(O4.e2m1_decode(xq) * 2).astype(np.int64)
    wi = np.rint(O4.e2m1_decode(wq) * 2).astype(np.int64)
    assert np.array_equal(y * 4, (xi @ wi.T).astype(np.float64))
    # with scales: explicit triple loop
    sx = rng.integers(0x20, 0x60, (M, K // 16)).astype(np.uint8)
    sw = rng.integers(0x20, 0x60, (N, K // 16)).astype(np.uint8)
    gx = rng.uniform(0.5, 2, M).astype(np.float32)
    gw = rng.uniform(0.5, 2, N).astype(np.float32)
    y = O4.gemm_fprop_nvfp4(xq, sx, gx, wq, sw, gw)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += (float(O4.e2m1_decode(xq[m, k])) * float(O8.e4m3_decode(sx[m, k // 16])) *
                        float(O4.e2m1_decode(wq[n, k])) * float(O8.e4m3_decode(sw[n, k // 16])))
            assert y[m, n] == pytest.approx(acc * float(gx[m]) * float(gw[n]), rel=1e-14)
