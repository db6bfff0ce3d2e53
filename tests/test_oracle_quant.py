"""Pins of the oracle's quantisers: hand-worked groups, brute force on tiny
inputs with an independent encoder and explicit loops, and invariants that
the scale rule S = amax/448 implies."""
import numpy as np
import pytest

from oracle import jetfp8_oracle as O
from tests.test_oracle_e4m3 import _brute_force_encode


def _parse_pairs(s):
    out = {}
    for item in s.split(","):
        i, v = item.split(":")
        out[int(i)] = v
    return out


def test_group_quant_hand_cases(golden):
    for case, fill, entries, s_exp, codes, fill_code in golden("group_quant_hand_cases.txt"):
        x = np.full(128, float(fill), dtype=np.float32)
        for i, v in _parse_pairs(entries).items():
            x[i] = np.float32(float(v))
        q, s = O.quant_rowgroups(x[None, :])
        assert s.shape == (1, 1) and s[0, 0] == np.float32(float(s_exp)), case
        want = np.full(128, int(fill_code.split(":")[1], 16), dtype=np.uint8)
        for i, c in _parse_pairs(codes).items():
            want[i] = int(c, 16)
        assert np.array_equal(q[0], want), (case, q[0][:4], want[:4])


def _brute_rowgroups(x):
    """Explicit loops: per row and group, amax, S = fp32(amax/448), codes."""
    R, C = x.shape
    q = np.zeros((R, C), np.uint8)
    s = np.zeros((C // 128, R), np.float32)
    for r in range(R):
        for g in range(C // 128):
            grp = [float(v) for v in x[r, 128 * g:128 * (g + 1)]]
            amax = 0.0
            for v in grp:
                amax = max(amax, abs(v))
            sc = np.float32(np.float32(amax) / np.float32(448.0)) if amax > 0 else np.float32(1.0)
            s[g, r] = sc
            for j, v in enumerate(grp):
                q[r, 128 * g + j] = _brute_force_encode(float(np.float32(np.float32(v) / sc)))
    return q, s


@pytest.fixture
def tiny_x():
    g = np.random.default_rng(3)
    x = g.standard_normal((5, 256)).astype(np.float32)
    x[1, 7] *= 20
    x[2, 128:] = 0.0
    x[3, :3] = [448.0, -448.0, 17.0]
    return x


def test_rowgroups_brute_force(tiny_x):
    q, s = O.quant_rowgroups(tiny_x)
    qb, sb = _brute_rowgroups(tiny_x)
    assert np.array_equal(s, sb)
    assert np.array_equal(q, qb)


def test_rowgroup_invariants():
    g = np.random.default_rng(4)
    x = (g.standard_normal((64, 1024)) * np.exp(g.uniform(-8, 8, (64, 1)))).astype(np.float32)
    q, s = O.quant_rowgroups(x)
    d = O.e4m3_decode(q).reshape(64, 8, 128)
    sc = s.T[:, :, None].astype(np.float64)
    xg = x.reshape(64, 8, 128).astype(np.float64)
    assert np.all(np.abs(d) <= 448.0)                              # |x̂·S| <= 448·S
    # dequantisation error within half an E4M3 spacing of x/S (plus the FP32 quotient rounding)
    v = np.abs(xg / sc)
    e = np.maximum(np.floor(np.log2(np.maximum(v, 2.0 ** -20))), -6)
    half_ulp = 0.5 * 2.0 ** (e - 3)
    assert np.all(np.abs(d - xg / sc) <= half_ulp * (1 + 1e-6) + 448 * 2.0 ** -23)
    # the amax element of each group maps to ±448
    assert np.all((np.abs(d) == 448.0).any(axis=2))


def test_weight_blocks_brute_force():
    g = np.random.default_rng(5)
    w = (g.standard_normal((256, 384)) * 0.02).astype(np.float32)
    w[130, 300] = 1.0
    q, s, qT = O.quant_weight_128x128(w)
    assert s.shape == (2, 3)
    for nb in range(2):
        for kb in range(3):
            blk = w[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)]
            amax = max(abs(float(v)) for v in blk.reshape(-1))
            assert s[nb, kb] == np.float32(np.float32(amax) / np.float32(448))
            for (i, j) in [(0, 0), (5, 77), (127, 127), (2, 1)]:
                want = _brute_force_encode(float(np.float32(blk[i, j] / s[nb, kb])))
                assert q[128 * nb + i, 128 * kb + j] == want
    assert np.array_equal(qT, q.T)                      # reuse by transpose only


def test_requant_power_of_two_scales_exact():
    """With power-of-two row scales the dequantised value is exact, so the
    requantised codes follow from a hand-checkable column quantisation."""
    g = np.random.default_rng(6)
    codes = g.integers(0, 0x7E, size=(128, 128)).astype(np.uint8)
    codes[g.random((128, 128)) < 0.5] |= 0x80
    s = np.ldexp(1.0, g.integers(-10, 4, size=(1, 128))).astype(np.float32)
    qT, sT = O.requant_rowgrp_to_colgrp(codes, s)
    x = O.e4m3_decode(codes) * s[0][:, None]            # exact
    for k in [0, 3, 64, 127]:
        col = x[:, k]
        amax = np.abs(col).max()
        sc = np.float32(np.float32(amax) / np.float32(448))
        assert sT[0, k] == sc
        for m in [0, 1, 50, 127]:
            assert qT[k, m] == _brute_force_encode(float(np.float32(np.float32(col[m]) / sc)))


def test_requant_idempotent_when_columns_already_saturated():
    """Columns whose amax is 448 under unit row scales keep their codes."""
    g = np.random.default_rng(7)
    codes = g.integers(0, 0x7E, size=(128, 256)).astype(np.uint8)
    codes[0, :] = 0x7E
    s = np.ones((2, 128), np.float32)
    qT, sT = O.requant_rowgrp_to_colgrp(codes, s)
    assert np.all(sT == 1.0)
    assert np.array_equal(qT, codes.T)


def test_requant_brute_force_general():
    g = np.random.default_rng(8)
    x = g.standard_normal((256, 256)).astype(np.float32)
    q, s = O.quant_rowgroups(x)
    qT, sT = O.requant_rowgrp_to_colgrp(q, s)
    # explicit loops from the definition
    deq = np.zeros((256, 256), np.float32)
    for m in range(256):
        for k in range(256):
            deq[m, k] = np.float32(np.float32(O._decode_one(int(q[m, k]))) * s[k // 128, m])
    qb, sb = _brute_rowgroups(np.ascontiguousarray(deq.T))
    assert np.array_equal(sT, sb) and np.array_equal(qT, qb)


def test_grad_dual_brute_force():
    g = np.random.default_rng(9)
    dy = (g.standard_normal((128, 256)) * 1e-3).astype(np.float32)
    q_row, s_row, qT_col, sT_col = O.quant_grad_dual(dy)
    qb, sb = _brute_rowgroups(dy)
    assert np.array_equal(q_row, qb) and np.array_equal(s_row, sb)
    # 128×1 column groups: loops down each column of 128 tokens
    for n in [0, 17, 255]:
        col = dy[:, n]
        amax = max(abs(float(v)) for v in col)
        sc = np.float32(np.float32(amax) / np.float32(448))
        assert sT_col[0, n] == sc
        for m in [0, 64, 127]:
            assert qT_col[n, m] == _brute_force_encode(float(np.float32(col[m] / sc)))
    assert qT_col.shape == (256, 128) and sT_col.shape == (1, 256)
