"""Pins of the oracle GEMMs: exact int64 dot products with unit scales,
explicit-loop block-scaled sums with random scales, and the identities that
tie DGrad and WGrad to the forward definition."""
import numpy as np
import pytest

from oracle import jetfp8_oracle as O


def _codes(g, shape):
    c = g.integers(0, 0x7F, size=shape).astype(np.uint8)    # finite magnitudes
    c[g.random(shape) < 0.5] |= 0x80
    return c


def _int_dec(code):
    """dec(code)·2^9 as an exact integer (every E4M3 value is a multiple of 2^-9)."""
    v = O._decode_one(int(code)) * 512
    assert v == int(v)
    return int(v)


def test_unit_scales_exact_int64():
    g = np.random.default_rng(10)
    A = _codes(g, (3, 256)); B = _codes(g, (4, 256))
    out = O.block_scaled_gemm(A, np.ones((2, 3), np.float32), B, lambda kb: np.ones(4, np.float32))
    for i in range(3):
        for j in range(4):
            acc = 0
            for k in range(256):
                acc += _int_dec(A[i, k]) * _int_dec(B[j, k])
            assert out[i, j] == acc * 2.0 ** -18           # exact


def test_fprop_explicit_loops():
    g = np.random.default_rng(11)
    M, K, N = 3, 256, 256
    xq = _codes(g, (M, K)); wq = _codes(g, (N, K))
    sx = g.uniform(0.01, 2, (K // 128, M)).astype(np.float32)
    sw = g.uniform(0.01, 2, (N // 128, K // 128)).astype(np.float32)
    y = O.gemm_fprop(xq, sx, wq, sw)
    for m in range(M):
        for n in [0, 1, 130, 255]:
            tot = 0.0
            for kb in range(K // 128):
                p = sum(O._decode_one(int(xq[m, k])) * O._decode_one(int(wq[n, k]))
                        for k in range(128 * kb, 128 * kb + 128))
                tot += float(sx[kb, m]) * float(sw[n // 128, kb]) * p
            assert y[m, n] == pytest.approx(tot, rel=1e-13, abs=1e-13)
    # row/column subsets give the same values
    sub = O.gemm_fprop(xq, sx, wq, sw, rows=[2, 0], cols=[255, 3])
    assert np.array_equal(sub, y[[2, 0]][:, [255, 3]])


def test_dgrad_through_transposed_weight_equals_definition():
    """∇X[m,k] = Σ_n S∇Y[m,n/128]·Sw[n/128,k/128]·dec(∇Ŷ[m,n])·dec(Ŵ[n,k])."""
    g = np.random.default_rng(12)
    M, N, K = 2, 256, 384
    dyq = _codes(g, (M, N)); wq = _codes(g, (N, K))
    sdy = g.uniform(0.01, 2, (N // 128, M)).astype(np.float32)
    sw = g.uniform(0.01, 2, (N // 128, K // 128)).astype(np.float32)
    dx = O.gemm_dgrad(dyq, sdy, np.ascontiguousarray(wq.T), sw)
    assert dx.shape == (M, K)
    for m in range(M):
        for k in [0, 129, 383]:
            tot = 0.0
            for n in range(N):
                tot += (float(sdy[n // 128, m]) * float(sw[n // 128, k // 128])
                        * O._decode_one(int(dyq[m, n])) * O._decode_one(int(wq[n, k])))
            assert dx[m, k] == pytest.approx(tot, rel=1e-12)


def test_wgrad_equals_definition_over_tokens():
    """∇W[n,k] = Σ_m S∇Yᵀ[m/128,n]·SXᵀ[m/128,k]·dec(∇Ŷᵀ[n,m])·dec(X̂ᵀ[k,m])."""
    g = np.random.default_rng(13)
    M, N, K = 256, 3, 4
    dyqT = _codes(g, (N, M)); xqT = _codes(g, (K, M))
    sdyT = g.uniform(0.01, 2, (M // 128, N)).astype(np.float32)
    sxT = g.uniform(0.01, 2, (M // 128, K)).astype(np.float32)
    dw = O.gemm_wgrad(dyqT, sdyT, xqT, sxT)
    for n in range(N):
        for k in range(K):
            tot = 0.0
            for m in range(M):
                tot += (float(sdyT[m // 128, n]) * float(sxT[m // 128, k])
                        * O._decode_one(int(dyqT[n, m])) * O._decode_one(int(xqT[k, m])))
            assert dw[n, k] == pytest.approx(tot, rel=1e-12)


def test_fprop_of_quantised_inputs_tracks_float_matmul():
    """End to end: FP8 FProp of quantised N(0,1)/N(0,0.02) data stays close to
    the unquantised product (relative Frobenius error of a few percent)."""
    g = np.random.default_rng(14)
    x = g.standard_normal((64, 512)).astype(np.float32)
    w = (g.standard_normal((256, 512)) * 0.02).astype(np.float32)
    xq, sx = O.quant_act_1x128(x)
    wq, sw, _ = O.quant_weight_128x128(w)
    y = O.gemm_fprop(xq, sx, wq, sw)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) < 0.06
