"""GPU parity of the quantisers against the CPU oracle, through the C ABI.
Codes and scales must be bit-identical."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from oracle import jetfp8_oracle as O
from tests.gpu_util import check_errors, h, q_act, q_grad, q_weight, requant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _assert_rowquant(q, s, xf):
    oq, os_ = O.quant_rowgroups(xf)
    M = xf.shape[0]
    assert np.array_equal(h(s)[:, :M], os_), "scales differ"
    gq = h(q)
    if not np.array_equal(gq, oq):
        bad = np.argwhere(gq != oq)
        i, j = bad[0]
        raise AssertionError(f"{len(bad)} codes differ; first at {(i, j)}: x={xf[i, j]!r} "
                             f"gpu={gq[i, j]:#04x} oracle={oq[i, j]:#04x}")


@pytest.mark.parametrize("M,K", [(256, 512), (1, 128), (3, 256), (130, 384), (257, 1024), (1000, 4096)])
def test_quant_act_parity(dev, M, K):
    x = W.activations(M, K, seed=0, stream=M)
    q, s = q_act(x, dev)
    _assert_rowquant(q, s, W.bf16_values(x))


def test_quant_act_edge_values(dev):
    """Zero groups, signed zeros, ties of the E4M3 grid, tiny (subnormal-scale)
    groups, huge groups, and every positive code's midpoint under S = 1."""
    K = 128
    rows = []
    r = np.zeros(K, np.float32); rows.append(r)                       # all zero -> S = 1
    r = np.zeros(K, np.float32); r[::2] = -0.0; r[1] = 0.0; rows.append(r)
    r = np.zeros(K, np.float32); r[0] = 448; r[1:19] = [17, 19, -17, -19, 0.0009765625, 1.5 * 2**-10,
                                                         2**-12, -2**-12, 240, 3.1, 0.3, 2**-6, 7 * 2**-9,
                                                         -448, 1, -1, 2, 0.5]; rows.append(r)
    r = (np.arange(K, dtype=np.float32) - 64) * np.float32(1e-38); rows.append(r)   # subnormal S
    r = (np.arange(K, dtype=np.float32) - 64) * np.float32(1e36); rows.append(r)
    d = O.e4m3_decode(np.arange(0x7F))
    mids = ((d[:-1] + d[1:]) / 2).astype(np.float32)
    for c in range(0, len(mids), K - 1):
        r = np.zeros(K, np.float32); r[0] = 448
        chunk = mids[c:c + K - 1]; r[1:1 + len(chunk)] = chunk; rows.append(r)
    x = W.to_bf16(np.stack(rows))
    q, s = q_act(x, dev)
    _assert_rowquant(q, s, W.bf16_values(x))


def _near_tie_groups(n_groups, rel, seed):
    """Groups of bf16 values whose quotient v/S lies within `rel` (relative) of an
    E4M3 rounding midpoint, S = fp32(amax/448) of the group's own maximum.  For
    each candidate maximum (a bf16 value) every smaller positive bf16 value is
    tried; the near ones go into that maximum's group with random signs."""
    rng = np.random.default_rng(seed)
    allv = (np.arange(0x3000, 0x4800, dtype=np.uint32) << 16).view(np.float32)   # ≈ [4.7e-10, 131072)
    d = O.e4m3_decode(np.arange(0x7F)).astype(np.float64)
    mids = (d[:-1] + d[1:]) / 2
    groups = []
    for amax in rng.permutation(allv[(allv > 1e-3) & (allv < 1e3)]):
        S = np.float32(np.float32(amax) / np.float32(448.0))
        cand = allv[allv < amax]
        qv = cand.astype(np.float64) / np.float64(S)
        k = np.clip(np.searchsorted(mids, qv), 1, len(mids) - 1)
        dist = np.minimum(np.abs(qv - mids[k - 1]), np.abs(qv - mids[k])) / qv
        near = cand[dist < rel]
        if len(near) == 0:
            continue
        row = np.zeros(128, np.float32)
        row[0] = amax
        pick = near[:127] * rng.choice(np.float32([-1.0, 1.0]), size=min(len(near), 127))
        row[1:1 + len(pick)] = pick
        groups.append(row)
        if len(groups) == n_groups:
            break
    return np.stack(groups)


def test_quant_act_near_rounding_boundaries(dev):
    """Quotients v/S within 2^-19 of an E4M3 rounding boundary, over many
    different scales: the bracketing products (from an approximate reciprocal
    of S) must give exactly the codes of RN(v/S) or defer to the division."""
    rows = _near_tie_groups(96, 2.0 ** -19, seed=7)
    assert len(rows) >= 64
    x = W.to_bf16(rows)
    assert np.array_equal(W.bf16_values(x), rows)     # the values are bf16 already
    q, s = q_act(x, dev)
    _assert_rowquant(q, s, rows)


@pytest.mark.parametrize("N,K", [(384, 512), (128, 128), (1024, 2048)])
def test_quant_weight_parity(dev, N, K):
    w = W.weights(N, K, seed=1)
    q, s, qT = q_weight(w, dev)
    oq, os_, oqT = O.quant_weight_128x128(W.bf16_values(w))
    assert np.array_equal(h(s), os_)
    assert np.array_equal(h(q), oq)
    assert np.array_equal(h(qT), oqT)


def test_quant_weight_without_transpose(dev):
    w = W.weights(256, 384, seed=2)
    q, s, _ = q_weight(w, dev, with_t=False)
    oq, os_, _ = O.quant_weight_128x128(W.bf16_values(w))
    assert np.array_equal(h(q), oq) and np.array_equal(h(s), os_)


def test_quant_weight_grouped_equals_single(dev):
    """Four weights of different shapes (one without a transpose) in one grouped
    launch: every output equals the single launch's bit for bit and the oracle's."""
    shapes = [(384, 256), (128, 128), (256, 640), (512, 384)]
    probs, singles = [], []
    for i, (N, K) in enumerate(shapes):
        w = W.weights(N, K, seed=60 + i).to(dev)
        out = (torch.empty(N, K, dtype=torch.uint8, device=dev),
               torch.empty(N // 128, K // 128, dtype=torch.float32, device=dev),
               None if i == 1 else torch.empty(K, N, dtype=torch.uint8, device=dev))
        probs.append((w, *out))
        singles.append(q_weight(w.cpu(), dev, with_t=i != 1))
    J.jetfp8_quant_weight_grouped(probs)
    check_errors()
    for i, ((w, q, s, qT), (q1, s1, qT1)) in enumerate(zip(probs, singles)):
        assert torch.equal(q, q1) and torch.equal(s, s1), i
        if qT is not None:
            assert torch.equal(qT, qT1), i
        oq, os_, oqT = O.quant_weight_128x128(W.bf16_values(w.cpu()))
        assert np.array_equal(h(q), oq) and np.array_equal(h(s), os_), i
        if qT is not None:
            assert np.array_equal(h(qT), oqT), i


@pytest.mark.parametrize("M,K", [(256, 512), (128, 128), (1024, 1536)])
def test_requant_parity(dev, M, K):
    x = W.activations(M, K, seed=0, stream=7)
    q, s = q_act(x, dev)
    qT, sT = requant(q, s, dev)
    oq, os_ = O.quant_act_1x128(W.bf16_values(x))
    oqT, osT = O.requant_rowgrp_to_colgrp(oq, os_)
    assert np.array_equal(h(sT), osT)
    assert np.array_equal(h(qT), oqT)


def test_requant_decodes_every_code(dev):
    """All 254 finite codes through the GPU decode with power-of-two row
    scales (exact dequantisation)."""
    g = np.random.default_rng(0)
    codes = np.tile(np.concatenate([np.arange(0x7F), np.arange(0x80, 0xFF)]).astype(np.uint8), 130)[:128 * 256]
    codes = codes.reshape(128, 256)
    g.shuffle(codes, axis=1)
    s = np.ldexp(1.0, g.integers(-8, 8, size=(2, 128))).astype(np.float32)
    q = torch.from_numpy(codes).to(dev)
    st = torch.from_numpy(s).to(dev)
    qT, sT = requant(q, st, dev)
    oqT, osT = O.requant_rowgrp_to_colgrp(codes, s)
    assert np.array_equal(h(sT), osT) and np.array_equal(h(qT), oqT)


@pytest.mark.parametrize("M,N", [(256, 384), (128, 128), (512, 1024)])
def test_quant_grad_dual_parity(dev, M, N):
    dy = W.gradients(M, N, seed=3)
    q, s, qT, sT = q_grad(dy, dev)
    oq, os_, oqT, osT = O.quant_grad_dual(W.bf16_values(dy))
    assert np.array_equal(h(s)[:, :M], os_) and np.array_equal(h(q), oq)
    assert np.array_equal(h(sT), osT) and np.array_equal(h(qT), oqT)


@pytest.mark.parametrize("M", [1, 200])
def test_quant_grad_rows_only_ragged(dev, M):
    dy = W.gradients(M, 384, seed=4)
    q, s, _, _ = q_grad(dy, dev, with_col=False)
    _assert_rowquant(q, s, W.bf16_values(dy))


def test_quant_grad_dual_rejects_ragged_columns(dev):
    dy = W.gradients(200, 128, seed=5).to(dev)
    q, s = J.empty_rowgroup_quant(200, 128, dev)
    qT = torch.empty(128, 200, dtype=torch.uint8, device=dev)
    sT = torch.empty(*J.scale_shape(128, 200), dtype=torch.float32, device=dev)
    with pytest.raises(J.JetFP8Error, match="UNSUPPORTED_SHAPE"):
        J.jetfp8_quant_grad_dual(dy, q, s, qT, sT)


@pytest.mark.parametrize("M,H", [(64, 4096), (5, 384), (300, 1024)])
def test_rmsnorm_quant_parity(dev, M, H):
    x = W.activations(M, H, seed=6)
    gamma = W.uniform((H,), 0.5, 1.5, seed=6, stream=9)
    q, s = J.empty_rowgroup_quant(M, H, dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    J.jetfp8_rmsnorm_quant(x.to(dev), gamma.to(dev), 1e-6, q, s, rstd, y)
    check_errors()
    oy, orstd, oq, os_ = O.rmsnorm_quant(W.bf16_values(x), W.bf16_values(gamma), 1e-6)
    gy = h(y.float()).astype(np.float64)
    # y within one bf16 ulp of the FP64 result rounded to bf16
    ulp = np.ldexp(1.0, np.frexp(np.abs(oy))[1] - 8)
    assert np.all(np.abs(gy - oy) <= ulp)
    # rstd: Σx² in FP32 as 16-square chains per lane and group, a binary tree
    # over a lane's groups and a butterfly over the lanes (at most 25 roundings
    # of positive terms), one more each for /H and +eps, halved by the square
    # root, plus the reciprocal square root's rounding -> at most 14·2^-24 to
    # first order; the test allows 16·2^-24.
    assert np.allclose(h(rstd), orstd, rtol=16 * 2.0 ** -24, atol=0)
    # the fused quantiser is bit-exact on the GPU's own y
    gq, gs = O.quant_rowgroups(gy.astype(np.float32))
    assert np.array_equal(h(s)[:, :M], gs) and np.array_equal(h(q), gq)
    # and end to end the codes match the oracle's except at rare bf16 ties
    mismatch = np.mean(h(q) != oq)
    assert mismatch < 1e-3


@pytest.mark.parametrize("M,I", [(64, 1024), (3, 128)])
def test_swiglu_quant_parity(dev, M, I):
    gu = W.normal((M, 2 * I), 2.0, seed=7)
    q, s = J.empty_rowgroup_quant(M, I, dev)
    hb = torch.empty(M, I, dtype=torch.bfloat16, device=dev)
    J.jetfp8_swiglu_quant(gu.to(dev), q, s, hb)
    check_errors()
    oh, oq, os_ = O.swiglu_quant(W.bf16_values(gu))
    gh = h(hb.float()).astype(np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(oh))[1] - 8)
    assert np.all(np.abs(gh - oh) <= ulp + 1e-40)
    gq, gs = O.quant_rowgroups(gh.astype(np.float32))
    assert np.array_equal(h(s)[:, :M], gs) and np.array_equal(h(q), gq)


def test_swiglu_bwd_parity(dev):
    M, I = 64, 512
    gu = W.normal((M, 2 * I), 2.0, seed=8)
    dh = W.normal((M, I), 1e-3, seed=8, stream=3)
    dgu = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dev)
    J.jetfp8_swiglu_bwd(gu.to(dev), dh.to(dev), dgu)
    check_errors()
    od = O.swiglu_bwd(W.bf16_values(gu), W.bf16_values(dh))
    gd = h(dgu.float()).astype(np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(od))[1] - 8)
    assert np.all(np.abs(gd - od) <= ulp + 1e-40)


# ---------------------------------------------------------------------------
# The division-free scale over every bf16 maximum, and the TMA-fed kernels'
# segment and width variants
# ---------------------------------------------------------------------------
def _group_maxima():
    """Every positive finite bf16 value (0x0001 .. 0x7F7F), then 0: 32640 = 255·128."""
    a = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    a = np.concatenate([a, np.zeros(1, np.float32)])
    assert a[-2] == np.float32(3.3895314e38) and np.all(np.isfinite(a)) and len(a) == 255 * 128
    return a


def _every_bf16_max_groups(seed):
    """[32640, 128] bf16 values: row r holds the r-th group maximum a_r at a
    random position (random sign) and otherwise values of magnitude ≤ a_r;
    the last row is all zeros."""
    a = _group_maxima()
    g = np.random.default_rng(seed)
    u = g.uniform(-1.0, 1.0, size=(len(a), 128)).astype(np.float64)
    x = W.to_bf16((u * a[:, None].astype(np.float64)).astype(np.float32))
    xf = W.bf16_values(x)
    assert np.all(np.abs(xf) <= a[:, None])
    pos = g.integers(0, 128, size=len(a))
    xf[np.arange(len(a)), pos] = a * np.where(g.random(len(a)) < 0.5, -1.0, 1.0).astype(np.float32)
    return W.to_bf16(xf), a


def test_quant_act_every_bf16_group_max(dev):
    """S = fp32(amax/448) from the kernels' division-free sequence, for every
    positive finite bf16 group maximum (one group each), codes included."""
    x, a = _every_bf16_max_groups(seed=41)
    q, s = q_act(x, dev)
    want = np.where(a == 0, np.float32(1.0), (a / np.float32(448.0)).astype(np.float32))
    assert np.array_equal(h(s)[0, :len(a)], want)
    _assert_rowquant(q, s, W.bf16_values(x))


def test_quant_grad_dual_every_bf16_group_max(dev):
    """The dual quantiser over every bf16 maximum, once as row groups (a
    [32640, 128] gradient) and once as 128-token column groups (its transpose)."""
    x, a = _every_bf16_max_groups(seed=42)
    xf = W.bf16_values(x)
    for t in (x, W.to_bf16(np.ascontiguousarray(xf.T))):
        q, s, qT, sT = q_grad(t, dev)
        oq, os_, oqT, osT = O.quant_grad_dual(W.bf16_values(t))
        M = t.shape[0]
        assert np.array_equal(h(s)[:, :M], os_) and np.array_equal(h(q), oq)
        assert np.array_equal(h(sT), osT) and np.array_equal(h(qT), oqT)


def test_quant_weight_block_max_sweep(dev):
    """128×128 blocks whose maxima step through the bf16 range (every 16th
    positive finite value, both extremes included)."""
    a = _group_maxima()[:-1]
    a = np.concatenate([a[::16][:2039], a[-1:]])
    assert a[-1] == np.float32(3.3895314e38) and len(a) == 2040
    nb = len(a)
    g = np.random.default_rng(43)
    blocks = (g.uniform(-1, 1, size=(nb, 128, 128)) * a[:, None, None].astype(np.float64)).astype(np.float32)
    blocks = W.bf16_values(W.to_bf16(blocks.reshape(nb * 128, 128))).reshape(nb, 128, 128)
    blocks[np.arange(nb), g.integers(0, 128, nb), g.integers(0, 128, nb)] = a
    # lay the blocks out as a [nb/8·128, 8·128] weight (8 blocks per block row)
    w = blocks.reshape(nb // 8, 8, 128, 128).transpose(0, 2, 1, 3).reshape(nb // 8 * 128, 8 * 128)
    wt = W.to_bf16(np.ascontiguousarray(w))
    q, s, qT = q_weight(wt, dev)
    oq, os_, oqT = O.quant_weight_128x128(W.bf16_values(wt))
    assert np.array_equal(h(s), os_) and np.array_equal(h(q), oq) and np.array_equal(h(qT), oqT)


def test_requant_scales_across_the_fp32_range(dev):
    """Requantisation with row scales log-uniform over most of the FP32 range,
    so column maxima x̃ = fp32(dec(q)·S) take the division-free scale above
    2^-100 and the division below it."""
    M, K = 1024, 1024
    g = np.random.default_rng(44)
    finite = np.concatenate([np.arange(0x7F), np.arange(0x80, 0xFF)]).astype(np.uint8)
    codes = g.choice(finite, size=(M, K))
    # one exponent per (k-block, 128-row band), jittered per row: a column
    # group's maximum follows its band's exponent, from 2^-126 to 2^100
    band = g.integers(-126, 100, size=(K // 128, M // 128))
    e = np.repeat(band, 128, axis=1) + g.integers(0, 4, size=(K // 128, M))
    s = np.ldexp(g.uniform(1.0, 2.0, size=(K // 128, M)), e).astype(np.float32)
    qT, sT = requant(torch.from_numpy(codes).to(dev), torch.from_numpy(s).to(dev), dev)
    oqT, osT = O.requant_rowgrp_to_colgrp(codes, s)
    assert np.any(osT < 2.0 ** -100 / 448) and np.any(osT > 1.0)
    assert np.array_equal(h(sT), osT) and np.array_equal(h(qT), oqT)


@pytest.mark.parametrize("M,K", [(5, 14336), (3, 4224), (9, 8192), (700, 256)])
def test_quant_act_row_segments(dev, M, K):
    """Rows longer than one streamed segment (4096 elements), with a short last one."""
    x = W.activations(M, K, seed=45, stream=K)
    q, s = q_act(x, dev)
    _assert_rowquant(q, s, W.bf16_values(x))


@pytest.mark.parametrize("M,H", [(40, 5120), (33, 8192), (17, 12288)])
def test_rmsnorm_quant_row_widths(dev, M, H):
    """The three R1 variants: rows streamed whole through 8 KB or 16 KB slots,
    and wider rows through the register kernel."""
    x = W.activations(M, H, seed=46)
    gamma = W.uniform((H,), 0.5, 1.5, seed=46, stream=9)
    q, s = J.empty_rowgroup_quant(M, H, dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    J.jetfp8_rmsnorm_quant(x.to(dev), gamma.to(dev), 1e-6, q, s, rstd, y)
    check_errors()
    oy, orstd, oq, os_ = O.rmsnorm_quant(W.bf16_values(x), W.bf16_values(gamma), 1e-6)
    gy = h(y.float()).astype(np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(oy))[1] - 8)
    assert np.all(np.abs(gy - oy) <= ulp)
    assert np.allclose(h(rstd), orstd, rtol=16 * 2.0 ** -24, atol=0)
    gq, gs = O.quant_rowgroups(gy.astype(np.float32))
    assert np.array_equal(h(s)[:, :M], gs) and np.array_equal(h(q), gq)
