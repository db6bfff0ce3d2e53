"""Full-size parity, sampled: the quantisers and GEMMs at the sizes and in the
launch configuration the benchmark times (Llama-3.1-8B linears at 8192
tokens, their four WGrads as one grouped launch) and the Qwen3-8B decode
FProp, against the FP64 oracle on row stripes, column stripes and weight
blocks that the oracle computes on their own (every group lies wholly inside
a sample: stripes are 128-aligned).  Codes and scales bit-exact; GEMMs within
|Δ| <= 1e-2·|ref| + 1e-3·rms(ref)."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from oracle import jetfp8_oracle as O
from tests.gpu_util import check_errors, gemm_tol_ok, h, q_act, q_grad, q_weight, requant

pytestmark = pytest.mark.gpu

M_TRAIN = 8192


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _stripes(n, rng, k=2, width=128, edges=True):
    """k random 128-aligned stripes (plus the first and last when `edges`)."""
    blocks = set(rng.choice(n // width, size=k, replace=False).tolist())
    if edges:
        blocks |= {0, n // width - 1}
    return np.concatenate([np.arange(b * width, (b + 1) * width) for b in sorted(blocks)])


def _assert_close(got, ref, what):
    ok, worst = gemm_tol_ok(got, ref)
    assert ok, f"{what}: worst |Δ|/bound = {worst:.3g}"


def _lin(name):
    return next(l for l in W.llama8b_training(M_TRAIN) if l.name == name)


def test_quant_grad_dual_full_size(dev):
    """Q4 on the gate/up gradient [8192, 28672]: row groups of sampled rows and
    the transposed 128-token column groups of the same stripes."""
    lin = _lin("gate_up")
    rng = np.random.default_rng(1)
    dy = W.device_normal((lin.M, lin.N), 1e-3, dev, seed=3)
    q, s, qT, sT = q_grad(dy, dev)
    rows = _stripes(lin.M, rng)
    oq, os_, oqT, osT = O.quant_grad_dual(h(dy[rows].float()))
    assert np.array_equal(h(q[rows]), oq) and np.array_equal(h(s)[:, rows], os_)
    assert np.array_equal(h(qT[:, rows]), oqT)
    assert np.array_equal(h(sT)[rows[::128] // 128], osT)


def test_quant_weight_full_size(dev):
    """Q2 with Ŵᵀ on the gate/up weight [28672, 4096]: sampled 128-row block rows."""
    lin = _lin("gate_up")
    rng = np.random.default_rng(2)
    w = W.device_normal((lin.N, lin.K), 0.02, dev, seed=2)
    q, s, qT = q_weight(w, dev)
    rows = _stripes(lin.N, rng)
    oq, os_, oqT = O.quant_weight_128x128(h(w[rows].float()))
    assert np.array_equal(h(q[rows]), oq)
    assert np.array_equal(h(s)[rows[::128] // 128], os_)
    assert np.array_equal(h(qT[:, rows]), oqT)


def test_quant_act_and_requant_full_size(dev):
    """Q1 then Q3 on the down-projection input [8192, 14336]."""
    lin = _lin("down")
    rng = np.random.default_rng(3)
    x = W.device_activations(lin.M, lin.K, dev, seed=1)
    xq, sx = q_act(x, dev)
    xqT, sxT = requant(xq, sx, dev)
    rows = _stripes(lin.M, rng)
    oq, os_ = O.quant_act_1x128(h(x[rows].float()))
    assert np.array_equal(h(xq[rows]), oq) and np.array_equal(h(sx)[:, rows], os_)
    oqT, osT = O.requant_rowgrp_to_colgrp(oq, os_)
    assert np.array_equal(h(xqT[:, rows]), oqT)
    assert np.array_equal(h(sxT)[rows[::128] // 128], osT)


def test_rmsnorm_quant_full_size(dev):
    """R1 on the QKV / gate-up input [8192, 4096] (rows sampled)."""
    M, H = M_TRAIN, 4096
    rng = np.random.default_rng(4)
    x = W.device_activations(M, H, dev, seed=6)
    gamma = W.device_uniform((H,), 0.5, 1.5, dev, seed=7)
    q, s = J.empty_rowgroup_quant(M, H, dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    y = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    J.jetfp8_rmsnorm_quant(x, gamma, 1e-6, q, s, rstd, y)
    check_errors()
    rows = _stripes(M, rng)
    oy, orstd, oq, os_ = O.rmsnorm_quant(h(x[rows].float()), h(gamma.float()), 1e-6)
    gy = h(y[rows].float()).astype(np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(oy))[1] - 8)
    assert np.all(np.abs(gy - oy) <= ulp)
    assert np.allclose(h(rstd[rows]), orstd, rtol=16 * 2.0 ** -24, atol=0)
    gq, gs = O.quant_rowgroups(gy.astype(np.float32))
    assert np.array_equal(h(q[rows]), gq) and np.array_equal(h(s)[:, rows], gs)
    assert np.mean(h(q[rows]) != oq) < 1e-3


def test_grouped_wgrad_full_size(dev):
    """The four WGrads of the Llama-3.1-8B layer at 8192 tokens, bf16 ∇W: each
    single launch (the benchmark's launches) equals its problem in one grouped
    launch bit for bit, and sampled row and column stripes of the QKV and
    down-projection gradients match the oracle."""
    lins = W.llama8b_training(M_TRAIN)
    rng = np.random.default_rng(6)
    ops, dws = [], []
    for i, lin in enumerate(lins):
        x = W.device_activations(lin.M, lin.K, dev, seed=10 + i)
        dy = W.device_normal((lin.M, lin.N), 1e-3, dev, seed=20 + i)
        xq, sx = q_act(x, dev)
        xqT, sxT = requant(xq, sx, dev)
        del x, xq, sx
        _, _, dyqT, sdyT = q_grad(dy, dev)
        del dy
        ops.append((dyqT, sdyT, xqT, sxT))
        dws.append(torch.empty(lin.N, lin.K, dtype=torch.bfloat16, device=dev))
    J.jetfp8_gemm_wgrad_grouped([(*o, dw) for o, dw in zip(ops, dws)])
    check_errors()
    for o, dw in zip(ops, dws):
        single = torch.empty_like(dw)
        J.jetfp8_gemm_wgrad(*o, single)
        check_errors()
        assert torch.equal(single, dw)
        del single
    for i in (0, 3):
        dyqT, sdyT, xqT, sxT = (h(t) for t in ops[i])
        N, K = dws[i].shape
        rows, cols = _stripes(N, rng, k=1, edges=False), _stripes(K, rng, k=1, edges=False)
        _assert_close(h(dws[i][rows].float()), O.gemm_wgrad(dyqT, sdyT, xqT, sxT, rows=rows),
                      f"{lins[i].name} rows")
        _assert_close(h(dws[i][:, cols].float()), O.gemm_wgrad(dyqT, sdyT, xqT, sxT, cols=cols),
                      f"{lins[i].name} cols")


@pytest.mark.parametrize("M", [64, 256])
def test_decode_fprop_qwen3_full_size(dev, M):
    """Qwen3-8B decode FProp (channel-outlier activations, as the decode
    workload): gate/up (N = 24576) and down (K = 12288) at M tokens, every row
    on sampled column stripes and sampled rows on every column."""
    rng = np.random.default_rng(7 + M)
    for lin in W.qwen3_8b_decode(M):
        if lin.name not in ("gate_up", "down"):
            continue
        x = W.channel_outlier_activations(M, lin.K, seed=8, stream=M)
        w = W.device_normal((lin.N, lin.K), 0.02, dev, seed=9)
        xq, sx = q_act(x, dev)
        wq, sw, _ = q_weight(w, dev, with_t=False)
        y = torch.empty(M, lin.N, dtype=torch.bfloat16, device=dev)
        J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
        check_errors()
        hx, hsx, hw, hsw = h(xq), h(sx)[:, :M], h(wq), h(sw)
        cols = _stripes(lin.N, rng)
        rows = np.sort(rng.choice(M, size=4, replace=False))
        _assert_close(h(y[:, cols].float()), O.gemm_fprop(hx, hsx, hw, hsw, cols=cols), f"{lin.name} cols")
        _assert_close(h(y[rows].float()), O.gemm_fprop(hx, hsx, hw, hsw, rows=rows), f"{lin.name} rows")


# --------------------------------------------------------------------------
# Sub-block references: slices taken on the device, the oracle given only the
# rows, columns and scale blocks it needs (stripes are whole 128-blocks).
# --------------------------------------------------------------------------
def _fprop_ref(xq, sx, wq, sw, r, c):
    return O.gemm_fprop(h(xq[r]), h(sx)[:, r], h(wq[c]), h(sw)[c[::128] // 128])


def _dgrad_ref(dyq, sdy, wqT, sw, r, c):
    return O.gemm_dgrad(h(dyq[r]), h(sdy)[:, r], h(wqT[c]), h(sw)[:, c[::128] // 128])


def _wgrad_ref(dyqT, sdyT, xqT, sxT, r, c):
    return O.gemm_wgrad(h(dyqT[r]), h(sdyT)[:, r], h(xqT[c]), h(sxT)[:, c])


def _sub(t, r, c):
    return h(t[r][:, c].float())


def _rowquant_exact(q, s, vals_f32, r):
    """Codes and scales of rows r equal the oracle's 1×128 quantiser of vals."""
    oq, os_ = O.quant_rowgroups(vals_f32)
    assert np.array_equal(h(q[r]), oq) and np.array_equal(h(s)[:, r], os_)


def _bf16_within_ulp(got, ref):
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    return np.all(np.abs(got - ref) <= ulp + 1e-40)


def test_gated_mlp_chain_full_size(dev):
    """The gated-MLP block chain at 16384 tokens (hidden 4096, intermediate
    14336): RMSNorm+quant → gate/up FProp → SwiGLU+quant → down FProp, and the
    backward (dual gradient quantiser, DGrads, requantised operands, the two
    WGrads as one grouped launch, SwiGLU backward); every stage against the
    oracle on sampled stripes of the inputs the GPU actually gave it."""
    M, H, I = 16384, 4096, 14336
    rng = np.random.default_rng(11)
    bf = torch.bfloat16
    x = W.device_activations(M, H, dev, seed=31)
    gamma = W.device_uniform((H,), 0.5, 1.5, dev, seed=32)
    dy = W.device_normal((M, H), 1e-3, dev, seed=35)
    # forward
    xq, sx = J.empty_rowgroup_quant(M, H, dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    xn = torch.empty(M, H, dtype=bf, device=dev)
    J.jetfp8_rmsnorm_quant(x, gamma, 1e-6, xq, sx, rstd, xn)
    wq_gu, sw_gu, wqT_gu = q_weight(W.device_normal((2 * I, H), 0.02, dev, seed=33), dev)
    gu = torch.empty(M, 2 * I, dtype=bf, device=dev)
    J.jetfp8_gemm_fprop(xq, sx, wq_gu, sw_gu, gu)
    hq, hs = J.empty_rowgroup_quant(M, I, dev)
    hb = torch.empty(M, I, dtype=bf, device=dev)
    J.jetfp8_swiglu_quant(gu, hq, hs, hb)
    wq_d, sw_d, wqT_d = q_weight(W.device_normal((H, I), 0.02, dev, seed=34), dev)
    out = torch.empty(M, H, dtype=bf, device=dev)
    J.jetfp8_gemm_fprop(hq, hs, wq_d, sw_d, out)
    # backward
    dyq, sdy, dyqT, sdyT = q_grad(dy, dev)
    dh = torch.empty(M, I, dtype=bf, device=dev)
    J.jetfp8_gemm_dgrad(dyq, sdy, wqT_d, sw_d, dh)
    hqT, hsT = requant(hq, hs, dev)
    dgu = torch.empty(M, 2 * I, dtype=bf, device=dev)
    J.jetfp8_swiglu_bwd(gu, dh, dgu)
    dguq, sdgu, dguqT, sdguT = q_grad(dgu, dev)
    dxn = torch.empty(M, H, dtype=bf, device=dev)
    J.jetfp8_gemm_dgrad(dguq, sdgu, wqT_gu, sw_gu, dxn)
    xqT, sxT = requant(xq, sx, dev)
    dw_d = torch.empty(H, I, dtype=bf, device=dev)
    dw_gu = torch.empty(2 * I, H, dtype=bf, device=dev)
    J.jetfp8_gemm_wgrad_grouped([(dyqT, sdyT, hqT, hsT, dw_d), (dguqT, sdguT, xqT, sxT, dw_gu)])
    check_errors()

    r = _stripes(M, rng)
    cH, cI, cG = _stripes(H, rng), _stripes(I, rng), _stripes(2 * I, rng)
    # R1
    oy, _, _, _ = O.rmsnorm_quant(h(x[r].float()), h(gamma.float()), 1e-6)
    gy = h(xn[r].float()).astype(np.float64)
    assert _bf16_within_ulp(gy, oy)
    _rowquant_exact(xq, sx, gy.astype(np.float32), r)
    # gate/up FProp, SwiGLU + quantiser, down FProp
    _assert_close(_sub(gu, r, cG), _fprop_ref(xq, sx, wq_gu, sw_gu, r, cG), "gate/up fprop")
    oh, _, _ = O.swiglu_quant(h(gu[r].float()))
    gh = h(hb[r].float()).astype(np.float64)
    assert _bf16_within_ulp(gh, oh)
    _rowquant_exact(hq, hs, gh.astype(np.float32), r)
    _assert_close(_sub(out, r, cH), _fprop_ref(hq, hs, wq_d, sw_d, r, cH), "down fprop")
    # gradient quantiser, down DGrad, requant of h
    oq, os_, oqT, osT = O.quant_grad_dual(h(dy[r].float()))
    assert np.array_equal(h(dyq[r]), oq) and np.array_equal(h(sdy)[:, r], os_)
    assert np.array_equal(h(dyqT[:, r]), oqT) and np.array_equal(h(sdyT)[r[::128] // 128], osT)
    _assert_close(_sub(dh, r, cI), _dgrad_ref(dyq, sdy, wqT_d, sw_d, r, cI), "down dgrad")
    rq, rs = O.requant_rowgrp_to_colgrp(h(hq[r]), h(hs)[:, r])
    assert np.array_equal(h(hqT[:, r]), rq) and np.array_equal(h(hsT)[r[::128] // 128], rs)
    # SwiGLU backward, its gradient quantiser, gate/up DGrad, requant of X̂
    assert _bf16_within_ulp(h(dgu[r].float()).astype(np.float64),
                            O.swiglu_bwd(h(gu[r].float()), h(dh[r].float())))
    oq, os_, oqT, osT = O.quant_grad_dual(h(dgu[r].float()))
    assert np.array_equal(h(dguq[r]), oq) and np.array_equal(h(sdgu)[:, r], os_)
    assert np.array_equal(h(dguqT[:, r]), oqT) and np.array_equal(h(sdguT)[r[::128] // 128], osT)
    _assert_close(_sub(dxn, r, cH), _dgrad_ref(dguq, sdgu, wqT_gu, sw_gu, r, cH), "gate/up dgrad")
    rq, rs = O.requant_rowgrp_to_colgrp(h(xq[r]), h(sx)[:, r])
    assert np.array_equal(h(xqT[:, r]), rq) and np.array_equal(h(sxT)[r[::128] // 128], rs)
    # the two WGrads (one grouped launch)
    _assert_close(_sub(dw_d, cH, cI), _wgrad_ref(dyqT, sdyT, hqT, hsT, cH, cI), "down wgrad")
    _assert_close(_sub(dw_gu, cG, cH), _wgrad_ref(dguqT, sdguT, xqT, sxT, cG, cH), "gate/up wgrad")


def test_dense32b_gate_up_and_weight_requant_full_size(dev):
    """The 32B-class gate/up linear at 16384 tokens (K = 5120, N = 51200):
    FProp, DGrad and WGrad on sampled sub-blocks; then every 32B-class layer
    weight requantised after a synthetic update W += N(0, 1e-4), sampled
    128-row block stripes against the oracle on the updated weights."""
    lin = next(l for l in W.dense32b_training() if l.name == "gate_up")
    M, K, N = lin.M, lin.K, lin.N
    rng = np.random.default_rng(12)
    x = W.device_activations(M, K, dev, seed=41)
    xq, sx = q_act(x, dev)
    del x
    wq, sw, wqT = q_weight(W.device_normal((N, K), 0.02, dev, seed=42), dev)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
    dy = W.device_normal((M, N), 1e-3, dev, seed=43)
    dyq, sdy, dyqT, sdyT = q_grad(dy, dev)
    del dy
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_dgrad(dyq, sdy, wqT, sw, dx)
    xqT, sxT = requant(xq, sx, dev)
    dw = torch.empty(N, K, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw)
    check_errors()
    r, cN, cK = _stripes(M, rng), _stripes(N, rng), _stripes(K, rng)
    _assert_close(_sub(y, r, cN), _fprop_ref(xq, sx, wq, sw, r, cN), "fprop")
    _assert_close(_sub(dx, r, cK), _dgrad_ref(dyq, sdy, wqT, sw, r, cK), "dgrad")
    _assert_close(_sub(dw, cN, cK), _wgrad_ref(dyqT, sdyT, xqT, sxT, cN, cK), "wgrad")
    del y, dx, dw, dyq, dyqT, wq, wqT
    for i, l in enumerate(W.dense32b_training()):
        w = W.device_normal((l.N, l.K), 0.02, dev, seed=50 + i)
        upd = W.device_normal((l.N, l.K), 1e-4, dev, seed=60 + i)
        w2 = (w.float() + upd.float()).to(torch.bfloat16)
        q2, s2, qT2 = q_weight(w2, dev)
        rows = _stripes(l.N, rng)
        oq, os_, oqT = O.quant_weight_128x128(h(w2[rows].float()))
        assert np.array_equal(h(q2[rows]), oq), l.name
        assert np.array_equal(h(s2)[rows[::128] // 128], os_), l.name
        assert np.array_equal(h(qT2[:, rows]), oqT), l.name
