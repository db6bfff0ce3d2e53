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
    """The four WGrads of the Llama-3.1-8B layer at 8192 tokens in one grouped
    launch (the benchmark's launch), bf16 ∇W: sampled row and column stripes
    of the QKV and down-projection gradients against the oracle."""
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
