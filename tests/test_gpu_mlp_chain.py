"""The decoder-MLP chain through the library (the gated-MLP workload: RMSNorm
→ gate/up → SwiGLU → down, and its backward), every stage checked against the
oracle on the inputs the GPU actually gave it, so the stages' layouts and
hand-offs are exercised together: RMSNorm+quantiser output into FProp,
FProp output into the SwiGLU quantiser, the quantised h into the down
FProp and (requantised) into its WGrad, the down DGrad output into the
SwiGLU backward, and its output into the dual gradient quantiser."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from oracle import jetfp8_oracle as O
from tests.gpu_util import check_errors, gemm_tol_ok, h, q_grad, q_weight, requant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _close(got, ref, what):
    ok, worst = gemm_tol_ok(got, ref)
    assert ok, f"{what}: worst |Δ|/bound = {worst:.3g}"


def _bf16_within_ulp(got, ref):
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    return np.all(np.abs(got - ref) <= ulp + 1e-40)


def test_gated_mlp_forward_backward_chain(dev):
    M, Hd, I = 256, 512, 384
    x = W.activations(M, Hd, seed=31)
    gamma = W.uniform((Hd,), 0.5, 1.5, seed=31, stream=1)
    w_gu = W.weights(2 * I, Hd, seed=31, stream=2)
    w_d = W.weights(Hd, I, seed=31, stream=3)
    dy = W.gradients(M, Hd, seed=31, stream=4)
    bf = torch.bfloat16

    # ---- forward ----
    xq, sx = J.empty_rowgroup_quant(M, Hd, dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    xn = torch.empty(M, Hd, dtype=bf, device=dev)
    J.jetfp8_rmsnorm_quant(x.to(dev), gamma.to(dev), 1e-6, xq, sx, rstd, xn)
    wq_gu, sw_gu, wqT_gu = q_weight(w_gu, dev)
    gu = torch.empty(M, 2 * I, dtype=bf, device=dev)
    J.jetfp8_gemm_fprop(xq, sx, wq_gu, sw_gu, gu)
    hq, hs = J.empty_rowgroup_quant(M, I, dev)
    hb = torch.empty(M, I, dtype=bf, device=dev)
    J.jetfp8_swiglu_quant(gu, hq, hs, hb)
    wq_d, sw_d, wqT_d = q_weight(w_d, dev)
    out = torch.empty(M, Hd, dtype=bf, device=dev)
    J.jetfp8_gemm_fprop(hq, hs, wq_d, sw_d, out)
    check_errors()

    oy, _, _, _ = O.rmsnorm_quant(W.bf16_values(x), W.bf16_values(gamma), 1e-6)
    gy = h(xn.float()).astype(np.float64)
    assert _bf16_within_ulp(gy, oy)
    gq, gs = O.quant_rowgroups(gy.astype(np.float32))
    assert np.array_equal(h(xq), gq) and np.array_equal(h(sx)[:, :M], gs)
    _close(h(gu.float()), O.gemm_fprop(h(xq), h(sx)[:, :M], h(wq_gu), h(sw_gu)), "gate/up fprop")
    oh, _, _ = O.swiglu_quant(h(gu.float()))
    gh = h(hb.float()).astype(np.float64)
    assert _bf16_within_ulp(gh, oh)
    ghq, ghs = O.quant_rowgroups(gh.astype(np.float32))
    assert np.array_equal(h(hq), ghq) and np.array_equal(h(hs)[:, :M], ghs)
    _close(h(out.float()), O.gemm_fprop(h(hq), h(hs)[:, :M], h(wq_d), h(sw_d)), "down fprop")

    # ---- backward ----
    dyq, sdy, dyqT, sdyT = q_grad(dy, dev)
    dh = torch.empty(M, I, dtype=bf, device=dev)
    J.jetfp8_gemm_dgrad(dyq, sdy, wqT_d, sw_d, dh)
    hqT, hsT = requant(hq, hs, dev)
    dw_d = torch.empty(Hd, I, dtype=torch.float32, device=dev)
    J.jetfp8_gemm_wgrad(dyqT, sdyT, hqT, hsT, dw_d)
    dgu = torch.empty(M, 2 * I, dtype=bf, device=dev)
    J.jetfp8_swiglu_bwd(gu, dh, dgu)
    dguq, sdgu, dguqT, sdguT = q_grad(dgu, dev)
    dxn = torch.empty(M, Hd, dtype=bf, device=dev)
    J.jetfp8_gemm_dgrad(dguq, sdgu, wqT_gu, sw_gu, dxn)
    xqT, sxT = requant(xq, sx, dev)
    dw_gu = torch.empty(2 * I, Hd, dtype=torch.float32, device=dev)
    J.jetfp8_gemm_wgrad(dguqT, sdguT, xqT, sxT, dw_gu)
    check_errors()

    oq, os_, oqT, osT = O.quant_grad_dual(W.bf16_values(dy))
    assert np.array_equal(h(dyq), oq) and np.array_equal(h(dyqT), oqT)
    assert np.array_equal(h(sdy)[:, :M], os_) and np.array_equal(h(sdyT), osT)
    _close(h(dh.float()), O.gemm_dgrad(h(dyq), h(sdy)[:, :M], h(wqT_d), h(sw_d)), "down dgrad")
    rq, rs = O.requant_rowgrp_to_colgrp(h(hq), h(hs)[:, :M])
    assert np.array_equal(h(hqT), rq) and np.array_equal(h(hsT), rs)
    _close(h(dw_d), O.gemm_wgrad(h(dyqT), h(sdyT), h(hqT), h(hsT)), "down wgrad")
    assert _bf16_within_ulp(h(dgu.float()).astype(np.float64),
                            O.swiglu_bwd(h(gu.float()), h(dh.float())))
    oq, os_, oqT, osT = O.quant_grad_dual(h(dgu.float()))
    assert np.array_equal(h(dguq), oq) and np.array_equal(h(dguqT), oqT)
    _close(h(dxn.float()), O.gemm_dgrad(h(dguq), h(sdgu)[:, :M], h(wqT_gu), h(sw_gu)), "gate/up dgrad")
    _close(h(dw_gu), O.gemm_wgrad(h(dguqT), h(sdguT), h(xqT), h(sxT)), "gate/up wgrad")
