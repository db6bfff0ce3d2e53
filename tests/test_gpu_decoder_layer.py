"""A decoder layer in the unified FP8 flow (every linear, quantiser, RMSNorm and
SwiGLU through the C ABI; BF16 attention core): the rollout-sized forward equals
the training-sized forward bit for bit for every sequence (Figure 5 of the Jet-RL
summary page: the inference graph is a subgraph of the training graph), and the
whole layer's outputs and gradients stay close to an FP32 autograd reference of
the same, unquantised layer (FP8 quantisation error only); and every library call
of one forward + backward matches the oracle on the inputs it received inside
the layer."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from fp8_mixed_granularity_gb300.decoder_layer import DecoderLayerFP8, LayerShape
from oracle import jetfp8_oracle as O
from tests.gpu_util import check_errors, gemm_tol_ok, h, rmsnorm_bwd_bounds

pytestmark = pytest.mark.gpu
SHAPE = LayerShape(hidden=512, heads=4, kv_heads=2, head_dim=128, intermediate=384)
B, S = 4, 64


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _weights(dev):
    s = SHAPE
    D, I = s.hidden, s.intermediate
    return {
        "wqkv": W.normal((s.qkv_width, D), 0.02, seed=50, stream=1).to(dev),
        "wo": W.normal((D, s.attn_width), 0.02, seed=50, stream=2).to(dev),
        "wgu": W.normal((2 * I, D), 0.02, seed=50, stream=3).to(dev),
        "wd": W.normal((D, I), 0.02, seed=50, stream=4).to(dev),
        "gamma1": W.uniform((D,), 0.5, 1.5, seed=50, stream=5).to(dev),
        "gamma2": W.uniform((D,), 0.5, 1.5, seed=50, stream=6).to(dev),
    }


def test_layer_forward_rows_do_not_depend_on_the_batch(dev):
    w = _weights(dev)
    x = W.activations(B * S, SHAPE.hidden, seed=51).to(dev)
    y_all = DecoderLayerFP8(SHAPE, w, dev).forward(x, B, S)
    for b0, nb in [(0, 1), (1, 2), (3, 1)]:
        xs = x[b0 * S:(b0 + nb) * S].contiguous()
        ys = DecoderLayerFP8(SHAPE, w, dev).forward(xs, nb, S)
        assert torch.equal(ys, y_all[b0 * S:(b0 + nb) * S]), (b0, nb)


def _reference(x, w, dy):
    """FP32 autograd of the same layer without quantisation."""
    s = SHAPE
    f = {k: v.float().clone().requires_grad_() for k, v in w.items()}
    xf = x.float().clone().requires_grad_()

    def rms(t, g):
        return t * torch.rsqrt((t * t).mean(dim=1, keepdim=True) + 1e-6) * g

    qkv = rms(xf, f["gamma1"]) @ f["wqkv"].T
    t = qkv.view(B, S, s.heads + 2 * s.kv_heads, s.head_dim).permute(0, 2, 1, 3)
    q, k, v = t[:, :s.heads], t[:, s.heads:s.heads + s.kv_heads], t[:, s.heads + s.kv_heads:]
    a = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
    h1 = xf + a.permute(0, 2, 1, 3).reshape(B * S, s.attn_width) @ f["wo"].T
    gu = rms(h1, f["gamma2"]) @ f["wgu"].T
    g_, u_ = gu[:, :s.intermediate], gu[:, s.intermediate:]
    y = h1 + (torch.nn.functional.silu(g_) * u_) @ f["wd"].T
    y.backward(dy.float())
    return y.detach(), xf.grad, {k: v.grad for k, v in f.items()}


def _rel(got, ref):
    got, ref = got.float(), ref.float()
    return float((got - ref).norm() / ref.norm())


def test_layer_forward_backward_close_to_fp32_reference(dev):
    w = _weights(dev)
    x = W.activations(B * S, SHAPE.hidden, seed=52).to(dev)
    dy = W.normal((B * S, SHAPE.hidden), 1e-3, seed=52, stream=1).to(dev)
    layer = DecoderLayerFP8(SHAPE, w, dev)
    y = layer.forward(x, B, S)
    dx, grads = layer.backward(dy)
    torch.cuda.synchronize()
    y_ref, dx_ref, g_ref = _reference(x, w, dy)
    errs = {"y": _rel(y, y_ref), "dx": _rel(dx, dx_ref)}
    errs.update({k: _rel(grads[k], g_ref[k]) for k in grads})
    print("relative errors against the FP32 reference:", {k: round(v, 4) for k, v in errs.items()})
    # E4M3 keeps 3 mantissa bits (≈ 3 % per element); per-group scales keep the
    # relative error of whole tensors at that order after the chained GEMMs
    assert errs["y"] < 0.02, errs
    assert all(np.isfinite(v) and v < 0.15 for v in errs.values()), errs


def _f64(t):
    return h(t.float()).astype(np.float64)


def _ulp(v):
    return np.ldexp(1.0, np.frexp(np.abs(v))[1] - 8)


def test_layer_stages_match_the_oracle(dev):
    """Every library call of one forward + backward of the layer, checked against
    the oracle on the inputs it received inside the layer: weight, activation,
    gradient and requantised codes and scales bit for bit; R1 and X1 through their
    normalised output (the same deterministic call, repeated with that output
    requested, gives the layer's codes, and its output is within one bf16 ulp of
    the oracle's with the codes exactly the oracle quantiser's on it); FProp, DGrad
    and WGrad within |Δ| <= 1e-2·|ref| + 1e-3·rms(ref) (plus the bf16 rounding of a
    residual add); the SwiGLU backward within one bf16 ulp; the RMSNorm backward
    within its derived bound.  The BF16 attention core is PyTorch's and is not
    checked here."""
    s = SHAPE
    T, D, I = B * S, s.hidden, s.intermediate
    w = _weights(dev)
    x = W.activations(T, D, seed=53).to(dev)
    dy = W.normal((T, D), 1e-3, seed=53, stream=1).to(dev)
    layer = DecoderLayerFP8(SHAPE, w, dev)
    y = layer.forward(x, B, S)
    dx, grads = layer.backward(dy)
    torch.cuda.synchronize()
    check_errors()
    sv, tr = layer.saved, layer.trace
    lins = {"wqkv": layer.qkv, "wo": layer.o, "wgu": layer.gu, "wd": layer.down}

    # Q2 (one grouped launch): every weight's codes, scales and transpose
    for name, lin in lins.items():
        oq, os_, oqT = O.quant_weight_128x128(_f64(w[name]).astype(np.float32))
        assert np.array_equal(h(lin.wq), oq) and np.array_equal(h(lin.sw), os_), name
        assert np.array_equal(h(lin.wqT), oqT), name

    def fprop_ref(xq, sx, lin):
        return O.gemm_fprop(h(xq), h(sx)[:, :T], h(lin.wq), h(lin.sw))

    def gemm(got, ref, what):
        ok, worst = gemm_tol_ok(got, ref)
        assert ok, (what, worst)

    def residual(out, base, ref, what):
        # out = bf16(base + GEMM): the GEMM bar plus the add's bf16 rounding
        got = _f64(out) - _f64(base)
        rms = float(np.sqrt(np.mean(ref * ref)))
        assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 1e-3 * rms + _ulp(_f64(out))), what

    def rmsnorm_stage(xin, gamma, rstd, xq, sx, what):
        q2, s2 = J.empty_rowgroup_quant(T, D, dev)
        r2 = torch.empty(T, dtype=torch.float32, device=dev)
        yb = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
        J.jetfp8_rmsnorm_quant(xin, gamma, 1e-6, q2, s2, r2, yb)
        check_errors()
        assert torch.equal(q2, xq) and torch.equal(s2, sx) and torch.equal(r2, rstd), what
        oy, orstd, _, _ = O.rmsnorm_quant(_f64(xin), _f64(gamma), 1e-6)
        gy = _f64(yb)
        assert np.all(np.abs(gy - oy) <= _ulp(oy)), what
        assert np.allclose(h(rstd), orstd, rtol=16 * 2.0 ** -24, atol=0), what
        gq, gs = O.quant_rowgroups(gy.astype(np.float32))
        assert np.array_equal(h(sx)[:, :T], gs) and np.array_equal(h(xq), gq), what

    # ---- forward ----
    rmsnorm_stage(x, w["gamma1"], sv["rstd1"], sv["xq1"], sv["sx1"], "R1 (attention norm)")
    q, k, v, a = sv["graph"]
    qkv = torch.cat([q, k, v], 1).detach().permute(0, 2, 1, 3).reshape(T, s.qkv_width)
    gemm(_f64(qkv), fprop_ref(sv["xq1"], sv["sx1"], layer.qkv), "QKV FProp")
    attn = a.detach().permute(0, 2, 1, 3).reshape(T, s.attn_width)
    oq, os_ = O.quant_act_1x128(_f64(attn).astype(np.float32))
    assert np.array_equal(h(sv["aq"]), oq) and np.array_equal(h(sv["sa"])[:, :T], os_), "Q1 (attention output)"
    residual(sv["h1"], x, fprop_ref(sv["aq"], sv["sa"], layer.o), "O FProp")
    rmsnorm_stage(sv["h1"], w["gamma2"], sv["rstd2"], sv["xq2"], sv["sx2"], "R1 (MLP norm)")
    gemm(_f64(sv["gu"]), fprop_ref(sv["xq2"], sv["sx2"], layer.gu), "gate/up FProp")
    q2, s2 = J.empty_rowgroup_quant(T, I, dev)
    hb = torch.empty(T, I, dtype=torch.bfloat16, device=dev)
    J.jetfp8_swiglu_quant(sv["gu"], q2, s2, hb)
    check_errors()
    assert torch.equal(q2, sv["hq"]) and torch.equal(s2, sv["hs"]), "X1 repeat"
    oh, _, _ = O.swiglu_quant(_f64(sv["gu"]))
    gh = _f64(hb)
    assert np.all(np.abs(gh - oh) <= _ulp(oh) + 1e-40), "X1 h"
    gq, gs = O.quant_rowgroups(gh.astype(np.float32))
    assert np.array_equal(h(sv["hq"]), gq) and np.array_equal(h(sv["hs"])[:, :T], gs), "X1 codes"
    residual(y, sv["h1"], fprop_ref(sv["hq"], sv["hs"], layer.down), "down FProp")

    # ---- backward ----
    def linear_bwd(lin, name, dyin, xq, sx, dxout, what):
        dyq, sdy = lin.last["dyq"], lin.last["sdy"]
        dyqT, sdyT, xqT, sxT, dw = tr["wgrad"][name]
        oqr, osr, oqc, osc = O.quant_grad_dual(_f64(dyin).astype(np.float32))
        assert np.array_equal(h(dyq), oqr) and np.array_equal(h(sdy)[:, :T], osr), what + " Q4 rows"
        assert np.array_equal(h(dyqT), oqc) and np.array_equal(h(sdyT), osc), what + " Q4 columns"
        gemm(_f64(dxout), O.gemm_dgrad(h(dyq), h(sdy)[:, :T], h(lin.wqT), h(lin.sw)), what + " DGrad")
        oxT, osT = O.requant_rowgrp_to_colgrp(h(xq), h(sx)[:, :T])
        assert np.array_equal(h(xqT), oxT) and np.array_equal(h(sxT), osT), what + " Q3"
        gemm(h(dw).astype(np.float64), O.gemm_wgrad(h(dyqT), h(sdyT), h(xqT), h(sxT)), what + " WGrad")

    def norm_bwd(xin, gamma, rstd, dyin, dxout, dg, what):
        exact, bound, dg_bound_of = rmsnorm_bwd_bounds(_f64(xin), _f64(gamma), h(rstd).astype(np.float64),
                                                       _f64(dyin))
        assert np.all(np.abs(_f64(dxout) - exact) <= _ulp(exact) + bound), what
        _, odg = O.rmsnorm_bwd(_f64(xin), _f64(gamma), h(rstd).astype(np.float64), _f64(dyin))
        assert np.all(np.abs(h(dg).astype(np.float64) - odg) <= dg_bound_of(odg)), what + " ∇γ"

    linear_bwd(layer.down, "wd", dy, sv["hq"], sv["hs"], tr["dh"], "down")
    od = O.swiglu_bwd(_f64(sv["gu"]), _f64(tr["dh"]))
    assert np.all(np.abs(_f64(tr["dgu"]) - od) <= _ulp(od) + 1e-40), "X2"
    linear_bwd(layer.gu, "wgu", tr["dgu"], sv["xq2"], sv["sx2"], tr["dxn2"], "gate/up")
    norm_bwd(sv["h1"], w["gamma2"], sv["rstd2"], tr["dxn2"], tr["dn2"], grads["gamma2"], "RMSNorm bwd (MLP)")
    linear_bwd(layer.o, "wo", tr["dh1"], sv["aq"], sv["sa"], tr["dattn"], "O")
    linear_bwd(layer.qkv, "wqkv", tr["dqkv"], sv["xq1"], sv["sx1"], tr["dxn1"], "QKV")
    norm_bwd(x, w["gamma1"], sv["rstd1"], tr["dxn1"], tr["dn1"], grads["gamma1"], "RMSNorm bwd (attention)")
