"""A decoder layer in the unified FP8 flow (every linear, quantiser, RMSNorm and
SwiGLU through the C ABI; BF16 attention core): the rollout-sized forward equals
the training-sized forward bit for bit for every sequence (Figure 5 of the Jet-RL
summary page: the inference graph is a subgraph of the training graph), and the
whole layer's outputs and gradients stay close to an FP32 autograd reference of
the same, unquantised layer (FP8 quantisation error only; each stage's exact
parity is tested on its own)."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import workloads as W
from fp8_mixed_granularity_gb300.decoder_layer import DecoderLayerFP8, LayerShape

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
