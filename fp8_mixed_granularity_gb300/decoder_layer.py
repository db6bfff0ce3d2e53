"""A decoder layer in the unified FP8 precision flow, through the jetfp8 C ABI.

Every linear layer runs the Jet-RL mixed-granularity path ("Jet-RL：通过统一训练与推理精度流实现
On-Policy FP8 强化学习", 核心方法 and 方法步骤详情): activations quantised in 1×128
groups (fused with RMSNorm where the linear follows a norm, with SwiGLU before the
down projection), weights in 128×128 blocks, FP8 FProp / DGrad / WGrad with FP32
scales, gradients quantised from BF16 in both groupings, the saved activation
requantised for WGrad.  The attention core stays BF16, as on the pages; it is
PyTorch's scaled-dot-product attention, called one sequence at a time so that a
sequence's result does not depend on the batch it is computed in.  Residual adds
are BF16 tensor additions.  No rotary position embedding (the pages do not
describe the model beyond its linear layers).

    forward   h1 = x + O(attn(QKV(rmsnorm₁(x))))
              y  = h1 + Down(swiglu(GateUp(rmsnorm₂(h1))))
    backward  the same chain in reverse; RMSNorm backward from the saved r.

`forward` keeps what `backward` needs; weights are quantised (with their
transposes) at every forward, as a training step sees new weights each step.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import jetfp8 as J

_BF, _U8, _F32 = torch.bfloat16, torch.uint8, torch.float32


@dataclass(frozen=True)
class LayerShape:
    hidden: int          # D
    heads: int           # query heads
    kv_heads: int        # key/value heads (grouped-query attention)
    head_dim: int        # 128
    intermediate: int    # I

    @property
    def qkv_width(self) -> int:
        return (self.heads + 2 * self.kv_heads) * self.head_dim

    @property
    def attn_width(self) -> int:
        return self.heads * self.head_dim

    def linears(self, tokens: int):
        """(name, M, N, K) of the four linear layers."""
        D, I = self.hidden, self.intermediate
        return [("qkv", tokens, self.qkv_width, D), ("o", tokens, D, self.attn_width),
                ("gate_up", tokens, 2 * I, D), ("down", tokens, D, I)]


def llama8b() -> LayerShape:
    return LayerShape(hidden=4096, heads=32, kv_heads=8, head_dim=128, intermediate=14336)


class _QLinear:
    """One FP8 linear: its quantised weight (filled by the layer's grouped Q2), FProp, and the backward pair."""

    def __init__(self, N: int, K: int, dev):
        self.N, self.K = N, K
        self.wq = torch.empty(N, K, dtype=_U8, device=dev)
        self.sw = torch.empty(N // 128, K // 128, dtype=_F32, device=dev)
        self.wqT = torch.empty(K, N, dtype=_U8, device=dev)

    def fprop(self, xq, sx):
        y = torch.empty(xq.shape[0], self.N, dtype=_BF, device=xq.device)
        J.jetfp8_gemm_fprop(xq, sx, self.wq, self.sw, y)
        return y

    def backward(self, dy, xq, sx):
        """dy bf16 [M, N] -> (dx bf16 [M, K], WGrad problem); xq, sx: the saved
        quantised input (requantised here into 128-token groups for WGrad).
        The WGrad problem (dyqT, sdyT, xqT, sxT, dW fp32 [N, K]) is computed
        later, with the layer's other WGrads, in one grouped launch."""
        M = dy.shape[0]
        dev = dy.device
        dyq, sdy = J.empty_rowgroup_quant(M, self.N, dev)
        dyqT, sdyT = J.empty_rowgroup_quant(self.N, M, dev)
        J.jetfp8_quant_grad_dual(dy, dyq, sdy, dyqT, sdyT)
        dx = torch.empty(M, self.K, dtype=_BF, device=dev)
        J.jetfp8_gemm_dgrad(dyq, sdy, self.wqT, self.sw, dx)
        xqT, sxT = J.empty_rowgroup_quant(self.K, M, dev)
        J.jetfp8_requant_rowgrp_to_colgrp(xq, sx, xqT, sxT)
        dw = torch.empty(self.N, self.K, dtype=_F32, device=dev)
        # the quantised gradient of the last backward (references only), for inspection
        self.last = dict(dyq=dyq, sdy=sdy)
        return dx, (dyqT, sdyT, xqT, sxT, dw)


class DecoderLayerFP8:
    """Weights (bf16): wqkv [qkv_width, D], wo [D, attn_width], wgu [2I, D]
    (gate rows then up rows), wd [D, I], gamma1/gamma2 [D].  Tokens are
    `batch` sequences of `seq` tokens, row-major [batch·seq, D]."""

    def __init__(self, shape: LayerShape, weights: dict, dev, eps: float = 1e-6):
        self.s, self.w, self.eps, self.dev = shape, weights, eps, dev
        D, I = shape.hidden, shape.intermediate
        self.qkv = _QLinear(shape.qkv_width, D, dev)
        self.o = _QLinear(D, shape.attn_width, dev)
        self.gu = _QLinear(2 * I, D, dev)
        self.down = _QLinear(D, I, dev)
        self.saved = None

    def _attention(self, qkv, batch, seq):
        """BF16 causal grouped-query attention, one sequence at a time."""
        s = self.s
        hq, hkv, d = s.heads, s.kv_heads, s.head_dim
        t = qkv.view(batch, seq, hq + 2 * hkv, d).permute(0, 2, 1, 3)   # [B, heads, S, d]
        q = t[:, :hq].detach().clone().requires_grad_()
        k = t[:, hq:hq + hkv].detach().clone().requires_grad_()
        v = t[:, hq + hkv:].detach().clone().requires_grad_()
        outs = [torch.nn.functional.scaled_dot_product_attention(
                    q[b:b + 1], k[b:b + 1], v[b:b + 1], is_causal=True, enable_gqa=True)
                for b in range(batch)]
        a = torch.cat(outs, 0)                                           # [B, hq, S, d]
        flat = a.detach().permute(0, 2, 1, 3).reshape(batch * seq, hq * d).contiguous()
        return flat, (q, k, v, a)

    def forward(self, x, batch: int, seq: int):
        s, w, dev = self.s, self.w, self.dev
        T, D = x.shape
        # the four weights in one grouped launch (each output as the single launch's)
        J.jetfp8_quant_weight_grouped([(w[name], lin.wq, lin.sw, lin.wqT) for lin, name in (
            (self.qkv, "wqkv"), (self.o, "wo"), (self.gu, "wgu"), (self.down, "wd"))])
        # attention block: RMSNorm fused with the 1×128 quantiser, QKV, attention, O
        xq1, sx1 = J.empty_rowgroup_quant(T, D, dev)
        rstd1 = torch.empty(T, dtype=_F32, device=dev)
        J.jetfp8_rmsnorm_quant(x, w["gamma1"], self.eps, xq1, sx1, rstd1)
        qkv = self.qkv.fprop(xq1, sx1)
        attn, graph = self._attention(qkv, batch, seq)
        aq, sa = J.empty_rowgroup_quant(T, s.attn_width, dev)
        J.jetfp8_quant_act_1x128(attn, aq, sa)
        h1 = x + self.o.fprop(aq, sa)
        # MLP block: RMSNorm + quantiser, gate/up, SwiGLU + quantiser, down
        xq2, sx2 = J.empty_rowgroup_quant(T, D, dev)
        rstd2 = torch.empty(T, dtype=_F32, device=dev)
        J.jetfp8_rmsnorm_quant(h1, w["gamma2"], self.eps, xq2, sx2, rstd2)
        gu = self.gu.fprop(xq2, sx2)
        hq, hs = J.empty_rowgroup_quant(T, s.intermediate, dev)
        J.jetfp8_swiglu_quant(gu, hq, hs)
        y = h1 + self.down.fprop(hq, hs)
        self.saved = dict(x=x, rstd1=rstd1, xq1=xq1, sx1=sx1, graph=graph, aq=aq, sa=sa, h1=h1,
                          rstd2=rstd2, xq2=xq2, sx2=sx2, gu=gu, hq=hq, hs=hs, batch=batch, seq=seq)
        return y

    def backward(self, dy):
        """dy bf16 [T, D] -> (dx bf16 [T, D], grads dict: fp32 weight and γ gradients).
        The four weight gradients do not feed anything later in the backward:
        they are computed at the end, in one grouped WGrad launch."""
        sv, w, s, dev = self.saved, self.w, self.s, self.dev
        T, D = dy.shape
        grads, wgrads = {}, {}
        ws = torch.empty(J.jetfp8_rmsnorm_bwd_workspace_bytes(T, D), dtype=_U8, device=dev)
        # MLP block
        dh, wgrads["wd"] = self.down.backward(dy, sv["hq"], sv["hs"])
        dgu = torch.empty(T, 2 * s.intermediate, dtype=_BF, device=dev)
        J.jetfp8_swiglu_bwd(sv["gu"], dh, dgu)
        dxn2, wgrads["wgu"] = self.gu.backward(dgu, sv["xq2"], sv["sx2"])
        dn2 = torch.empty(T, D, dtype=_BF, device=dev)
        grads["gamma2"] = torch.empty(D, dtype=_F32, device=dev)
        J.jetfp8_rmsnorm_bwd(sv["h1"], w["gamma2"], sv["rstd2"], dxn2, dn2, grads["gamma2"], ws)
        dh1 = dy + dn2
        # attention block
        dattn, wgrads["wo"] = self.o.backward(dh1, sv["aq"], sv["sa"])
        q, k, v, a = sv["graph"]
        B, S, hq, d = sv["batch"], sv["seq"], s.heads, s.head_dim
        da = dattn.view(B, S, hq, d).permute(0, 2, 1, 3)
        dq, dk, dv = torch.autograd.grad(a, (q, k, v), da)
        dqkv = torch.cat([dq, dk, dv], 1).permute(0, 2, 1, 3).reshape(T, s.qkv_width).contiguous()
        dxn1, wgrads["wqkv"] = self.qkv.backward(dqkv, sv["xq1"], sv["sx1"])
        dn1 = torch.empty(T, D, dtype=_BF, device=dev)
        grads["gamma1"] = torch.empty(D, dtype=_F32, device=dev)
        J.jetfp8_rmsnorm_bwd(sv["x"], w["gamma1"], sv["rstd1"], dxn1, dn1, grads["gamma1"], ws)
        dx = dh1 + dn1
        J.jetfp8_gemm_wgrad_grouped(list(wgrads.values()))
        grads.update({k: p[4] for k, p in wgrads.items()})
        # the backward's intermediates (references only), for inspection
        self.trace = dict(dh=dh, dgu=dgu, dxn2=dxn2, dn2=dn2, dh1=dh1, dattn=dattn, dqkv=dqkv,
                          dxn1=dxn1, dn1=dn1, wgrad=wgrads)
        return dx, grads
