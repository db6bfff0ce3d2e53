"""One FP8 linear layer's forward and backward through the jetfp8 C ABI.

The order of calls follows the Jet-RL method steps ("Jet-RL：通过统一训练与推理精度流实现
On-Policy FP8 强化学习", 方法步骤详情):

  forward   X --(RMSNorm+)1×128 quant--> X̂ (kept for backward, step 3)
            W --128×128 quant--> Ŵ, Ŵᵀ (step 1; the transpose serves DGrad, step 4)
            Y = X̂·Ŵᵀ (FProp, step 2)
  backward  ∇Y (BF16) --dual quant--> 1×128 rows + 128×1 columns (step 4)
            ∇X = ∇Ŷ·Ŵ (DGrad with Ŵᵀ)
            X̂ --requantise 1×128→128×1, transpose--> X̂ᵀ
            ∇W = ∇Ŷᵀ·X̂ (WGrad)

All buffers are allocated once, on the device, by `LinearBuffers`; a step
only launches kernels.  Every call goes to the CUDA library: there is no
other code path.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import jetfp8 as J
from .workloads import Linear


@dataclass
class LinearBuffers:
    lin: Linear
    device: torch.device
    rmsnorm: bool = False          # the layer input passes through RMSNorm first
    wgrad_fp32: bool = False
    t: dict = field(default_factory=dict)

    def __post_init__(self):
        M, K, N = self.lin.M, self.lin.K, self.lin.N
        d, u8, f32, bf = self.device, torch.uint8, torch.float32, torch.bfloat16
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=d)  # noqa: E731
        self.t.update(
            xq=e(M, K, dt=u8), sx=e(*J.scale_shape(M, K), dt=f32),
            wq=e(N, K, dt=u8), sw=e(N // 128, K // 128, dt=f32), wqT=e(K, N, dt=u8),
            y=e(M, N, dt=bf),
            dyq=e(M, N, dt=u8), sdy=e(*J.scale_shape(M, N), dt=f32),
            dyqT=e(N, M, dt=u8), sdyT=e(*J.scale_shape(N, M), dt=f32),
            dx=e(M, K, dt=bf),
            xqT=e(K, M, dt=u8), sxT=e(*J.scale_shape(K, M), dt=f32),
            dw=e(N, K, dt=f32 if self.wgrad_fp32 else bf),
        )
        if self.rmsnorm:
            self.t.update(rstd=e(M, dt=f32))

    # Each method returns the number of kernels it launched.
    def forward(self, x: torch.Tensor, w: torch.Tensor | None, gamma: torch.Tensor | None = None,
                stream=None, events=None) -> int:
        """Input quantiser, Q2 of w (skipped when w is None: the weight was
        already quantised, e.g. by `quant_weights_grouped`) and FProp."""
        t = self.t
        if self.rmsnorm:
            _timed(events, "rmsnorm_quant",
                   lambda: J.jetfp8_rmsnorm_quant(x, gamma, 1e-6, t["xq"], t["sx"], t["rstd"], None, stream), stream)
        else:
            _timed(events, "quant_act", lambda: J.jetfp8_quant_act_1x128(x, t["xq"], t["sx"], stream), stream)
        n = 2
        if w is not None:
            _timed(events, "quant_weight",
                   lambda: J.jetfp8_quant_weight_128x128(w, t["wq"], t["sw"], t["wqT"], stream), stream)
            n += 1
        _timed(events, "gemm_fprop",
               lambda: J.jetfp8_gemm_fprop(t["xq"], t["sx"], t["wq"], t["sw"], t["y"], stream), stream)
        return n

    def backward(self, dy: torch.Tensor, stream=None, events=None, wgrad: bool = True) -> int:
        """Q4, F2, Q3 and (unless `wgrad` is False, for a later grouped
        launch by `wgrad_grouped`) F3.  Returns the number of launches."""
        t = self.t
        _timed(events, "quant_grad_dual",
               lambda: J.jetfp8_quant_grad_dual(dy, t["dyq"], t["sdy"], t["dyqT"], t["sdyT"], stream), stream)
        _timed(events, "gemm_dgrad",
               lambda: J.jetfp8_gemm_dgrad(t["dyq"], t["sdy"], t["wqT"], t["sw"], t["dx"], stream), stream)
        _timed(events, "requant",
               lambda: J.jetfp8_requant_rowgrp_to_colgrp(t["xq"], t["sx"], t["xqT"], t["sxT"], stream), stream)
        if not wgrad:
            return 3
        _timed(events, "gemm_wgrad",
               lambda: J.jetfp8_gemm_wgrad(t["dyqT"], t["sdyT"], t["xqT"], t["sxT"], t["dw"], stream), stream)
        return 4


def quant_weights_grouped(bufs, weights, stream=None, events=None) -> int:
    """Q2 (with the transposes) of the weights of several linears in grouped
    launches of up to MAX_GROUP weights each, before their forwards (which then
    take w=None).  Returns the number of launches."""
    n = 0
    for i in range(0, len(bufs), J.MAX_GROUP):
        probs = [(w, b.t["wq"], b.t["sw"], b.t["wqT"])
                 for b, w in zip(bufs[i:i + J.MAX_GROUP], weights[i:i + J.MAX_GROUP])]
        _timed(events, "quant_weight_grouped", lambda: J.jetfp8_quant_weight_grouped(probs, stream), stream)
        n += 1
    return n


def wgrad_grouped(bufs, stream=None, events=None) -> int:
    """F3 of several linears (same token count; their backward already ran
    with wgrad=False) in grouped launches of up to MAX_GROUP problems each.
    Returns the number of launches."""
    n = 0
    for i in range(0, len(bufs), J.MAX_GROUP):
        probs = [(b.t["dyqT"], b.t["sdyT"], b.t["xqT"], b.t["sxT"], b.t["dw"]) for b in bufs[i:i + J.MAX_GROUP]]
        _timed(events, "gemm_wgrad_grouped", lambda: J.jetfp8_gemm_wgrad_grouped(probs, stream), stream)
        n += 1
    return n


class EventLog(list):
    """A list for `events` whose CUDA events are created as graph event-record
    nodes (`external`), for timing launches inside a captured CUDA graph."""
    external = True


def _timed(events, name, fn, stream=None):
    """Run fn, which launches on `stream` (None: the current stream); if
    `events` (a list) is given, bracket it with CUDA events recorded on that
    same stream and append (name, start, end)."""
    if events is None:
        fn()
        return
    st = torch.cuda.current_stream() if stream is None else stream
    kw = {"external": True} if getattr(events, "external", False) else {}
    s = torch.cuda.Event(enable_timing=True, **kw)
    e = torch.cuda.Event(enable_timing=True, **kw)
    s.record(st)
    fn()
    e.record(st)
    events.append((name, s, e))
