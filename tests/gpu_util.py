"""Helpers for the GPU parity tests: run each C-ABI entry point on seeded
inputs and bring the results back as numpy arrays."""
import numpy as np
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J


def h(t):
    return t.detach().cpu().numpy()


def check_errors():
    J.jetfp8_get_last_device_error()


def q_act(x_bf16, dev):
    M, K = x_bf16.shape
    q, s = J.empty_rowgroup_quant(M, K, dev)
    s.fill_(float("nan"))          # padding must never be read
    J.jetfp8_quant_act_1x128(x_bf16.to(dev), q, s)
    check_errors()
    return q, s


def q_weight(w_bf16, dev, with_t=True):
    N, K = w_bf16.shape
    q = torch.empty(N, K, dtype=torch.uint8, device=dev)
    s = torch.empty(N // 128, K // 128, dtype=torch.float32, device=dev)
    qT = torch.empty(K, N, dtype=torch.uint8, device=dev) if with_t else None
    J.jetfp8_quant_weight_128x128(w_bf16.to(dev), q, s, qT)
    check_errors()
    return q, s, qT


def q_grad(dy_bf16, dev, with_col=True):
    M, N = dy_bf16.shape
    q, s = J.empty_rowgroup_quant(M, N, dev)
    s.fill_(float("nan"))
    qT, sT = J.empty_rowgroup_quant(N, M, dev) if with_col else (None, None)
    J.jetfp8_quant_grad_dual(dy_bf16.to(dev), q, s, qT, sT)
    check_errors()
    return q, s, qT, sT


def requant(q, s, dev):
    M, K = q.shape
    qT, sT = J.empty_rowgroup_quant(K, M, dev)
    J.jetfp8_requant_rowgrp_to_colgrp(q, s, qT, sT)
    check_errors()
    return qT, sT


def gemm_tol_ok(got, ref, rel=1e-2, rms_frac=1e-3):
    """|Δ| <= rel·|ref| + rms_frac·rms(ref) elementwise; returns (ok, worst ratio)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bound = rel * np.abs(ref) + rms_frac * rms
    ratio = np.abs(got - ref) / np.maximum(bound, 1e-300)
    return bool(np.all(ratio <= 1.0)), float(ratio.max()) if ratio.size else 0.0


def rmsnorm_bwd_bounds(xf, gf, r, dyf):
    """For the RMSNorm backward on FP64 copies of its inputs (x, γ, the GPU's r,
    dy): the exact ∇x before rounding and the per-element bound on the kernel's
    FP32 evaluation error (each FP32 operation rounded separately, row sums as
    16-term FP32 chunks added in FP32 and combined in FP64; factor 2 margin),
    and the bound on ∇γ.  ∇γ is an FP32 chain over at most 128 rows per partial
    (a 128-row chunk, or one warp's rows plus the warps of its CTA; each term
    two roundings) and FP64 additions of the partials: (3·128 + partials)
    roundings per term covers both with rows per warp below 370."""
    U = 2.0 ** -24
    M, H = xf.shape
    gdy = dyf * gf[None, :]
    S = np.abs(gdy * xf).sum(axis=1)
    dot = (gdy * xf).sum(axis=1)
    c = r ** 3 * dot / H
    exact = r[:, None] * gdy - xf * c[:, None]
    dc = r ** 3 / H * (17 + H / 512) * U * S + U * np.abs(c)
    bound = 2 * (2 * U * np.abs(r[:, None] * gdy) + np.abs(xf) * dc[:, None]
                 + U * np.abs(xf * c[:, None]) + U * np.abs(exact))
    terms = np.abs(dyf * xf * r[:, None]).sum(axis=0)
    chunks = (M + 127) // 128
    return exact, bound, lambda odg: 2 * ((3 * 128 + chunks) * U * terms + U * np.abs(odg))
