"""CPU oracle for the mixed-granularity E4M3 linear layer.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously-correct
statement of what the GPU path computes.  Only the test-suite, the smoke check
and the benchmark's CPU-baseline leg may import it.  It shares no code with the
CUDA library and never calls it.

Citations name the page and its section:

  [digest]  "Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习"
            (paper.rainbus.top digest of arXiv 2601.14243)
  [summary] "Jet-RL: Enabling On-Policy FP8 Reinforcement Learning with Unified
            Training and Rollout Precision Flow" (sciencestack.ai)

What the pages fix, and the readings taken where they are silent:

* E4M3 has 4 exponent bits, 3 mantissa bits and a largest finite value of
  448 ([digest] 前置知识 › FP8 量化 (E4M3 格式)).  448 as the maximum pins the
  "FN" encoding: exponent bias 7, no infinities, S.1111.111 is NaN.
* Scale S = max|X| / 448 and X̂ = cast(X / S) (same section).  The bracket
  printed around X/S is read as the cast to E4M3 with round-to-nearest-even,
  not a ceiling; the cast saturates to ±448; the sign of zero is kept.
* Scales are FP32.  S is the correctly rounded FP32 quotient amax/448, and
  the element quotient x/S is the correctly rounded FP32 quotient, which is
  then rounded to E4M3.  (Where floating point decides a code, both sides take
  the decision in the kernel's precision, FP32.)  A group whose amax is 0 gets
  S = 1.
* Granularity: 1×128 groups along a row for activations and gradients,
  128×128 blocks for weights ([digest] 前置知识 › Per-group / Per-block 量化粒度;
  方法步骤详情, step 1).
* The saved FP8 activation is dequantised (one FP32 multiply) and requantised
  in 128×1 groups for the weight-gradient GEMM ([digest] 方法步骤详情, step 4;
  技术新颖性).
* GEMMs accumulate each 128-wide contraction block exactly (FP64 holds the sum
  of 128 E4M3 products exactly), scale it by the two FP32 scales and sum the
  blocks in FP64 in increasing block order ([digest] 核心方法: FProp
  (1×128)×(128×128), DGrad reuses it, WGrad (1×128)×(128×1)).
* RMSNorm: r = 1/sqrt(mean(x²)+eps) in FP64, y = bf16_rne((x·r)·γ), then the
  1×128 quantiser on y ([digest] 方法步骤详情, step 5: fused RMSNorm kernel).
* SwiGLU (decoder MLP support): h = bf16_rne(silu(g)·u), silu(g) = g/(1+e^-g),
  computed in FP64; its backward in FP64, rounded once to bf16.  The pages do
  not describe it; it exists because the fused MLP chain needs it.
* RMSNorm backward (decoder-layer support; the pages fuse the forward only):
  the exact derivative of y = (x·r)·γ, r = (mean(x²)+eps)^-1/2, evaluated in
  FP64 with the r the forward saved (FP32), ∇x rounded once to bf16; ∇γ is the
  FP64 sum over rows.

Layouts here are logical: a group-scale array for an [R, C] tensor quantised in
1×128 row groups is float32 [C/128, R] (group index major).  Padding of the
leading dimension is a property of the GPU buffers and is stripped by tests.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0          # [digest] 前置知识 › FP8 量化 (E4M3 格式): Δmax = 448
GROUP = 128               # [digest] 前置知识 › Per-group / Per-block 量化粒度

__all__ = [
    "E4M3_MAX", "GROUP", "e4m3_decode", "e4m3_encode", "bf16_rne",
    "quant_rowgroups", "quant_act_1x128", "quant_weight_128x128",
    "requant_rowgrp_to_colgrp", "quant_grad_dual", "block_scaled_gemm",
    "gemm_fprop", "gemm_dgrad", "gemm_wgrad", "rmsnorm_quant",
    "swiglu_quant", "swiglu_bwd", "rmsnorm_bwd",
]


# ---------------------------------------------------------------------------
# Step 1: E4M3 decode, from the bit fields of the format
# ---------------------------------------------------------------------------
def _decode_one(code: int) -> float:
    """Value of one E4M3FN byte: s|eeee|mmm, bias 7, e=15,m=7 is NaN."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    sign = -1.0 if s else 1.0
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:                                   # subnormal: (m/8)·2^(1-7)
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_DECODE_TABLE = np.array([_decode_one(c) for c in range(256)], dtype=np.float64)
# magnitudes of the 127 non-negative finite codes 0x00..0x7E, strictly increasing
_POS_MAGS = _DECODE_TABLE[:0x7F].copy()


def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3FN bytes to float64 (exact)."""
    return _DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


# ---------------------------------------------------------------------------
# Step 2: E4M3 encode, saturating round-to-nearest-even
# ---------------------------------------------------------------------------
def e4m3_encode(v) -> np.ndarray:
    """Round finite float32 values to E4M3FN codes.

    |v| >= 448 saturates to 448.  Otherwise |v| is rounded to the E4M3 grid of
    its binade (spacing 2^(e-3), with e clamped at -6 for the subnormal range),
    ties to the even multiple; the sign bit of v is kept (so -0 and negative
    values that round to zero give 0x80).
    """
    v = np.asarray(v, dtype=np.float32)
    if np.isnan(v).any() or np.isinf(v).any():
        raise ValueError("e4m3_encode: input must be finite")
    a = np.abs(v.astype(np.float64))
    _, ex = np.frexp(a)                      # a = f·2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)               # floor(log2 a), clamped to the subnormal exponent
    ulp = np.ldexp(1.0, e - 3)
    mag = np.rint(a / ulp) * ulp             # exact: a/ulp is a power-of-two scaling; rint is RNE
    mag = np.where(a >= E4M3_MAX, E4M3_MAX, np.minimum(mag, E4M3_MAX))
    idx = np.searchsorted(_POS_MAGS, mag)
    if not np.array_equal(_POS_MAGS[np.minimum(idx, 0x7E)], mag):
        raise AssertionError("e4m3_encode: rounded magnitude is not an E4M3 value")
    sign = np.signbit(v).astype(np.uint8) << 7
    return (idx.astype(np.uint8) | sign).astype(np.uint8)


def bf16_rne(v) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significant bits), ties
    to even.  Returned as float64 holding the bf16 value.  Normal range only."""
    v = np.asarray(v, dtype=np.float64)
    f, ex = np.frexp(v)                      # f in [0.5, 1)
    return np.ldexp(np.rint(f * 256.0), ex - 8)


# ---------------------------------------------------------------------------
# Step 3: group quantisation
# ---------------------------------------------------------------------------
def _scale_of(amax_f32: np.ndarray) -> np.ndarray:
    """S = amax/448 as a correctly rounded FP32 quotient; S = 1 where amax = 0."""
    s = (amax_f32.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax_f32 == 0, np.float32(1.0), s).astype(np.float32)


def _quant_with_scale(x_f32: np.ndarray, s_f32: np.ndarray) -> np.ndarray:
    """q = E4M3(fp32(x / S)), broadcasting S over its group."""
    return e4m3_encode((x_f32 / s_f32).astype(np.float32))


def quant_rowgroups(x) -> tuple[np.ndarray, np.ndarray]:
    """1×128 quantisation along the last axis of a 2-D float32 array [R, C].

    Returns q uint8 [R, C] and S float32 [C/128, R] (S[g, r] is the scale of
    row r, columns 128g..128g+127)."""
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    if C % GROUP:
        raise ValueError("row length must be a multiple of 128")
    xg = x.reshape(R, C // GROUP, GROUP)
    amax = np.abs(xg).max(axis=2)                     # [R, G], exact
    s = _scale_of(amax)                               # [R, G]
    q = _quant_with_scale(xg, s[:, :, None]).reshape(R, C)
    return q, np.ascontiguousarray(s.T)


def quant_act_1x128(x):
    """Activation quantiser: 1×128 groups along K of X [M, K]
    ([digest] 方法步骤详情, steps 1-2).  Returns (q [M,K], S [K/128, M])."""
    return quant_rowgroups(x)


def quant_weight_128x128(w):
    """Weight quantiser: one scale per 128×128 block of W [N, K]
    ([digest] 方法步骤详情, step 1).  The transposed payload Ŵᵀ used by DGrad
    holds the same codes transposed (step 4: weight quantisation is reused
    between passes, only transposed).

    Returns (q [N,K], S [N/128, K/128], qT [K,N])."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if N % GROUP or K % GROUP:
        raise ValueError("weight dims must be multiples of 128")
    wb = w.reshape(N // GROUP, GROUP, K // GROUP, GROUP)
    amax = np.abs(wb).max(axis=(1, 3))               # [N/128, K/128]
    s = _scale_of(amax)
    q = _quant_with_scale(wb, s[:, None, :, None]).reshape(N, K)
    return q, s, np.ascontiguousarray(q.T)


# ---------------------------------------------------------------------------
# Step 4: requantise the saved activation from 1×128 to 128×1 groups
# ---------------------------------------------------------------------------
def requant_rowgrp_to_colgrp(q, s):
    """q uint8 [M, K] with S float32 [K/128, M] (1×128 row groups) ->
    qT uint8 [K, M] and S' float32 [M/128, K]: the 128×1 column groups of the
    dequantised tensor, written transposed ([digest] 方法步骤详情, step 4).

    Dequantisation is one FP32 multiply dec(q)·S_row (dec(q) is exact in FP32)."""
    q = np.asarray(q, dtype=np.uint8)
    M, K = q.shape
    if M % GROUP or K % GROUP:
        raise ValueError("M and K must be multiples of 128")
    s = np.asarray(s, dtype=np.float32)
    s_full = np.repeat(s.T, GROUP, axis=1)            # [M, K]: scale of each element's row group
    xt = (e4m3_decode(q).astype(np.float32) * s_full).astype(np.float32)
    qT, sT = quant_rowgroups(np.ascontiguousarray(xt.T))   # 1×128 groups of the transpose
    return qT, sT


def quant_grad_dual(dy):
    """Gradient quantiser, ∇Y kept in BF16 and quantised twice from one read
    ([digest] 方法步骤详情, step 4; 前置知识 › Per-group / Per-block 量化粒度):
      (i)  1×128 groups along N, for DGrad: q_row [M,N], S_row [N/128, M];
      (ii) 128×1 groups along M (tokens), transposed, for WGrad:
           qT_col [N,M], S_col [M/128, N]."""
    dy = np.asarray(dy, dtype=np.float32)
    q_row, s_row = quant_rowgroups(dy)
    qT_col, sT_col = quant_rowgroups(np.ascontiguousarray(dy.T))
    return q_row, s_row, qT_col, sT_col


# ---------------------------------------------------------------------------
# Step 5: block-scaled GEMMs
# ---------------------------------------------------------------------------
def block_scaled_gemm(a_q, a_s, b_q, b_scale) -> np.ndarray:
    """out[i, j] = Σ_kb a_s[kb, i] · b_scale(kb)[j] · Σ_{k in kb} dec(a[i,k])·dec(b[j,k]).

    a_q uint8 [R, Kc], a_s float32 [Kc/128, R]; b_q uint8 [C, Kc];
    b_scale(kb) -> float32 [C]: the B-side scale of every output column for
    contraction block kb.  Each block's dot products are exact in FP64; the
    scaled block results are summed in FP64 in increasing kb."""
    a = e4m3_decode(a_q)
    b = e4m3_decode(b_q)
    R, Kc = a.shape
    C, Kc2 = b.shape
    if Kc != Kc2 or Kc % GROUP:
        raise ValueError("contraction lengths differ or are not multiples of 128")
    out = np.zeros((R, C), dtype=np.float64)
    for kb in range(Kc // GROUP):
        sl = slice(kb * GROUP, (kb + 1) * GROUP)
        p = a[:, sl] @ b[:, sl].T                              # exact in FP64
        sa = np.asarray(a_s[kb], dtype=np.float64)[:, None]
        sb = np.asarray(b_scale(kb), dtype=np.float64)[None, :]
        out += (sa * sb) * p
    return out


def gemm_fprop(xq, sx, wq, sw, rows=None, cols=None):
    """FProp Y = X̂·Ŵᵀ with (1×128)×(128×128) scales ([digest] 核心方法;
    方法步骤详情, step 2).  xq [M,K], sx [K/128, M], wq [N,K], sw [N/128, K/128].
    Optional index arrays restrict the output to rows × cols."""
    rows = np.arange(xq.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(wq.shape[0]) if cols is None else np.asarray(cols)
    sw = np.asarray(sw, dtype=np.float32)
    return block_scaled_gemm(xq[rows], np.asarray(sx)[:, rows], wq[cols],
                             lambda kb: sw[cols // GROUP, kb])


def gemm_dgrad(dyq, sdy, wqT, sw, rows=None, cols=None):
    """DGrad ∇X = ∇Ŷ·Ŵ, reusing the (1×128)×(128×128) configuration with the
    transposed weight payload ([digest] 核心方法; 方法步骤详情, step 4).
    dyq [M,N], sdy [N/128, M], wqT [K,N], sw [N/128, K/128] (the forward scales:
    contraction block kb runs over N, the output column k sits in block k/128)."""
    rows = np.arange(dyq.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(wqT.shape[0]) if cols is None else np.asarray(cols)
    sw = np.asarray(sw, dtype=np.float32)
    return block_scaled_gemm(dyq[rows], np.asarray(sdy)[:, rows], wqT[cols],
                             lambda kb: sw[kb, cols // GROUP])


def gemm_wgrad(dyqT, sdyT, xqT, sxT, rows=None, cols=None):
    """WGrad ∇W = ∇Ŷᵀ·X̂ with (1×128)×(128×1) scales: both operands carry one
    scale per 128 tokens, the contraction axis ([digest] 核心方法; 方法步骤详情,
    step 4).  dyqT [N,M], sdyT [M/128, N], xqT [K,M], sxT [M/128, K]."""
    rows = np.arange(dyqT.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(xqT.shape[0]) if cols is None else np.asarray(cols)
    sxT = np.asarray(sxT, dtype=np.float32)
    return block_scaled_gemm(dyqT[rows], np.asarray(sdyT)[:, rows], xqT[cols],
                             lambda kb: sxT[kb, cols])


# ---------------------------------------------------------------------------
# Step 6: RMSNorm fused with the 1×128 quantiser
# ---------------------------------------------------------------------------
def rmsnorm_quant(x, gamma, eps):
    """r = 1/sqrt(Σx²/H + eps) (FP64); y = bf16_rne((x·r)·γ); then 1×128
    quantisation of y ([digest] 方法步骤详情, step 5).

    Returns (y float64 holding bf16 values [M,H], rstd float64 [M],
             q uint8 [M,H], S float32 [H/128, M])."""
    xd = np.asarray(x, dtype=np.float64)
    g = np.asarray(gamma, dtype=np.float64)
    H = xd.shape[1]
    rstd = 1.0 / np.sqrt((xd * xd).sum(axis=1) / H + float(np.float32(eps)))
    y = bf16_rne((xd * rstd[:, None]) * g[None, :])
    q, s = quant_rowgroups(y.astype(np.float32))
    return y, rstd, q, s


# ---------------------------------------------------------------------------
# Step 7: SwiGLU support for the decoder-MLP chain (not on the pages)
# ---------------------------------------------------------------------------
def swiglu_quant(gu):
    """gu [M, 2I] holds gate in columns [0, I) and up in [I, 2I).
    h = bf16_rne(silu(g)·u) with silu(g) = g/(1+e^-g) in FP64, then 1×128
    quantisation of h.  Returns (h float64 of bf16 values [M,I], q, S)."""
    gu = np.asarray(gu, dtype=np.float64)
    I = gu.shape[1] // 2
    g, u = gu[:, :I], gu[:, I:]
    h = bf16_rne(g / (1.0 + np.exp(-g)) * u)
    q, s = quant_rowgroups(h.astype(np.float32))
    return h, q, s


def swiglu_bwd(gu, dh):
    """Backward of h = silu(g)·u: with σ = 1/(1+e^-g),
    ∂h/∂u = g·σ, ∂h/∂g = u·σ·(1 + g·(1-σ)).  FP64, one bf16 rounding.
    Returns d_gu [M, 2I] (float64 of bf16 values): [∇g | ∇u]."""
    gu = np.asarray(gu, dtype=np.float64)
    dh = np.asarray(dh, dtype=np.float64)
    I = gu.shape[1] // 2
    g, u = gu[:, :I], gu[:, I:]
    sig = 1.0 / (1.0 + np.exp(-g))
    dg = dh * u * sig * (1.0 + g * (1.0 - sig))
    du = dh * g * sig
    return bf16_rne(np.concatenate([dg, du], axis=1))


# ---------------------------------------------------------------------------
# Step 8: RMSNorm backward (decoder-layer support, not on the pages)
# ---------------------------------------------------------------------------
def rmsnorm_bwd(x, gamma, rstd, dy):
    """Backward of y = (x·r)·γ with r = 1/sqrt(Σx²/H + eps) per row, given the
    forward's saved r:
        ∂L/∂x_i = r·γ_i·dy_i − x_i·r³·(Σ_j γ_j·dy_j·x_j)/H
        ∂L/∂γ_j = Σ_rows dy_j·x_j·r
    (r depends on x through Σx²: ∂r/∂x_i = −x_i·r³/H).  FP64; ∇x is rounded
    once to bf16, ∇γ is returned in FP64.
    Returns (dx float64 of bf16 values [M, H], dgamma float64 [H])."""
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(gamma, dtype=np.float64)
    r = np.asarray(rstd, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    H = x.shape[1]
    gd = dy * g[None, :]
    dot = (gd * x).sum(axis=1)
    dx = r[:, None] * gd - x * (r ** 3 * dot / H)[:, None]
    dgamma = (dy * x * r[:, None]).sum(axis=0)
    return bf16_rne(dx), dgamma
