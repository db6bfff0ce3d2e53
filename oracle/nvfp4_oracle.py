"""CPU oracle for the FP4 (NVFP4-style) variant of the unified precision flow.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU legs may import it.  It shares no code with the CUDA library
and never calls it.

The pages name FP4 only as future work: the unified precision flow carried to
FP4 or lower precision as hardware support matures, NVIDIA Blackwell given as
the example ([digest] "Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习",
未来方向, item (1)).  They define no FP4 format or granularity, so this variant
takes the plainest reading that keeps the flow's defining property — a token's
forward result does not depend on which batch it is computed in, so rollout and
training see the same numbers ([summary] "Jet-RL: Enabling On-Policy FP8
Reinforcement Learning with Unified Training and Rollout Precision Flow",
Figure 5) — on the FP4 format the Blackwell tensor cores scale in hardware:

* Codes are E2M1: sign, two exponent bits (bias 1), one mantissa bit; the
  magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Encoding rounds to nearest with
  ties to the even code, saturates at ±6, and keeps the sign of zero.
* Every 16 consecutive elements of a row (along the contraction) share one
  E4M3 block scale; every row (a token of X, an output channel of W) has one
  FP32 row scale.  A per-tensor scale would make a token's codes depend on the
  other tokens of its batch, so the second-level scale is per row.
* Row r:  g = RN32(amax_r / 2688)  (2688 = 6·448; amax_r = 0 gives g = 1),
          h = RN32(6·g).
  Block b of the row:  s_b = E4M3(RN32(amax_b / h))  (round to nearest even,
          saturating at 448; a non-negative, "unsigned E4M3" scale),
          d_b = RN32(dec(s_b)·g).
  Element:  q = E2M1(RN32(x / d_b)); when d_b = 0 the code is a zero with the
          sign of x.
  Every operation is one correctly rounded FP32 operation, so the GPU takes
  each decision in the same precision.
* FProp: Y[m,n] = gx[m]·gw[n]·Σ_k dec(qx[m,k])·dec(sx[m,k/16])·dec(qw[n,k])·dec(sw[n,k/16]).
  The oracle sums the products in FP64 (each product has at most 10
  significant bits) and applies the row scales in FP64.

Layouts here are logical: codes int8 [R, K] (values 0..15), block scales uint8
E4M3 codes [R, K/16], row scales float32 [R].  The GPU's packed and blocked
layouts are converted by the tests.
"""
from __future__ import annotations

import numpy as np

from oracle.jetfp8_oracle import e4m3_decode, e4m3_encode

E2M1_MAX = 6.0
BLOCK = 16
ROW_SCALE_DIV = 6.0 * 448.0        # 2688: the row maximum maps to E2M1 6 under E4M3 448

__all__ = ["E2M1_MAX", "BLOCK", "e2m1_decode", "e2m1_encode", "quant_nvfp4_rows", "dequant_nvfp4_rows",
           "gemm_fprop_nvfp4"]

# magnitude of code c (bits 0-2): exponent field e = c >> 1, mantissa bit m = c & 1
_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(codes) -> np.ndarray:
    """FP64 values of E2M1 codes (bit 3 = sign): e = 0 gives m·0.5 (subnormal),
    else (1 + m/2)·2^(e-1)."""
    c = np.asarray(codes).astype(np.int64)
    e, m = (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e - 1.0))
    return np.where(c & 8, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """Round FP values to E2M1 codes: nearest magnitude, ties to the even code
    (mantissa bit 0), saturating at 6; the sign bit follows the sign of v
    (negative zero included)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E2M1_MAX)
    # the code just below (or at) a, and the one above it
    lo = np.searchsorted(_MAGS, a, side="right") - 1
    hi = np.minimum(lo + 1, 7)
    dlo, dhi = a - _MAGS[lo], _MAGS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi != lo) & (lo % 2 == 1))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.int8)


def _f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32)


def quant_nvfp4_rows(x) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantise rows of x (FP32-representable values, [R, K], K % 16 == 0).
    Returns codes int8 [R, K], block scales uint8 E4M3 codes [R, K/16] and row
    scales float32 [R], each step one FP32 rounding as the module header states."""
    x = _f32(x)
    R, K = x.shape
    assert K % BLOCK == 0
    amax_r = np.max(np.abs(x), axis=1) if K else np.zeros(R, np.float32)
    g = np.where(amax_r > 0, amax_r / np.float32(ROW_SCALE_DIV), np.float32(1.0)).astype(np.float32)
    h = (np.float32(6.0) * g).astype(np.float32)
    xb = x.reshape(R, K // BLOCK, BLOCK)
    amax_b = np.max(np.abs(xb), axis=2)
    t = (amax_b / h[:, None]).astype(np.float32)
    s = e4m3_encode(t).astype(np.uint8)
    d = (e4m3_decode(s).astype(np.float32) * g[:, None]).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (xb / d[:, :, None]).astype(np.float32)
    codes = e2m1_encode(quot)
    zero = np.where(np.signbit(xb), 8, 0).astype(np.int8)
    codes = np.where((d == 0)[:, :, None], zero, codes).reshape(R, K)
    return codes, s, g


def dequant_nvfp4_rows(codes, s, g) -> np.ndarray:
    """x̂ = dec(q)·dec(s_b)·g in FP64."""
    R, K = codes.shape
    v = e2m1_decode(codes).reshape(R, K // BLOCK, BLOCK)
    v = v * e4m3_decode(s)[:, :, None] * np.asarray(g, np.float64)[:, None, None]
    return v.reshape(R, K)


def gemm_fprop_nvfp4(xq, sx, gx, wq, sw, gw, rows=None, cols=None) -> np.ndarray:
    """Y = X̂ Ŵᵀ for NVFP4 rows (FP64).  rows / cols select output rows of X and
    output columns (rows of W)."""
    if rows is not None:
        xq, sx, gx = xq[rows], sx[rows], np.asarray(gx)[rows]
    if cols is not None:
        wq, sw, gw = wq[cols], sw[cols], np.asarray(gw)[cols]
    xb = e2m1_decode(xq) * np.repeat(e4m3_decode(sx), BLOCK, axis=1)
    wb = e2m1_decode(wq) * np.repeat(e4m3_decode(sw), BLOCK, axis=1)
    return (xb @ wb.T) * np.asarray(gx, np.float64)[:, None] * np.asarray(gw, np.float64)[None, :]
