"""Pins of the oracle RMSNorm+quant and SwiGLU support steps: closed forms on
constant rows, torch's float64 functional ops as an independent check, and
the quantiser identity on the normalised output."""
import numpy as np
import pytest
import torch

from oracle import jetfp8_oracle as O


def test_rmsnorm_constant_rows_closed_form():
    H = 256
    x = np.zeros((3, H), np.float32)
    x[0, :] = 2.0
    x[1, :] = -0.5
    x[2, ::2] = 3.0; x[2, 1::2] = -3.0
    gamma = np.ones(H, np.float32)
    y, rstd, q, s = O.rmsnorm_quant(x, gamma, 0.0)
    assert rstd[0] == 0.5 and rstd[1] == 2.0 and rstd[2] == pytest.approx(1 / 3, rel=1e-15)
    assert np.all(y[0] == 1.0) and np.all(y[1] == -1.0)
    assert np.all(np.abs(y[2]) == 1.0)
    # y = ±1 in every group: amax 1, S = fp32(1/448), codes ±448
    assert np.all(s == np.float32(1.0) / np.float32(448.0))
    assert np.all((q & 0x7F) == 0x7E)


def test_rmsnorm_matches_torch_float64():
    g = np.random.default_rng(15)
    x = g.standard_normal((16, 512)).astype(np.float32)
    gamma = g.uniform(0.5, 1.5, 512).astype(np.float32)
    eps = 1e-6
    y, rstd, q, s = O.rmsnorm_quant(x, gamma, eps)
    xt = torch.from_numpy(x).double()
    ref = torch.nn.functional.rms_norm(xt, (512,), weight=torch.from_numpy(gamma).double(),
                                       eps=float(np.float32(eps))).numpy()
    # within one bf16 rounding of the float64 result
    assert np.all(np.abs(y - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
    ref_rstd = 1.0 / np.sqrt((x.astype(np.float64) ** 2).mean(axis=1) + float(np.float32(eps)))
    assert np.allclose(rstd, ref_rstd, rtol=1e-15)
    q2, s2 = O.quant_rowgroups(y.astype(np.float32))
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_swiglu_matches_torch_float64():
    g = np.random.default_rng(16)
    gu = (g.standard_normal((8, 512)) * 2).astype(np.float32)
    h, q, s = O.swiglu_quant(gu)
    t = torch.from_numpy(gu).double()
    ref = (torch.nn.functional.silu(t[:, :256]) * t[:, 256:]).numpy()
    assert np.all(np.abs(h - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-300)
    dh = g.standard_normal((8, 256)).astype(np.float32)
    d = O.swiglu_bwd(gu, dh)
    tg = t.clone().requires_grad_(True)
    out = torch.nn.functional.silu(tg[:, :256]) * tg[:, 256:]
    out.backward(torch.from_numpy(dh).double())
    refd = tg.grad.numpy()
    assert np.all(np.abs(d - refd) <= np.abs(refd) * 2.0 ** -8 + 1e-300)
