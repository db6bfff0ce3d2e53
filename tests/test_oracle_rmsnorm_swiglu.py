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


def _rmsnorm_forward_f64(x, gamma, eps):
    r = 1.0 / np.sqrt((x * x).sum(axis=1) / x.shape[1] + eps)
    return (x * r[:, None]) * gamma[None, :], r


def test_rmsnorm_bwd_matches_central_differences():
    """The oracle's backward (without its final bf16 rounding) against central
    differences of the FP64 forward, L = Σ y·dy, on a tiny problem."""
    rng = np.random.default_rng(3)
    M, H, eps = 3, 8, 1e-6
    x = rng.standard_normal((M, H))
    gamma = rng.uniform(0.5, 1.5, H)
    dy = rng.standard_normal((M, H))
    _, r = _rmsnorm_forward_f64(x, gamma, eps)
    loss = lambda xx, gg: float((_rmsnorm_forward_f64(xx, gg, eps)[0] * dy).sum())  # noqa: E731
    h = 1e-6
    dx_fd = np.zeros_like(x)
    for i in range(M):
        for j in range(H):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            dx_fd[i, j] = (loss(xp, gamma) - loss(xm, gamma)) / (2 * h)
    dg_fd = np.zeros(H)
    for j in range(H):
        gp, gm = gamma.copy(), gamma.copy()
        gp[j] += h
        gm[j] -= h
        dg_fd[j] = (loss(x, gp) - loss(x, gm)) / (2 * h)
    # the formula itself, before the bf16 rounding of dx
    gd = dy * gamma[None, :]
    dot = (gd * x).sum(axis=1)
    dx = r[:, None] * gd - x * (r ** 3 * dot / H)[:, None]
    assert np.allclose(dx, dx_fd, rtol=1e-6, atol=1e-8)
    _, dg = O.rmsnorm_bwd(x, gamma, r, dy)
    assert np.allclose(dg, dg_fd, rtol=1e-6, atol=1e-8)
    dxo, _ = O.rmsnorm_bwd(x, gamma, r, dy)
    assert np.array_equal(dxo, O.bf16_rne(dx))


def test_rmsnorm_bwd_matches_torch_autograd_float64():
    """Against torch autograd in FP64 on the CPU (an independent derivative)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    M, H, eps = 5, 256, 1e-6
    x = rng.standard_normal((M, H))
    gamma = rng.uniform(0.5, 1.5, H)
    dy = rng.standard_normal((M, H)) * 1e-3
    xt = torch.tensor(x, requires_grad=True)
    gt = torch.tensor(gamma, requires_grad=True)
    r = torch.rsqrt((xt * xt).mean(dim=1, keepdim=True) + eps)
    y = (xt * r) * gt
    (y * torch.tensor(dy)).sum().backward()
    dxo, dgo = O.rmsnorm_bwd(x, gamma, r.detach().numpy()[:, 0], dy)
    ref = xt.grad.numpy()
    # dxo is the FP64 formula rounded once to bf16: within one bf16 ulp of autograd
    assert np.all(np.abs(dxo - ref) <= np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8))
    assert np.allclose(dgo, gt.grad.numpy(), rtol=1e-12, atol=1e-15)
