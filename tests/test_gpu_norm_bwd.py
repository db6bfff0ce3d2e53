"""GPU parity of the RMSNorm backward (decoder-layer support) against the FP64
oracle, through the C ABI, with the r the GPU forward saved.  Bounds are
derived from the kernel's rounding sequence (all FP32 operations rounded
separately, row sums as 16-term FP32 chunks added in FP32 and combined in FP64,
∇γ as FP32 sums over 128-row chunks added in FP64), with a factor 2 margin."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from oracle import jetfp8_oracle as O
from tests.gpu_util import check_errors, h, rmsnorm_bwd_bounds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _run(dev, x, gamma, dy):
    M, H = x.shape
    xd, gd, dyd = x.to(dev), gamma.to(dev), dy.to(dev)
    q, s = J.empty_rowgroup_quant(M, H, dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    J.jetfp8_rmsnorm_quant(xd, gd, 1e-6, q, s, rstd)
    dx = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    dg = torch.empty(H, dtype=torch.float32, device=dev)
    ws = torch.empty(J.jetfp8_rmsnorm_bwd_workspace_bytes(M, H), dtype=torch.uint8, device=dev)
    J.jetfp8_rmsnorm_bwd(xd, gd, rstd, dyd, dx, dg, ws)
    check_errors()
    return rstd, dx, dg, ws


# rows up to 4096 wide take the fused kernel; wider rows the three-kernel path
@pytest.mark.parametrize("M,H", [(64, 4096), (300, 1024), (1, 128), (1000, 512), (200, 8192), (130, 5120)])
def test_rmsnorm_bwd_parity(dev, M, H):
    x = W.activations(M, H, seed=9)
    gamma = W.uniform((H,), 0.5, 1.5, seed=9, stream=1)
    dy = W.normal((M, H), 1e-3, seed=9, stream=2)
    rstd, dx, dg, _ = _run(dev, x, gamma, dy)
    xf, gf, dyf = (W.bf16_values(t).astype(np.float64) for t in (x, gamma, dy))
    r = h(rstd).astype(np.float64)
    odx, odg = O.rmsnorm_bwd(xf, gf, r, dyf)

    # exact ∇x before rounding, and the FP32 evaluation error bound per element
    exact, bound, dg_bound_of = rmsnorm_bwd_bounds(xf, gf, r, dyf)
    ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 8)
    gdx = h(dx.float()).astype(np.float64)
    assert np.all(np.abs(gdx - exact) <= ulp + bound)
    # where the bound is far below half an ulp, the codes match the oracle's rounding
    sure = bound < ulp / 8
    assert np.mean(gdx[sure] == odx[sure]) > 0.999

    assert np.all(np.abs(h(dg).astype(np.float64) - odg) <= dg_bound_of(odg))


def test_rmsnorm_bwd_is_deterministic(dev):
    M, H = 1000, 512
    x = W.activations(M, H, seed=10)
    gamma = W.uniform((H,), 0.5, 1.5, seed=10, stream=1)
    dy = W.normal((M, H), 1e-3, seed=10, stream=2)
    _, dx1, dg1, _ = _run(dev, x, gamma, dy)
    _, dx2, dg2, _ = _run(dev, x, gamma, dy)
    assert torch.equal(dx1, dx2) and torch.equal(dg1, dg2)


def test_rmsnorm_bwd_rejects_small_workspace(dev):
    M, H = 300, 256
    t = lambda *s, dt=torch.bfloat16: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
    ws = torch.empty(J.jetfp8_rmsnorm_bwd_workspace_bytes(M, H) - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(J.JetFP8Error, match="INVALID_ARG"):
        J.jetfp8_rmsnorm_bwd(t(M, H), t(H), t(M, dt=torch.float32), t(M, H), t(M, H),
                             t(H, dt=torch.float32), ws)
