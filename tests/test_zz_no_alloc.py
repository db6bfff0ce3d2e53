"""The allocation-free RMSNorm backward (the library's fixed 8 MiB scratch)
against the workspace entry point: two consecutive calls on the same inputs
must both equal it bit for bit.  Kept in a file collected last; it also runs
on its own.  The refusal of sizes whose scratch would exceed 8 MiB is checked
on the host, where no device can be reached (tests/test_abi.py)."""
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from tests.gpu_util import check_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.mark.parametrize("M,H", [(1000, 512), (4096, 4096), (1, 128), (300, 8192)])
def test_noalloc_matches_workspace_entry_point(dev, M, H):
    x = W.activations(M, H, seed=12).to(dev)
    gamma = W.uniform((H,), 0.5, 1.5, seed=12, stream=1).to(dev)
    dy = W.normal((M, H), 1e-3, seed=12, stream=2).to(dev)
    q, s = J.empty_rowgroup_quant(M, H, dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    J.jetfp8_rmsnorm_quant(x, gamma, 1e-6, q, s, rstd)
    dx_ref = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    dg_ref = torch.empty(H, dtype=torch.float32, device=dev)
    ws = torch.empty(J.jetfp8_rmsnorm_bwd_workspace_bytes(M, H), dtype=torch.uint8, device=dev)
    J.jetfp8_rmsnorm_bwd(x, gamma, rstd, dy, dx_ref, dg_ref, ws)
    for _ in range(2):
        dx = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=dev)
        dg = torch.full((H,), float("nan"), dtype=torch.float32, device=dev)
        J.jetfp8_rmsnorm_bwd_noalloc(x, gamma, rstd, dy, dx, dg)
        check_errors()
        assert torch.equal(dx, dx_ref) and torch.equal(dg, dg_ref)
