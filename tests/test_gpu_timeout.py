"""The failure path on the GPU, without faulting it: the GEMM's TMA producer is
told to leave one block unloaded, so the tensor core's bounded wait for it runs
out; the kernel must record the timeout (reported as JETFP8_ERR_TIMEOUT by
jetfp8_get_last_device_error), shut down cleanly, and leave the context usable —
the next GEMM is checked against the oracle."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from oracle import jetfp8_oracle as O
from tests.gpu_util import gemm_tol_ok, h, q_act, q_weight

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _fprop_checked(dev, xq, sx, wq, sw, ref):
    y = torch.empty(xq.shape[0], wq.shape[0], dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
    J.jetfp8_get_last_device_error()          # raises on a recorded device error
    ok, worst = gemm_tol_ok(h(y.float()), ref)
    assert ok, f"worst |Δ|/bound = {worst:.3g}"


def test_bounded_wait_runs_out_and_context_survives(dev):
    M, N, K = 256, 512, 1024
    xq, sx = q_act(W.activations(M, K, seed=1), dev)
    wq, sw, _ = q_weight(W.weights(N, K, seed=2), dev, with_t=False)
    ref = O.gemm_fprop(h(xq), h(sx)[:, :M], h(wq), h(sw))
    _fprop_checked(dev, xq, sx, wq, sw, ref)

    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    J.jetfp8_test_gemm_fprop_drop_block(xq, sx, wq, sw, y, drop_kb=3)
    with pytest.raises(J.JetFP8Error, match="TIMEOUT"):
        J.jetfp8_get_last_device_error()
    # the error word was cleared by the report; the context still computes
    J.jetfp8_get_last_device_error()
    _fprop_checked(dev, xq, sx, wq, sw, ref)
    assert np.isfinite(h(sx)).all()
