"""The CTA-pair GEMM kernel (tcgen05 cta_group::2: a 256 × 256 tile over two
SMs), through the C ABI.  Every output element's arithmetic is the same as on
the single-CTA kernel — its 128-deep MMA blocks and their promotion in
increasing block order — so the two kernels' outputs must be identical bit
for bit; and the pair kernel's output must stay within the GEMM tolerance of
the FP64 oracle, including ragged row counts where the second CTA of a pair
has no rows at all."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from oracle import jetfp8_oracle as O
from tests.gpu_util import check_errors, gemm_tol_ok, h, q_act, q_grad, q_weight, requant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    yield d
    J.jetfp8_test_set_gemm_path(0)


def _run(path, fn):
    J.jetfp8_test_set_gemm_path(path)
    try:
        out = fn()
        check_errors()
        return out
    finally:
        J.jetfp8_test_set_gemm_path(0)


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                       b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 512, 512), (512, 1024, 2048), (1000, 768, 1152)])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_fprop_pair_equals_single_and_oracle(dev, M, N, K, out):
    x = W.activations(M, K, seed=3, stream=M)
    w = W.weights(N, K, seed=3, stream=N)
    xq, sx = q_act(x, dev)
    wq, sw, _ = q_weight(w, dev, with_t=False)

    def fprop():
        y = torch.empty(M, N, dtype=out, device=dev)
        J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
        return y
    y1, y2 = _run(1, fprop), _run(2, fprop)
    assert _same_bits(y1, y2), "pair and single-CTA FProp differ"
    ok, worst = gemm_tol_ok(h(y2.float()), O.gemm_fprop(h(xq), h(sx)[:, :M], h(wq), h(sw)))
    assert ok, f"fprop (pair): worst |Δ|/bound = {worst:.3g}"


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (384, 640, 768)])
def test_dgrad_pair_equals_single_and_oracle(dev, M, N, K):
    w = W.weights(N, K, seed=4)
    dy = W.gradients(M, N, seed=4)
    wq, sw, wqT = q_weight(w, dev)
    dq, ds, _, _ = q_grad(dy, dev, with_col=False)

    def dgrad():
        dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        J.jetfp8_gemm_dgrad(dq, ds, wqT, sw, dx)
        return dx
    d1, d2 = _run(1, dgrad), _run(2, dgrad)
    assert _same_bits(d1, d2), "pair and single-CTA DGrad differ"
    ok, worst = gemm_tol_ok(h(d2.float()), O.gemm_dgrad(h(dq), h(ds)[:, :M], h(wqT), h(sw)))
    assert ok, f"dgrad (pair): worst |Δ|/bound = {worst:.3g}"


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (512, 640, 256), (384, 1280, 1024)])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_wgrad_pair_equals_single_and_oracle(dev, M, N, K, out):
    x = W.activations(M, K, seed=5)
    dy = W.gradients(M, N, seed=5)
    xq, sx = q_act(x, dev)
    xqT, sxT = requant(xq, sx, dev)
    _, _, dqT, dsT = q_grad(dy, dev)

    def wgrad():
        dw = torch.empty(N, K, dtype=out, device=dev)
        J.jetfp8_gemm_wgrad(dqT, dsT, xqT, sxT, dw)
        return dw
    w1, w2 = _run(1, wgrad), _run(2, wgrad)
    assert _same_bits(w1, w2), "pair and single-CTA WGrad differ"
    ok, worst = gemm_tol_ok(h(w2.float()), O.gemm_wgrad(h(dqT), h(dsT), h(xqT), h(sxT)))
    assert ok, f"wgrad (pair): worst |Δ|/bound = {worst:.3g}"


def test_grouped_wgrad_pair_equals_single(dev):
    """Four WGrads of one token count in one grouped launch, on either kernel."""
    M = 512
    shapes = [(384, 256), (256, 768), (1024, 256), (256, 1280)]
    probs = []
    for i, (N, K) in enumerate(shapes):
        x = W.device_activations(M, K, dev, seed=20 + i)
        dy = W.device_normal((M, N), 1e-3, dev, seed=30 + i)
        xq, sx = q_act(x, dev)
        xqT, sxT = requant(xq, sx, dev)
        _, _, dqT, dsT = q_grad(dy, dev)
        probs.append((dqT, dsT, xqT, sxT))

    def grouped():
        outs = [torch.empty(p[0].shape[0], p[2].shape[0], dtype=torch.bfloat16, device=dev) for p in probs]
        J.jetfp8_gemm_wgrad_grouped([(*p, o) for p, o in zip(probs, outs)])
        return outs
    o1, o2 = _run(1, grouped), _run(2, grouped)
    for a, b in zip(o1, o2):
        assert _same_bits(a, b), "pair and single-CTA grouped WGrad differ"


def test_gemm_path_knob_validation(dev):
    lib = J.load_library()
    assert lib.jetfp8_test_set_gemm_path(3) == 1
    assert lib.jetfp8_test_set_gemm_path(-1) == 1
    assert lib.jetfp8_test_set_gemm_path(0) == 0
