"""The grouped WGrad (several linears' F3 in one persistent launch), through
the C ABI: every problem's output must equal its own jetfp8_gemm_wgrad call
bit for bit, whatever the other problems in the group, and stay within the
GEMM tolerance of the FP64 oracle."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from fp8_mixed_granularity_gb300.decoder_layer import llama8b
from oracle import jetfp8_oracle as O
from tests.gpu_util import check_errors, gemm_tol_ok, h, q_act, q_grad, requant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _operands(dev, M, N, K, seed):
    """(dyqT, sdyT, xqT, sxT) of one linear: Q4's column output and Q3's output."""
    x = W.device_activations(M, K, dev, seed=seed)
    dy = W.device_normal((M, N), 1e-3, dev, seed=seed + 1)
    xq, sx = q_act(x, dev)
    xqT, sxT = requant(xq, sx, dev)
    _, _, dyqT, sdyT = q_grad(dy, dev)
    return dyqT, sdyT, xqT, sxT


def _separate(ops, out_dtype, dev):
    outs = []
    for dyqT, sdyT, xqT, sxT in ops:
        dw = torch.empty(dyqT.shape[0], xqT.shape[0], dtype=out_dtype, device=dev)
        J.jetfp8_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw)
        outs.append(dw)
    check_errors()
    return outs


def _grouped(ops, out_dtype, dev):
    outs = [torch.full((o[0].shape[0], o[2].shape[0]), float("nan"), dtype=out_dtype, device=dev)
            for o in ops]
    J.jetfp8_gemm_wgrad_grouped([(*o, dw) for o, dw in zip(ops, outs)])
    check_errors()
    return outs


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_grouped_wgrad_llama_layer_equals_separate(dev, out_dtype):
    """The four WGrads of a Llama-3.1-8B layer (QKV, O, gate/up, down) at 256
    tokens: 6656 output tiles, so every CTA crosses problem boundaries."""
    M = 256
    ops = [_operands(dev, M, N, K, seed=10 * i) for i, (_, _, N, K) in enumerate(llama8b().linears(M))]
    ref = _separate(ops, out_dtype, dev)
    got = _grouped(ops, out_dtype, dev)
    for i, (a, b) in enumerate(zip(got, ref)):
        assert torch.equal(a.view(torch.int8 if out_dtype == torch.bfloat16 else torch.int32),
                           b.view(torch.int8 if out_dtype == torch.bfloat16 else torch.int32)), f"problem {i}"


def test_grouped_wgrad_narrow_tiles_odd_blocks_and_oracle(dev):
    """An output width that is not a multiple of 256 puts the whole group on
    128-wide tiles (the separate calls of the other problems run on 256-wide
    ones); 3 token blocks; then each problem against the oracle."""
    M = 384
    shapes = [(384, 384), (256, 512), (128, 128)]
    ops = [_operands(dev, M, N, K, seed=50 + i) for i, (N, K) in enumerate(shapes)]
    ref = _separate(ops, torch.float32, dev)
    got = _grouped(ops, torch.float32, dev)
    for i, (a, b) in enumerate(zip(got, ref)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"problem {i}"
    for (dyqT, sdyT, xqT, sxT), dw in zip(ops, got):
        ok, worst = gemm_tol_ok(h(dw), O.gemm_wgrad(h(dyqT), h(sdyT), h(xqT), h(sxT)))
        assert ok, f"worst |Δ|/bound = {worst:.3g}"
    # a group of one is the plain call
    one = _grouped(ops[1:2], torch.float32, dev)[0]
    assert torch.equal(one.view(torch.int32), ref[1].view(torch.int32))


def test_grouped_wgrad_many_tiles_odd_block_count(dev):
    """Two problems with 192 + 128 output tiles (more than the SMs) and five
    128-token blocks each: the scale-ring slots wrap at odd places inside tiles,
    between tiles and between problems; the grouped launch equals the single
    launches bit for bit."""
    M = 640
    shapes = [(6144, 1024), (4096, 1024)]
    ops = [_operands(dev, M, N, K, seed=70 + i) for i, (N, K) in enumerate(shapes)]
    ref = _separate(ops, torch.float32, dev)
    got = _grouped(ops, torch.float32, dev)
    for i, (a, b) in enumerate(zip(got, ref)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"problem {i}"


def test_grouped_wgrad_rejects_mixed_token_counts(dev):
    a = _operands(dev, 128, 128, 128, seed=70)
    b = _operands(dev, 256, 128, 128, seed=71)
    dws = [torch.empty(128, 128, dtype=torch.float32, device=dev) for _ in range(2)]
    with pytest.raises(J.JetFP8Error):
        J.jetfp8_gemm_wgrad_grouped([(*a, dws[0]), (*b, dws[1])])
