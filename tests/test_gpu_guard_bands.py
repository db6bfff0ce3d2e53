"""Out-of-bounds writes: every output of every entry point is a view into a
larger device buffer whose bytes before and after the view hold a canary pattern;
after the call (ragged shapes where the operation allows them) the canaries must
be intact.  Stands in for a memory checker, which is not used on these GPUs."""
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from tests.gpu_util import check_errors

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side (a multiple of 256: views stay aligned)
CANARY = 0xA5


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


class Guarded:
    """Allocates guarded outputs and checks their canaries."""

    def __init__(self, dev):
        self.dev = dev
        self.bufs = []

    def __call__(self, shape, dtype):
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        body = (nbytes + 255) // 256 * 256
        raw = torch.full((GUARD + body + GUARD,), CANARY, dtype=torch.uint8, device=self.dev)
        view = raw[GUARD:GUARD + nbytes].view(dtype).view(*shape)
        self.bufs.append((raw, nbytes))
        return view

    def check(self):
        torch.cuda.synchronize()
        for raw, nbytes in self.bufs:
            before = raw[:GUARD]
            after = raw[GUARD + nbytes:]
            assert bool((before == CANARY).all()), "write before the output"
            assert bool((after == CANARY).all()), "write after the output"


def _rowquant(g, M, K):
    return g((M, K), torch.uint8), g(J.scale_shape(M, K), torch.float32)


def test_quantisers_write_only_their_outputs(dev):
    g = Guarded(dev)
    M, K = 200, 384                                   # ragged M
    x = W.device_activations(M, K, dev, seed=1)
    q, s = _rowquant(g, M, K)
    J.jetfp8_quant_act_1x128(x, q, s)
    w = W.device_normal((256, K), 0.02, dev, seed=2)
    wq, ws, wqT = g((256, K), torch.uint8), g((2, K // 128), torch.float32), g((K, 256), torch.uint8)
    J.jetfp8_quant_weight_128x128(w, wq, ws, wqT)
    Mg = 256
    dy = W.device_normal((Mg, K), 1e-3, dev, seed=3)
    dq, ds = _rowquant(g, Mg, K)
    dqT, dsT = _rowquant(g, K, Mg)
    J.jetfp8_quant_grad_dual(dy, dq, ds, dqT, dsT)
    xq = torch.empty(Mg, K, dtype=torch.uint8, device=dev)
    sx = torch.empty(*J.scale_shape(Mg, K), dtype=torch.float32, device=dev)
    J.jetfp8_quant_act_1x128(W.device_activations(Mg, K, dev, seed=4), xq, sx)
    xqT, sxT = _rowquant(g, K, Mg)
    J.jetfp8_requant_rowgrp_to_colgrp(xq, sx, xqT, sxT)
    gamma = W.device_uniform((K,), 0.5, 1.5, dev, seed=5)
    rq, rs = _rowquant(g, M, K)
    rstd, y = g((M,), torch.float32), g((M, K), torch.bfloat16)
    J.jetfp8_rmsnorm_quant(x, gamma, 1e-6, rq, rs, rstd, y)
    gu = W.device_normal((M, 2 * K), 1.0, dev, seed=6)
    hq, hs = _rowquant(g, M, K)
    hb = g((M, K), torch.bfloat16)
    J.jetfp8_swiglu_quant(gu, hq, hs, hb)
    dgu = g((M, 2 * K), torch.bfloat16)
    J.jetfp8_swiglu_bwd(gu, W.device_normal((M, K), 1e-3, dev, seed=7), dgu)
    dx, dgam = g((M, K), torch.bfloat16), g((K,), torch.float32)
    ws_rb = g((J.jetfp8_rmsnorm_bwd_workspace_bytes(M, K),), torch.uint8)
    J.jetfp8_rmsnorm_bwd(x, gamma, rstd, W.device_normal((M, K), 1e-3, dev, seed=8), dx, dgam, ws_rb)
    check_errors()
    g.check()


@pytest.mark.parametrize("M", [200, 1])
def test_gemms_write_only_their_outputs(dev, M):
    """FProp / DGrad on ragged M (the TMA stores clip rows past M), the fused
    quantiser outputs, and WGrad (single and grouped)."""
    g = Guarded(dev)
    N, K = 512, 384
    xq = torch.empty(M, K, dtype=torch.uint8, device=dev)
    sx = torch.empty(*J.scale_shape(M, K), dtype=torch.float32, device=dev)
    J.jetfp8_quant_act_1x128(W.device_activations(M, K, dev, seed=1), xq, sx)
    wq = torch.empty(N, K, dtype=torch.uint8, device=dev)
    sw = torch.empty(N // 128, K // 128, dtype=torch.float32, device=dev)
    wqT = torch.empty(K, N, dtype=torch.uint8, device=dev)
    J.jetfp8_quant_weight_128x128(W.device_normal((N, K), 0.02, dev, seed=2), wq, sw, wqT)
    y = g((M, N), torch.bfloat16)
    J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
    y32 = g((M, N), torch.float32)
    J.jetfp8_gemm_fprop(xq, sx, wq, sw, y32)
    yq, ys = _rowquant(g, M, N)
    yb = g((M, N), torch.bfloat16)
    J.jetfp8_gemm_fprop_quant(xq, sx, wq, sw, yq, ys, yb)
    dyq = torch.empty(M, N, dtype=torch.uint8, device=dev)
    sdy = torch.empty(*J.scale_shape(M, N), dtype=torch.float32, device=dev)
    J.jetfp8_quant_grad_dual(W.device_normal((M, N), 1e-3, dev, seed=3), dyq, sdy, None, None)
    dx = g((M, K), torch.bfloat16)
    J.jetfp8_gemm_dgrad(dyq, sdy, wqT, sw, dx)
    if M % 128 == 0 or M == 200:
        Mw = 256                                      # WGrad contracts over whole 128-token blocks
        dyqT = torch.empty(N, Mw, dtype=torch.uint8, device=dev)
        sdyT = torch.empty(*J.scale_shape(N, Mw), dtype=torch.float32, device=dev)
        J.jetfp8_quant_grad_dual(W.device_normal((Mw, N), 1e-3, dev, seed=4),
                                 torch.empty(Mw, N, dtype=torch.uint8, device=dev),
                                 torch.empty(*J.scale_shape(Mw, N), dtype=torch.float32, device=dev),
                                 dyqT, sdyT)
        xq2 = torch.empty(Mw, K, dtype=torch.uint8, device=dev)
        sx2 = torch.empty(*J.scale_shape(Mw, K), dtype=torch.float32, device=dev)
        J.jetfp8_quant_act_1x128(W.device_activations(Mw, K, dev, seed=5), xq2, sx2)
        xqT = torch.empty(K, Mw, dtype=torch.uint8, device=dev)
        sxT = torch.empty(*J.scale_shape(K, Mw), dtype=torch.float32, device=dev)
        J.jetfp8_requant_rowgrp_to_colgrp(xq2, sx2, xqT, sxT)
        dw = g((N, K), torch.float32)
        J.jetfp8_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw)
        dws = [g((N, K), torch.bfloat16) for _ in range(2)]
        J.jetfp8_gemm_wgrad_grouped([(dyqT, sdyT, xqT, sxT, d) for d in dws])
    check_errors()
    g.check()


@pytest.mark.parametrize("M", [300, 1])
def test_pair_and_fp4_write_only_their_outputs(dev, M):
    """The CTA-pair GEMM kernel (ragged M: the second CTA of a pair may have no
    rows) and the FP4 variant's quantiser (codes, blocked scales with their
    padding rows, row scales) and FProp."""
    g = Guarded(dev)
    N, K = 512, 512
    xq = torch.empty(M, K, dtype=torch.uint8, device=dev)
    sx = torch.empty(*J.scale_shape(M, K), dtype=torch.float32, device=dev)
    J.jetfp8_quant_act_1x128(W.device_activations(M, K, dev, seed=6), xq, sx)
    wq = torch.empty(N, K, dtype=torch.uint8, device=dev)
    sw = torch.empty(N // 128, K // 128, dtype=torch.float32, device=dev)
    J.jetfp8_quant_weight_128x128(W.device_normal((N, K), 0.02, dev, seed=7), wq, sw, None)
    y = g((M, N), torch.bfloat16)
    J.jetfp8_test_set_gemm_path(2)
    try:
        J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
        y32 = g((M, N), torch.float32)
        J.jetfp8_gemm_fprop(xq, sx, wq, sw, y32)
    finally:
        J.jetfp8_test_set_gemm_path(0)
    x4 = W.device_activations(M, K, dev, seed=8)
    xq4 = g((M, K // 2), torch.uint8)
    xsf4 = g((J.jetfp8_nvfp4_scale_bytes(M, K),), torch.uint8)
    gx4 = g((M,), torch.float32)
    J.jetfp8_quant_nvfp4(x4, xq4, xsf4, gx4)
    wq4, wsf4, gw4 = J.empty_nvfp4(N // 2, K, dev)
    J.jetfp8_quant_nvfp4(W.device_normal((N // 2, K), 0.02, dev, seed=9), wq4, wsf4, gw4)
    y4 = g((M, N // 2), torch.bfloat16)
    J.jetfp8_gemm_fprop_nvfp4(xq4, xsf4, gx4, wq4, wsf4, gw4, y4)
    check_errors()
    g.check()
