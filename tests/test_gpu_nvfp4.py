"""FP4 variant of the precision flow (NVFP4-style) on the GPU, through the C
ABI: the row quantiser bit-exact against the oracle (codes, block scales in
the blocked layout, row scales), the block-scaled tcgen05 FProp within the
GEMM bar of the FP64 oracle, and the flow's property that a token's result
does not depend on its batch."""
import numpy as np
import pytest
import torch

from fp8_mixed_granularity_gb300 import jetfp8 as J
from fp8_mixed_granularity_gb300 import workloads as W
from oracle import nvfp4_oracle as O4
from tests.gpu_util import check_errors, gemm_tol_ok, h

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__ as g
    g.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def unpack_codes(qp):
    """uint8 [R, K/2] -> int8 codes [R, K] (element 2i in the low nibble)."""
    qp = np.asarray(qp, np.uint8)
    out = np.empty((qp.shape[0], qp.shape[1] * 2), np.int8)
    out[:, 0::2] = qp & 0xF
    out[:, 1::2] = qp >> 4
    return out


def unblock_scales(sf, R, K):
    """Blocked layout -> uint8 [R, K/16]: byte ((r/128·K/64 + b/4)·32 + r%32)·16 + ((r/32)%4)·4 + b%4."""
    sf = np.asarray(sf, np.uint8)
    r = np.arange(R)[:, None]
    b = np.arange(K // 16)[None, :]
    off = (((r // 128) * (K // 64) + b // 4) * 32 + r % 32) * 16 + ((r // 32) % 4) * 4 + b % 4
    return sf[off]


def quant(x_bf16, dev):
    R, K = x_bf16.shape
    q, sf, g = J.empty_nvfp4(R, K, dev)
    sf.fill_(0x7F)            # NaN codes: every byte must be written
    J.jetfp8_quant_nvfp4(x_bf16.to(dev), q, sf, g)
    check_errors()
    return q, sf, g


def _assert_quant(x_bf16, q, sf, g):
    R, K = x_bf16.shape
    oq, os_, og = O4.quant_nvfp4_rows(W.bf16_values(x_bf16))
    assert np.array_equal(h(g), og), "row scales"
    assert np.array_equal(unblock_scales(h(sf), R, K), os_), "block scales"
    assert np.array_equal(unpack_codes(h(q)), oq), "codes"
    # padding rows of the last atom carry zero scales
    sfh = h(sf)
    rows = (R + 127) // 128 * 128
    if rows > R:
        pad = unblock_scales(sfh, rows, K)[R:]
        assert np.all(pad == 0)


@pytest.mark.parametrize("R,K", [(1, 64), (130, 256), (300, 4096), (64, 14336)])
def test_quant_nvfp4_parity(dev, R, K):
    x = W.activations(R, K, seed=60, stream=K)
    q, sf, g = quant(x, dev)
    _assert_quant(x, q, sf, g)


def test_quant_nvfp4_edge_values(dev):
    """Zero rows and blocks, signed zeros, tiny and huge rows, every bf16
    magnitude class, and values on E2M1 rounding midpoints."""
    R, K = 12, 256
    g = np.random.default_rng(61)
    x = (g.standard_normal((R, K)) * 2.0).astype(np.float32)
    x[0] = 0.0
    x[1, :16] = 0.0
    x[1, 16] = -0.0
    x[2] *= np.float32(1e-38)                    # subnormal bf16 values: tiny row scale
    x[3] = np.float32(3.0e38) * np.sign(x[3])    # near the bf16 maximum
    x[4, :] = -0.0
    x[5, :16] = np.array([0.875, 1.75, 2.625, 3.5, 5.25, 7.0, 10.5, 0.4375, 1.3125, 2.1875, 3.0625,
                          4.375, 6.125, 8.75, -10.5, 0.0], np.float32)      # exact midpoints (hand case)
    x[6] = np.ldexp(1.0, g.integers(-133, 127, K)).astype(np.float32) * np.sign(g.standard_normal(K))
    xb = W.to_bf16(x)
    q, sf, gs = quant(xb, dev)
    _assert_quant(xb, q, sf, gs)


def test_quant_nvfp4_rows_do_not_depend_on_the_batch(dev):
    x = W.activations(700, 1024, seed=62)
    q, sf, g = quant(x, dev)
    sub = x[300:364]
    q1, sf1, g1 = quant(sub, dev)
    assert torch.equal(q[300:364], q1) and torch.equal(g[300:364], g1)
    assert np.array_equal(unblock_scales(h(sf), 700, 1024)[300:364], unblock_scales(h(sf1), 64, 1024))


def _fprop(xq, xsf, gx, wq, wsf, gw, M, N, dev):
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_fprop_nvfp4(xq, xsf, gx, wq, wsf, gw, y)
    check_errors()
    return y


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 512, 1024), (300, 768, 4096), (64, 256, 14336),
                                   (1000, 1280, 512)])
def test_gemm_fprop_nvfp4_parity(dev, M, N, K):
    x = W.activations(M, K, seed=63, stream=M)
    w = W.weights(N, K, seed=64, stream=N)
    xq, xsf, gx = quant(x, dev)
    wq, wsf, gw = quant(w, dev)
    y = _fprop(xq, xsf, gx, wq, wsf, gw, M, N, dev)
    ref = O4.gemm_fprop_nvfp4(unpack_codes(h(xq)), unblock_scales(h(xsf), M, K), h(gx),
                              unpack_codes(h(wq)), unblock_scales(h(wsf), N, K), h(gw))
    ok, worst = gemm_tol_ok(h(y.float()), ref)
    assert ok, f"nvfp4 fprop: worst |Δ|/bound = {worst:.3g}"


def test_gemm_fprop_nvfp4_unit_scales_exact(dev):
    """Codes with unit block scales and unit row scales: every product and
    partial sum is a multiple of 1/4 below 2^24, so the FP32 accumulation is
    exact and the output equals the integer dot product rounded once to bf16."""
    M, N, K = 128, 256, 512
    rng = np.random.default_rng(65)
    xc = rng.integers(0, 16, (M, K))
    wc = rng.integers(0, 16, (N, K))
    pack = lambda c: torch.from_numpy(((c[:, 1::2] << 4) | c[:, 0::2]).astype(np.uint8)).to(dev)
    one_sf = lambda R: torch.full((J.jetfp8_nvfp4_scale_bytes(R, K),), 0x38, dtype=torch.uint8, device=dev)
    ones = lambda R: torch.ones(R, dtype=torch.float32, device=dev)
    y = _fprop(pack(xc), one_sf(M), ones(M), pack(wc), one_sf(N), ones(N), M, N, dev)
    exact = O4.e2m1_decode(xc) @ O4.e2m1_decode(wc).T
    want = W.bf16_values(W.to_bf16(exact.astype(np.float32)))
    assert np.array_equal(h(y.float()), want)


def test_gemm_fprop_nvfp4_decode_rows_equal_training_rows(dev):
    """A decode-sized batch's rows equal the same tokens' rows of a training
    batch bit for bit: quantisation is per row and the GEMM's per-element
    arithmetic does not depend on the other rows."""
    K, N = 1024, 512
    x = W.activations(1024, K, seed=66)
    w = W.weights(N, K, seed=67)
    wq, wsf, gw = quant(w, dev)
    xq, xsf, gx = quant(x, dev)
    y_big = _fprop(xq, xsf, gx, wq, wsf, gw, 1024, N, dev)
    for lo, hi in [(0, 64), (512, 640), (960, 1024)]:
        sq, ssf, sg = quant(x[lo:hi], dev)
        y_small = _fprop(sq, ssf, sg, wq, wsf, gw, hi - lo, N, dev)
        assert torch.equal(y_small, y_big[lo:hi])
