"""GPU parity of the three block-scaled GEMMs against the FP64 oracle,
through the C ABI: |Δ| <= 1e-2·|ref| + 1e-3·rms(ref) per element.

Small and ragged shapes are compared in full; the full-size Llama-3.1-8B
gate/up and down shapes (the launch configuration the benchmark times) are
compared on sampled row and column stripes."""
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
    return d


def _fprop(dev, xq, sx, wq, sw, out_dtype=torch.bfloat16):
    y = torch.empty(xq.shape[0], wq.shape[0], dtype=out_dtype, device=dev)
    J.jetfp8_gemm_fprop(xq, sx, wq, sw, y)
    check_errors()
    return y


def _assert_close(got, ref, what):
    ok, worst = gemm_tol_ok(got, ref)
    assert ok, f"{what}: worst |Δ|/bound = {worst:.3g}"


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (1, 128, 128), (64, 256, 4096),
                                   (200, 640, 384), (1024, 1024, 2048), (130, 2304, 256)])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_fprop_parity(dev, M, N, K, out):
    x = W.activations(M, K, seed=0, stream=11)
    w = W.weights(N, K, seed=0, stream=12)
    xq, sx = q_act(x, dev)
    wq, sw, _ = q_weight(w, dev, with_t=False)
    y = _fprop(dev, xq, sx, wq, sw, out)
    ref = O.gemm_fprop(h(xq), h(sx)[:, :M], h(wq), h(sw))
    _assert_close(h(y.float()), ref, "fprop")


def test_fprop_decode_rows_bit_identical_to_training_batch(dev):
    """The rollout-sized call and the training-sized call see the same quantised
    graph: rows of a small batch equal the same rows of a large batch bit for
    bit (Figure 5 of the Jet-RL summary page: inference graph ⊂ training graph)."""
    M, N, K = 512, 1024, 2048
    x = W.channel_outlier_activations(M, K, seed=1)
    w = W.weights(N, K, seed=1)
    wq, sw, _ = q_weight(w, dev, with_t=False)
    xq, sx = q_act(x, dev)
    y_all = _fprop(dev, xq, sx, wq, sw)
    for lo, hi in [(0, 64), (128, 256), (300, 301)]:
        xq_s, sx_s = q_act(x[lo:hi], dev)
        assert np.array_equal(h(xq_s), h(xq)[lo:hi])
        y_s = _fprop(dev, xq_s, sx_s, wq, sw)
        assert torch.equal(y_s, y_all[lo:hi])


def test_fprop_decode_tiles_bit_identical_to_training_tiles(dev):
    """Decode-sized batches run on narrower output tiles (more SMs streaming the
    weights) than a training batch; every output element must still be the same
    bits, so a token's result does not depend on the batch it was computed in."""
    M, N, K = 8192, 1024, 2048          # 64 × 4 tiles of 128 × 256: the wide tiles
    x = W.normal((M, K), 1.0, seed=2, stream=21)
    w = W.weights(N, K, seed=2, stream=22)
    wq, sw, _ = q_weight(w, dev, with_t=False)
    xq, sx = q_act(x, dev)
    y_all = _fprop(dev, xq, sx, wq, sw)
    # 1, 64, 128 and 192 rows run on 64-wide tiles, 1920 rows (15 × 8 tiles of 128
    # columns in one wave, 15 × 16 of 64 in two) on 128-wide, 2560 rows on 256-wide
    for lo, hi in [(0, 64), (4096, 4224), (8000, 8192), (17, 18), (2048, 3968), (2048, 4608)]:
        xq_s, sx_s = q_act(x[lo:hi], dev)
        y_s = _fprop(dev, xq_s, sx_s, wq, sw)
        assert torch.equal(y_s, y_all[lo:hi]), (lo, hi)
    # decode-shaped parity against the oracle on the narrow tiles (N = 4096 -> 64-wide)
    x = W.activations(64, 512, seed=3, stream=23)
    w = W.weights(4096, 512, seed=3, stream=24)
    xq, sx = q_act(x, dev)
    wq, sw, _ = q_weight(w, dev, with_t=False)
    y = _fprop(dev, xq, sx, wq, sw, torch.float32)
    _assert_close(h(y), O.gemm_fprop(h(xq), h(sx)[:, :64], h(wq), h(sw)), "decode fprop")
    # and a ragged decode batch (100 rows) on 64-wide tiles (N = 6144), bf16 out
    x = W.activations(100, 512, seed=4, stream=25)
    w = W.weights(6144, 512, seed=4, stream=26)
    xq, sx = q_act(x, dev)
    wq, sw, _ = q_weight(w, dev, with_t=False)
    y = _fprop(dev, xq, sx, wq, sw)
    _assert_close(h(y.float()), O.gemm_fprop(h(xq), h(sx)[:, :100], h(wq), h(sw)), "decode fprop 64-wide")


@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (200, 768, 256), (1, 256, 128), (1024, 2048, 1024)])
def test_fprop_quant_fused_equals_separate(dev, M, N, K):
    """The epilogue-fused 1×128 quantiser gives the bf16 output of the plain
    FProp and, bit for bit, the codes and scales of the 1×128 quantiser applied
    to that output (on the GPU and in the oracle)."""
    x = W.activations(M, K, seed=0, stream=41)
    w = W.weights(N, K, seed=0, stream=42)
    xq, sx = q_act(x, dev)
    wq, sw, _ = q_weight(w, dev, with_t=False)
    y = _fprop(dev, xq, sx, wq, sw)
    yq, ys = J.empty_rowgroup_quant(M, N, dev)
    ys.fill_(float("nan"))
    y2 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_fprop_quant(xq, sx, wq, sw, yq, ys, y2)
    check_errors()
    assert torch.equal(y2, y)
    rq, rs = q_act(y, dev)
    assert torch.equal(yq, rq) and torch.equal(ys[:, :M], rs[:, :M])
    oq, os_ = O.quant_rowgroups(h(y.float()).astype(np.float32))
    assert np.array_equal(h(yq), oq) and np.array_equal(h(ys)[:, :M], os_)
    # codes only
    yq3, ys3 = J.empty_rowgroup_quant(M, N, dev)
    J.jetfp8_gemm_fprop_quant(xq, sx, wq, sw, yq3, ys3)
    check_errors()
    assert torch.equal(yq3, yq) and torch.equal(ys3[:, :M], ys[:, :M])


def test_dgrad_quant_fused_equals_separate(dev):
    M, N, K = 200, 384, 512
    dy = W.gradients(M, N, seed=0, stream=43)
    w = W.weights(N, K, seed=0, stream=44)
    dyq, sdy, _, _ = q_grad(dy, dev, with_col=False)
    _, sw, wqT = q_weight(w, dev)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_dgrad(dyq, sdy, wqT, sw, dx)
    dxq, dxs = J.empty_rowgroup_quant(M, K, dev)
    dx2 = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_dgrad_quant(dyq, sdy, wqT, sw, dxq, dxs, dx2)
    check_errors()
    assert torch.equal(dx2, dx)
    rq, rs = q_act(dx, dev)
    assert torch.equal(dxq, rq) and torch.equal(dxs[:, :M], rs[:, :M])


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (1, 256, 128), (200, 384, 640), (1024, 2048, 1024)])
def test_dgrad_parity(dev, M, N, K):
    dy = W.gradients(M, N, seed=2)
    w = W.weights(N, K, seed=2)
    dyq, sdy, _, _ = q_grad(dy, dev, with_col=False)
    wq, sw, wqT = q_weight(w, dev)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_dgrad(dyq, sdy, wqT, sw, dx)
    check_errors()
    ref = O.gemm_dgrad(h(dyq), h(sdy)[:, :M], h(wqT), h(sw))
    _assert_close(h(dx.float()), ref, "dgrad")


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (128, 128, 128), (1024, 640, 1152)])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_wgrad_parity(dev, M, N, K, out):
    x = W.activations(M, K, seed=3)
    dy = W.gradients(M, N, seed=3)
    xq, sx = q_act(x, dev)
    xqT, sxT = requant(xq, sx, dev)
    _, _, dyqT, sdyT = q_grad(dy, dev)
    dw = torch.empty(N, K, dtype=out, device=dev)
    J.jetfp8_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw)
    check_errors()
    ref = O.gemm_wgrad(h(dyqT), h(sdyT), h(xqT), h(sxT))
    _assert_close(h(dw.float()), ref, "wgrad")


def test_gemm_rejects_bad_shapes(dev):
    xq = torch.zeros(64, 100, dtype=torch.uint8, device=dev)
    with pytest.raises(J.JetFP8Error):
        J.jetfp8_gemm_fprop(xq, torch.zeros(1, 64, device=dev), torch.zeros(128, 100, dtype=torch.uint8, device=dev),
                            torch.zeros(1, 1, device=dev), torch.empty(64, 128, dtype=torch.bfloat16, device=dev))


# --------------------------------------------------------------------------
# Full-size, sampled: the Llama-3.1-8B training shapes at M = 8192 and two
# 32B-class shapes at M = 16384
# --------------------------------------------------------------------------
def _stripes(n, rng, k=2, width=128):
    starts = rng.choice(n // width, size=k, replace=False) * width
    return np.concatenate([np.arange(s, s + width) for s in starts])


def test_wgrad_many_tiles_odd_block_count(dev):
    """More output tiles than SMs (48 × 4 = 192, so some CTAs take two) and five
    128-token blocks per tile: the per-block column- and row-scale slots (eight
    of them, taken in block order across the CTA's tiles) wrap inside a tile and
    between tiles at odd places.  Sampled row and column stripes against the
    oracle."""
    M, N, K = 640, 6144, 1024
    rng = np.random.default_rng(17)
    x = W.device_activations(M, K, dev, seed=17)
    dy = W.device_normal((M, N), 1e-3, dev, seed=18)
    xq, sx = q_act(x, dev)
    xqT, sxT = requant(xq, sx, dev)
    _, _, dyqT, sdyT = q_grad(dy, dev)
    dw = torch.empty(N, K, dtype=torch.float32, device=dev)
    J.jetfp8_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw)
    check_errors()
    hdT, hsdT, hxT, hsxT = h(dyqT), h(sdyT), h(xqT), h(sxT)
    n_rows, k_cols = _stripes(N, rng), _stripes(K, rng)
    _assert_close(h(dw[n_rows]), O.gemm_wgrad(hdT, hsdT, hxT, hsxT, rows=n_rows), "wgrad rows")
    _assert_close(h(dw[:, k_cols]), O.gemm_wgrad(hdT, hsdT, hxT, hsxT, cols=k_cols), "wgrad cols")


@pytest.mark.parametrize(
    "lin",
    [l for l in W.llama8b_training() if l.name in ("gate_up", "down")]
    # 32B-class layer at M = 16384: QKV (N = 7168) and down (K = 25600, 200 blocks per output)
    + [l for l in W.dense32b_training() if l.name in ("qkv", "down")],
    ids=lambda l: f"{l.name}_{l.M}x{l.N}x{l.K}")
def test_full_size_linear_sampled(dev, lin):
    M, K, N = lin.M, lin.K, lin.N
    rng = np.random.default_rng(5)
    x = W.device_activations(M, K, dev, seed=1)
    w = W.device_normal((N, K), 0.02, dev, seed=2)
    dy = W.device_normal((M, N), 1e-3, dev, seed=3)
    xq, sx = q_act(x, dev)
    wq, sw, wqT = q_weight(w, dev)
    dyq, sdy, dyqT, sdyT = q_grad(dy, dev)
    xqT, sxT = requant(xq, sx, dev)
    # quantiser parity on sampled row stripes
    rows = _stripes(M, rng)
    oq, os_ = O.quant_act_1x128(h(x[rows].float()))
    assert np.array_equal(h(xq)[rows], oq) and np.array_equal(h(sx)[:, rows], os_)
    # GEMMs on stripes: full rows × sampled columns and sampled rows × full columns
    y = _fprop(dev, xq, sx, wq, sw)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_dgrad(dyq, sdy, wqT, sw, dx)
    dw = torch.empty(N, K, dtype=torch.bfloat16, device=dev)
    J.jetfp8_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw)
    check_errors()
    hx, hsx, hw, hsw, hwT = h(xq), h(sx)[:, :M], h(wq), h(sw), h(wqT)
    hd, hsd, hdT, hsdT, hxT, hsxT = h(dyq), h(sdy)[:, :M], h(dyqT), h(sdyT), h(xqT), h(sxT)
    r_rows, r_cols = _stripes(M, rng), _stripes(N, rng)
    _assert_close(h(y[r_rows].float()), O.gemm_fprop(hx, hsx, hw, hsw, rows=r_rows), "fprop rows")
    _assert_close(h(y[:, r_cols].float()), O.gemm_fprop(hx, hsx, hw, hsw, cols=r_cols), "fprop cols")
    k_cols = _stripes(K, rng)
    _assert_close(h(dx[r_rows].float()), O.gemm_dgrad(hd, hsd, hwT, hsw, rows=r_rows), "dgrad rows")
    _assert_close(h(dx[:, k_cols].float()), O.gemm_dgrad(hd, hsd, hwT, hsw, cols=k_cols), "dgrad cols")
    n_rows = _stripes(N, rng)
    _assert_close(h(dw[n_rows].float()), O.gemm_wgrad(hdT, hsdT, hxT, hsxT, rows=n_rows), "wgrad rows")
    _assert_close(h(dw[:, k_cols].float()), O.gemm_wgrad(hdT, hsdT, hxT, hsxT, cols=k_cols), "wgrad cols")
