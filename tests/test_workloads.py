"""The seeded synthetic inputs follow their stated recipe: reproducible streams,
bf16 values, N(0,1) activations with 0.1 % of entries ×20, W ~ N(0, 0.02²),
∇Y ~ N(0, 1e-3²), γ ~ U(0.5, 1.5), decode activations with per-channel scales
log-uniform in [1, 50]; the device generators (run here on the CPU device) draw
the same distributions; and the layer shapes are the stated ones."""
import numpy as np
import torch

from fp8_mixed_granularity_gb300 import workloads as W


def _is_bf16(t):
    return t.dtype == torch.bfloat16


def test_streams_are_reproducible_and_independent():
    a = W.bf16_values(W.activations(64, 256, seed=3, stream=1))
    b = W.bf16_values(W.activations(64, 256, seed=3, stream=1))
    c = W.bf16_values(W.activations(64, 256, seed=3, stream=2))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_activation_recipe():
    M, K = 512, 1024
    x = W.activations(M, K, seed=0)
    assert _is_bf16(x)
    v = W.bf16_values(x).astype(np.float64)
    # 0.1 % outliers: 20·z lies beyond 6.5 when |z| > 0.325, i.e. for 74.5 % of
    # them; an unscaled N(0,1) value almost never does
    n_out = int(round(1e-3 * M * K))
    assert abs(int((np.abs(v) > 6.5).sum()) - 0.745 * n_out) <= 0.1 * n_out
    core = v[np.abs(v) <= 6.5]
    assert abs(core.mean()) < 0.01 and abs(core.std() - 1.0) < 0.01


def test_weight_gradient_gamma_and_decode_recipes():
    w = W.bf16_values(W.weights(256, 1024, seed=1)).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.0005
    dy = W.bf16_values(W.gradients(256, 1024, seed=2)).astype(np.float64)
    assert abs(dy.std() - 1e-3) < 2.5e-5
    g = W.bf16_values(W.uniform((4096,), 0.5, 1.5, seed=3)).astype(np.float64)
    assert g.min() >= 0.5 and g.max() <= 1.5 and abs(g.mean() - 1.0) < 0.02
    x = W.bf16_values(W.channel_outlier_activations(2048, 512, seed=4)).astype(np.float64)
    c = x.std(axis=0)                                    # ≈ the channel scales
    assert c.min() > 0.8 and c.max() < 60
    assert abs(np.log(c).mean() - 0.5 * np.log(50.0)) < 0.2   # log-uniform in [1, 50]


def test_device_generators_match_the_recipe():
    dev = torch.device("cpu")
    x = W.device_activations(512, 1024, dev, seed=5)
    assert _is_bf16(x)
    v = x.float().numpy().astype(np.float64)
    n_out = int(round(1e-3 * v.size))
    assert abs(int((np.abs(v) > 6.5).sum()) - 0.745 * n_out) <= 0.1 * n_out
    assert torch.equal(x, W.device_activations(512, 1024, dev, seed=5))
    w = W.device_normal((256, 1024), 0.02, dev, seed=6).float().numpy()
    assert abs(w.std() - 0.02) < 0.0005
    g = W.device_uniform((4096,), 0.5, 1.5, dev, seed=7).float().numpy()
    assert g.min() >= 0.5 and g.max() <= 1.5


def test_layer_shapes():
    llama = {l.name: (l.M, l.K, l.N) for l in W.llama8b_training()}
    assert llama == {"qkv": (8192, 4096, 6144), "o": (8192, 4096, 4096),
                     "gate_up": (8192, 4096, 28672), "down": (8192, 14336, 4096)}
    d32 = {l.name: (l.M, l.K, l.N) for l in W.dense32b_training()}
    assert d32 == {"qkv": (16384, 5120, 7168), "o": (16384, 5120, 5120),
                   "gate_up": (16384, 5120, 51200), "down": (16384, 25600, 5120)}
    dec = {l.name: (l.K, l.N) for l in W.qwen3_8b_decode(64)}
    assert dec == {"qkv": (4096, 6144), "o": (4096, 4096), "gate_up": (4096, 24576), "down": (12288, 4096)}
    # Llama-3.1-8B layer step: F1 + F2 + F3 of the four linears
    assert sum(3 * l.gemm_flops for l in W.llama8b_training()) == 3 * 2 * 8192 * (
        4096 * 6144 + 4096 * 4096 + 4096 * 28672 + 14336 * 4096)
