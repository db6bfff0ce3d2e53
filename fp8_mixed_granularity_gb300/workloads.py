"""Seeded synthetic workloads for the mixed-granularity FP8 linear layer.

This module only draws random numbers and rounds them to bfloat16; it holds
none of the quantisation or GEMM arithmetic, so both the CUDA path and the CPU
oracle can be fed from it.

The value distributions stand in for the activations, weights and gradients of
the Llama-3.1-8B / Qwen3-8B / 32B-class models that the Jet-RL pages train
("Jet-RL：通过统一训练与推理精度流实现 On-Policy FP8 强化学习", 实验结果): no weights or
datasets are used.

  activations  X  ~ N(0, 1), 0.1 % of entries (uniform, without replacement) ×20
  decode X        ~ N(0, 1)·c_k, c_k log-uniform in [1, 50] per input channel
  weights      W  ~ N(0, 0.02²)
  gradients    ∇Y ~ N(0, 1e-3²)
  RMSNorm γ       ~ U(0.5, 1.5)
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

# ---------------------------------------------------------------------------
# Workload shapes
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class Linear:
    """One linear layer Y[M,N] = X[M,K]·W[N,K]ᵀ."""
    name: str
    M: int
    K: int
    N: int

    @property
    def gemm_flops(self) -> int:
        """2·M·N·K for one of FProp, DGrad or WGrad."""
        return 2 * self.M * self.N * self.K


def single_linear_small() -> list[Linear]:
    """Single linear layer, X [256,512], W [384,512], ∇Y [256,384]."""
    return [Linear("single", 256, 512, 384)]


def llama8b_training(M: int = 8192) -> list[Linear]:
    """Llama-3.1-8B layer linears at M training tokens (hidden 4096,
    intermediate 14336, 32 query + 8 KV heads of 128 → QKV N = 6144)."""
    return [Linear("qkv", M, 4096, 6144), Linear("o", M, 4096, 4096),
            Linear("gate_up", M, 4096, 2 * 14336), Linear("down", M, 14336, 4096)]


def qwen3_8b_decode(M: int) -> list[Linear]:
    """Qwen3-8B decode-shaped FProp (hidden 4096, intermediate 12288)."""
    return [Linear("qkv", M, 4096, 6144), Linear("o", M, 4096, 4096),
            Linear("gate_up", M, 4096, 2 * 12288), Linear("down", M, 12288, 4096)]


def dense32b_training(M: int = 16384) -> list[Linear]:
    """32B-class layer linears at M training tokens (hidden 5120,
    intermediate 25600, QKV N = 7168)."""
    return [Linear("qkv", M, 5120, 7168), Linear("o", M, 5120, 5120),
            Linear("gate_up", M, 5120, 2 * 25600), Linear("down", M, 25600, 5120)]


# ---------------------------------------------------------------------------
# Generators
# ---------------------------------------------------------------------------


def _rng(seed: int, stream: int) -> np.random.Generator:
    """Independent PCG64 stream `stream` of seed `seed`."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy -> bfloat16 torch (CPU), round to nearest even."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_values(t: torch.Tensor) -> np.ndarray:
    """bfloat16 torch tensor -> float32 numpy holding the same values."""
    return t.detach().to("cpu", torch.float32).numpy()


def activations(M: int, K: int, seed: int = 0, stream: int = 0,
                outlier_frac: float = 1e-3, outlier_mult: float = 20.0) -> torch.Tensor:
    """X ~ N(0,1) with a fraction of entries multiplied by `outlier_mult`."""
    g = _rng(seed, stream)
    x = g.standard_normal((M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * M * K))
    if n_out:
        idx = g.choice(M * K, size=n_out, replace=False)
        x.reshape(-1)[idx] *= np.float32(outlier_mult)
    return to_bf16(x)


def channel_outlier_activations(M: int, K: int, seed: int = 0, stream: int = 0,
                                lo: float = 1.0, hi: float = 50.0) -> torch.Tensor:
    """X ~ N(0,1)·c_k with c_k log-uniform in [lo, hi] per input channel k."""
    g = _rng(seed, stream)
    c = np.exp(g.uniform(np.log(lo), np.log(hi), size=K)).astype(np.float32)
    x = g.standard_normal((M, K), dtype=np.float32) * c[None, :]
    return to_bf16(x)


def normal(shape, std: float, seed: int = 0, stream: int = 0) -> torch.Tensor:
    """N(0, std²) in bfloat16."""
    g = _rng(seed, stream)
    return to_bf16(g.standard_normal(shape, dtype=np.float32) * np.float32(std))


def uniform(shape, lo: float, hi: float, seed: int = 0, stream: int = 0) -> torch.Tensor:
    """U(lo, hi) in bfloat16."""
    g = _rng(seed, stream)
    return to_bf16(g.uniform(lo, hi, size=shape).astype(np.float32))


def weights(N: int, K: int, seed: int = 0, stream: int = 1) -> torch.Tensor:
    return normal((N, K), 0.02, seed, stream)


def gradients(M: int, N: int, seed: int = 0, stream: int = 2) -> torch.Tensor:
    return normal((M, N), 1e-3, seed, stream)


# Device-side generators for the large benchmark workloads, where drawing
# hundreds of millions of normals on the host would dominate start-up.  Same
# distributions, seeded torch generator on the device.
def device_activations(M: int, K: int, device, seed: int = 0,
                       outlier_frac: float = 1e-3, outlier_mult: float = 20.0) -> torch.Tensor:
    gen = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn(M, K, device=device, generator=gen, dtype=torch.float32)
    n_out = int(round(outlier_frac * M * K))
    if n_out:
        idx = torch.randperm(M * K, device=device, generator=gen)[:n_out]
        x.view(-1)[idx] *= outlier_mult
    return x.to(torch.bfloat16)


def device_normal(shape, std: float, device, seed: int = 0) -> torch.Tensor:
    gen = torch.Generator(device=device).manual_seed(seed)
    return (torch.randn(*shape, device=device, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)


def device_uniform(shape, lo: float, hi: float, device, seed: int = 0) -> torch.Tensor:
    gen = torch.Generator(device=device).manual_seed(seed)
    return (torch.rand(*shape, device=device, generator=gen, dtype=torch.float32) * (hi - lo) + lo).to(torch.bfloat16)


def device_channel_outlier_activations(M: int, K: int, device, seed: int = 0,
                                       lo: float = 1.0, hi: float = 50.0) -> torch.Tensor:
    """X ~ N(0,1)·c_k, c_k log-uniform in [lo, hi] per input channel k, drawn on the device."""
    gen = torch.Generator(device=device).manual_seed(seed)
    c = torch.exp(torch.rand(K, device=device, generator=gen, dtype=torch.float32)
                  * (np.log(hi) - np.log(lo)) + np.log(lo))
    x = torch.randn(M, K, device=device, generator=gen, dtype=torch.float32) * c[None, :]
    return x.to(torch.bfloat16)
