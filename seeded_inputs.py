"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds none of the method's arithmetic: it only draws random
numbers and rounds activations to bf16 (the input dtype).  Quantization,
GEMM and scaling live in the CUDA library (product) and in ``oracle/``
(checker), each written separately.

Recipe (the pages benchmark Qwen3 models on ShareGPT traffic; these synthetic
tensors stand in for that data, with the linear-layer shapes of the models):
  * activations A[M, K] ~ N(0, 1), drawn in fp32 by numpy PCG64(seed), rounded
    to bf16 (round-to-nearest-even, by torch); optionally 1% of the entries,
    chosen uniformly by the same generator, are multiplied by 20 (outliers);
  * weights W[N, K] ~ N(0, 0.02) in fp32, numpy PCG64(seed + 1).
Large bench weights are drawn on the device by a seeded torch generator with
the same distribution (speed only; the parity tests use the numpy recipe).
"""
from __future__ import annotations

import numpy as np
import torch

# Linear-layer shapes (K = in_features, N = out_features) of the Qwen3 models
# the pages evaluate; qkv is the fused q/k/v projection, gate_up the fused
# gate/up projection of the MLP.
QWEN3_LINEARS = {
    "Qwen3-1.7B": {"qkv": (2048, 4096), "o": (2048, 2048), "gate_up": (2048, 12288), "down": (6144, 2048)},
    "Qwen3-8B": {"qkv": (4096, 6144), "o": (4096, 4096), "gate_up": (4096, 24576), "down": (12288, 4096)},
    "Qwen3-32B": {"qkv": (5120, 10240), "o": (8192, 5120), "gate_up": (5120, 51200), "down": (25600, 5120)},
}

# Token counts the pages tune the decode kernels for (max size 32).
TUNED_M = (1, 2, 4, 8, 16, 24, 32)


def activations(M: int, K: int, seed: int = 0, outliers: bool = False) -> torch.Tensor:
    """A[M, K] bf16 on the CPU, ~N(0,1), optionally with 1% x20 outliers."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, K), dtype=np.float32)
    if outliers:
        mask = rng.random((M, K)) < 0.01
        a = np.where(mask, a * np.float32(20.0), a).astype(np.float32)
    return torch.from_numpy(a).to(torch.bfloat16)


def weights(N: int, K: int, seed: int = 0, std: float = 0.02) -> np.ndarray:
    """W[N, K] fp32 on the CPU, ~N(0, std)."""
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    return (rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)).astype(np.float32)


def weights_device(N: int, K: int, seed: int, device, std: float = 0.02) -> torch.Tensor:
    """W[N, K] fp32 drawn on ``device`` by a seeded torch generator."""
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * (seed + 1))
    return torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * std


def activations_device(M: int, K: int, seed: int, device, outliers: bool = False) -> torch.Tensor:
    """A[M, K] bf16 drawn on ``device`` by a seeded torch generator."""
    g = torch.Generator(device=device)
    g.manual_seed(7_000_001 * (seed + 1))
    a = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outliers:
        mask = torch.rand((M, K), generator=g, device=device) < 0.01
        a = torch.where(mask, a * 20.0, a)
    return a.to(torch.bfloat16)


def bf16_to_f32_numpy(a: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16 tensor to a float32 numpy array."""
    return a.detach().to("cpu").to(torch.float32).numpy()
