"""Seeded synthetic inputs (no arithmetic of the method itself).

Shapes and distributions follow the workloads the pages describe: decode
projection weights drawn N(0, 0.02) before any quantization, activations
N(0, 1) (bf16), and, for the q4_0 x q8_1 decode layer, an RMS-normalised
activation row a / sqrt(mean(a^2) + 1e-5).  No trained weights or datasets
exist or are needed: only shapes matter for a memory-bound kernel.  Every
generator takes an explicit seed (numpy default_rng) so that the CUDA path,
the oracle and the benchmark see the same bytes.
"""
from __future__ import annotations

import numpy as np
import torch

WEIGHT_SIGMA = 0.02


def weights_f32(N: int, K: int, seed: int, sigma: float = WEIGHT_SIGMA) -> np.ndarray:
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(sigma)
    return w


def activations_f32(M: int, K: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).standard_normal((M, K), dtype=np.float32)


def rms_normalised_f32(M: int, K: int, seed: int, eps: float = 1e-5) -> np.ndarray:
    a = activations_f32(M, K, seed).astype(np.float64)
    return (a / np.sqrt((a * a).mean(axis=1, keepdims=True) + eps)).astype(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even, via torch), returned as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bits -> a torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def u8_tensor(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8)).to(device)
