"""Seeded synthetic inputs for the sharded-matmul workloads.

This module is shared by the CUDA path's tests/benchmark and by the CPU
oracle.  It holds none of the method's arithmetic: it only draws random
numbers and rounds them to the stored input type (torch's own fp32 ->
bfloat16 conversion), so both sides see bit-identical inputs.

Every generator uses a CPU ``torch.Generator`` seeded explicitly and draws
its tensors in a fixed order (A first, then B; X, W1, W2 for the MLP pair).
"""
from __future__ import annotations

import math
from typing import Dict, Tuple

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randint_matrix(shape: Tuple[int, int], lo: int, hi: int, seed: int = 0,
                   g: torch.Generator = None) -> torch.Tensor:
    """fp32 matrix of integers uniform in [lo, hi] (inclusive)."""
    g = g or _gen(seed)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int64).to(torch.float32)


def normal_matrix(shape: Tuple[int, int], std: float, dtype: str, seed: int = 0,
                  g: torch.Generator = None) -> torch.Tensor:
    """N(0, std^2) entries drawn in fp32, stored in ``dtype``."""
    g = g or _gen(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(DTYPES[dtype])


def uniform_matrix(shape, lo: float, hi: float, dtype: str, seed: int = 0,
                   g: torch.Generator = None) -> torch.Tensor:
    """Entries uniform in [lo, hi) drawn in fp32, stored in ``dtype``."""
    g = g or _gen(seed)
    x = torch.rand(shape, generator=g, dtype=torch.float32)
    x.mul_(hi - lo).add_(lo)
    return x.to(DTYPES[dtype])


# ---- the workloads ------------------------------------------------------

def split_k_integer(I: int = 64, J: int = 64, K: int = 64, seed: int = 0):
    """Integer-valued fp32 A [I,J], B [J,K], entries uniform in [-4, 4]."""
    g = _gen(seed)
    A = randint_matrix((I, J), -4, 4, g=g)
    B = randint_matrix((J, K), -4, 4, g=g)
    return A, B


def scaled_normal_pair(I: int, J: int, K: int, dtype: str = "bf16", seed: int = 0):
    """A [I,J], B [J,K] with entries N(0,1)/sqrt(J), stored in ``dtype``."""
    g = _gen(seed)
    s = 1.0 / math.sqrt(J)
    A = normal_matrix((I, J), s, dtype, g=g)
    B = normal_matrix((J, K), s, dtype, g=g)
    return A, B


def mlp_pair(T: int = 8192, D: int = 4096, F: int = 16384, seed: int = 0, dtype: str = "bf16",
             w_std: float = 0.02):
    """MLP block inputs: activations X [T,D] ~ N(0,1); W1 [D,F] and W2 [F,D]
    ~ N(0, w_std^2) (0.02 read as the standard deviation)."""
    g = _gen(seed)
    X = normal_matrix((T, D), 1.0, dtype, g=g)
    W1 = normal_matrix((D, F), w_std, dtype, g=g)
    W2 = normal_matrix((F, D), w_std, dtype, g=g)
    return X, W1, W2


def partial_buffers(n_ranks: int, numel: int, dtype: str, seed: int = 0):
    """``n_ranks`` partial-sum buffers of ``numel`` entries uniform in [-1, 1)."""
    g = _gen(seed)
    return [uniform_matrix((numel,), -1.0, 1.0, dtype, g=g) for _ in range(n_ranks)]


WORKED_EXAMPLE = (
    torch.tensor([[1.0, 2.0], [3.0, 4.0]]),
    torch.tensor([[5.0, 6.0], [7.0, 8.0]]),
)
