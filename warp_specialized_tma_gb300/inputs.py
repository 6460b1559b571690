"""Seeded synthetic operands for the bf16 GEMM workloads.

This module only draws random numbers and rounds them to bf16; it holds none of
the GEMM's arithmetic.  Both the CUDA path (bench, tests) and the CPU oracle's
callers take their inputs from here, so the two sides always see the same bf16
bit patterns.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws A first,
then B, in fp32 (``rand`` for uniform, ``randn`` for normal, ``randint`` for the
small-integer inputs), scaled to the stated distribution, and each value is
rounded to bf16 by ``Tensor.to(torch.bfloat16)`` (round to nearest even).
Operands are row-major with the contraction index contiguous (K-major): A is
M x lda, B is N x ldb, and columns K..ld-1 hold a large sentinel that no correct
kernel reads.
"""
from __future__ import annotations

import numpy as np
import torch

# The five synthetic workloads: name -> shape, value distribution and seed.
WORKLOADS = {
    "cube256": dict(M=256, N=256, K=256, dist="uniform", seed=1),
    "cube4096": dict(M=4096, N=4096, K=4096, dist="normal", seed=2),
    "cube8192": dict(M=8192, N=8192, K=8192, dist="uniform", seed=3),
    "longk": dict(M=2048, N=2048, K=32768, dist="normal0.1", seed=4),
    "ragged": dict(M=6143, N=5999, K=4104, dist="normal", seed=5),
}

# Nominal standard deviation of each distribution (for tolerance bookkeeping).
NOMINAL_SIGMA = {
    "uniform": 1.0 / np.sqrt(3.0),
    "normal": 1.0,
    "normal0.1": 0.1,
    "int2": np.sqrt(2.0),
    "ones": 1.0,
}

PAD_SENTINEL = 1024.0


def _draw(rows: int, cols: int, dist: str, gen: torch.Generator) -> torch.Tensor:
    shape = (rows, cols)
    if dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
    elif dist == "normal0.1":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * 0.1
    elif dist == "int2":
        x = torch.randint(-2, 3, shape, generator=gen, dtype=torch.int32).to(torch.float32)
    elif dist == "ones":
        x = torch.ones(shape, dtype=torch.float32)
    elif dist == "zeros":
        x = torch.zeros(shape, dtype=torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(torch.bfloat16)


def make_operand(rows: int, K: int, ld: int | None, dist: str,
                 gen: torch.Generator) -> torch.Tensor:
    """A rows x ld bf16 CPU tensor whose first K columns follow ``dist``."""
    ld = K if ld is None else int(ld)
    if ld < K:
        raise ValueError("leading dimension smaller than K")
    vals = _draw(rows, K, dist, gen)
    if ld == K:
        return vals.contiguous()
    out = torch.full((rows, ld), PAD_SENTINEL, dtype=torch.bfloat16)
    out[:, :K] = vals
    return out


def make_problem(M: int, N: int, K: int, dist: str, seed: int,
                 lda: int | None = None, ldb: int | None = None):
    """(A, B) for one GEMM: A is M x lda, B is N x ldb, bf16 on the CPU."""
    gen = torch.Generator()
    gen.manual_seed(int(seed))
    A = make_operand(M, K, lda, dist, gen)
    B = make_operand(N, K, ldb, dist, gen)
    return A, B


def make_workload(name: str, lda: int | None = None, ldb: int | None = None):
    w = WORKLOADS[name]
    return make_problem(w["M"], w["N"], w["K"], w["dist"], w["seed"], lda, ldb)


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 numpy view of a bf16 CPU tensor's bit patterns."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray) -> torch.Tensor:
    """bf16 CPU tensor from uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
