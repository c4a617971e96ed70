"""Seeded synthetic inputs for FP32 GEMM -- shared by the tests, the bench and the oracle checks.

This module holds no GEMM arithmetic: it only draws matrices.  Every matrix
is generated on the host with a seeded ``torch.Generator`` so that the oracle
and the GPU path see bit-identical inputs (the GPU copy is made from these
host arrays).

Distributions and shapes follow the workloads the pages measure: square
FP32 matrices from 256 to 8192 ("Vectorized Memory Access: Pushing CUDA SGEMM
to 29 TFLOPS on H100", section 6; "cuSgemm", "Benchmark Results"; "Beyond
Kernel 7", the results table at the top) and the long-K / tall-skinny shapes
added to exercise split-K.  Values are i.i.d. uniform on [-1, 1], standard
normal, or integers uniform on {-8, ..., 8}.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

DISTS = ("uniform", "normal", "int8range")


@dataclass(frozen=True)
class Workload:
    """One GEMM problem: shape, value distribution and seed."""
    name: str
    M: int
    N: int
    K: int
    dist: str
    seed: int

    @property
    def flops(self) -> int:
        """Floating-point operations counted as 2*M*N*K (an FFMA counts as two)."""
        return 2 * self.M * self.N * self.K

    @property
    def compulsory_bytes(self) -> int:
        """Bytes that must cross HBM at least once: read A and B, write C."""
        return 4 * (self.M * self.K + self.K * self.N + self.M * self.N)


# The configurations, by what they are.  Seeds are fixed per configuration.
SMALL_256 = Workload("square_256_uniform", 256, 256, 256, "uniform", 1000)
SMALL_256_INT = Workload("square_256_int", 256, 256, 256, "int8range", 1001)
SQUARE_1024 = Workload("square_1024_uniform", 1024, 1024, 1024, "uniform", 1010)
SWEEP = tuple(Workload(f"square_{n}_normal", n, n, n, "normal", 1020 + i)
              for i, n in enumerate((256, 512, 768, 1024, 1536, 2048)))
SQUARE_4096 = Workload("square_4096_uniform", 4096, 4096, 4096, "uniform", 1040)
SQUARE_8192 = Workload("square_8192_normal", 8192, 8192, 8192, "normal", 1050)
LONG_K = Workload("longk_1024x1024x16384_normal", 1024, 1024, 16384, "normal", 1051)
TALL = Workload("tall_16384x1024x4096_normal", 16384, 1024, 4096, "normal", 1052)

ALL = (SMALL_256, SMALL_256_INT, SQUARE_1024, *SWEEP, SQUARE_4096, SQUARE_8192, LONG_K, TALL)
BY_NAME = {w.name: w for w in ALL}


def matrix(rows: int, cols: int, dist: str, seed: int, stream: int = 0) -> torch.Tensor:
    """A (rows x cols) float32 CPU tensor drawn from ``dist`` with a seeded generator.

    ``stream`` separates the matrices of one workload (0 for A, 1 for B).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1000003 + int(stream))
    if dist == "uniform":
        x = torch.rand((rows, cols), generator=g, dtype=torch.float32)
        return x.mul_(2.0).sub_(1.0)
    if dist == "normal":
        return torch.randn((rows, cols), generator=g, dtype=torch.float32)
    if dist == "int8range":
        return torch.randint(-8, 9, (rows, cols), generator=g, dtype=torch.int32).to(torch.float32)
    raise ValueError(f"unknown distribution {dist!r}; expected one of {DISTS}")


def operands(w: Workload) -> tuple[torch.Tensor, torch.Tensor]:
    """Host (CPU) float32 A (M x K) and B (K x N) for workload ``w``."""
    return matrix(w.M, w.K, w.dist, w.seed, 0), matrix(w.K, w.N, w.dist, w.seed, 1)


def sample_indices(M: int, N: int, count: int, seed: int) -> tuple[torch.Tensor, torch.Tensor]:
    """``count`` seeded (row, col) pairs, always including the four corners of C."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7)
    r = torch.randint(0, M, (count,), generator=g, dtype=torch.int64)
    c = torch.randint(0, N, (count,), generator=g, dtype=torch.int64)
    corners_r = torch.tensor([0, 0, M - 1, M - 1], dtype=torch.int64)
    corners_c = torch.tensor([0, N - 1, 0, N - 1], dtype=torch.int64)
    return torch.cat([corners_r, r]), torch.cat([corners_c, c])
