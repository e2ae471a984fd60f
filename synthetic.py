"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random matrices; it holds none of the GEMM arithmetic
and is shared by the tests, the smoke check and the benchmark so that the GPU
library and the CPU oracle see identical operands.

Layouts follow the library boundary: A is row-major M x K; B is the K x N
operand stored column-major, i.e. an N x K row-major tensor (``Bnk``).

Distributions (matching the workloads the pages benchmark on; no public
dataset is involved):

``uniform``  i.i.d. uniform[-1, 1]
``normal``   i.i.d. N(0, 1), times ``scale``
``int3``     i.i.d. uniform on the integers {-3, ..., 3}
``binary``   i.i.d. uniform on {0, 1}

Values are drawn in FP32 with a ``torch.Generator`` seeded by ``seed`` on the
requested device and rounded once to the 16-bit type.
"""
from __future__ import annotations

import numpy as np
import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def matrix(rows: int, cols: int, dist: str, seed: int, dtype: str = "bf16",
           device: str = "cpu", scale: float = 1.0) -> torch.Tensor:
    """A ``rows x cols`` contiguous tensor of ``dtype`` ("f16" or "bf16")."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (int(rows), int(cols))
    if dist == "uniform":
        x = torch.rand(shape, generator=g, device=device, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if scale != 1.0:
            x = x * float(scale)
    elif dist == "int3":
        x = torch.randint(-3, 4, shape, generator=g, device=device, dtype=torch.int32).to(torch.float32)
    elif dist == "binary":
        x = torch.randint(0, 2, shape, generator=g, device=device, dtype=torch.int32).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(DTYPES[dtype]).contiguous()


def operands(M: int, N: int, K: int, dist: str, config: int, dtype: str = "bf16",
             device: str = "cpu", scale_a: float = 1.0, scale_b: float = 1.0,
             dist_b: str | None = None):
    """(A [M x K], Bnk [N x K]) with the per-workload seeds 1000+c and 2000+c."""
    A = matrix(M, K, dist, 1000 + config, dtype, device, scale_a)
    B = matrix(N, K, dist_b or dist, 2000 + config, dtype, device, scale_b)
    return A, B


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a 16-bit tensor, as a host numpy array."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# --- workload shape lists -------------------------------------------------

SMALL_SQUARE = 256                                   # FP16 256^3, uniform / integer / binary
SQUARE_SWEEP = (2048, 4096, 8192, 16384)             # BF16 n^3, N(0,1)
GRID_DIMS = (64, 128, 256, 512, 1024, 2048, 4096, 8192, 12288, 16384)
SKINNY = [(m, 14336, 4096) for m in (1, 16, 128, 1024)] + \
         [(m, 4096, 14336) for m in (1, 16, 128, 1024)] + [(1, 128, 4096)]
LARGE_RECT = [(16384, 16384, 8192), (8192, 28672, 8192), (32768, 8192, 4096)]


def grid_triples():
    """All 1000 (M, N, K) triples of the FP16 shape grid, lexicographic order."""
    return [(m, n, k) for m in GRID_DIMS for n in GRID_DIMS for k in GRID_DIMS]


def grid_quick_subset():
    """The seeded 100-triple subset of the shape grid used for quick runs."""
    idx = np.random.default_rng(3).choice(1000, 100, replace=False)
    t = grid_triples()
    return [t[int(i)] for i in idx]


def row_sample(M: int, n: int = 256, seed: int = 5) -> np.ndarray:
    """Sorted seeded sample of output rows for checks on very large C."""
    n = min(n, M)
    return np.sort(np.random.default_rng(seed).choice(M, n, replace=False)).astype(np.int64)
