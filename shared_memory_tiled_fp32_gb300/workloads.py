"""Seeded synthetic inputs for the FP32 GEMM workloads.

This module only draws random matrices; it holds none of the product's
arithmetic, so the CUDA path and the CPU oracle can both be fed from it.

Every workload is drawn with a torch CPU ``Generator`` seeded per workload,
A first and then B, so a given name always yields the same bytes:

* ``uniform``: i.i.d. uniform on [-1, 1), as ``2*rand - 1`` (exact in fp32);
* ``int``: i.i.d. integers uniform on {-2, ..., 2}, stored as float32;
* ``normal``: i.i.d. standard normal.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist: str  # "uniform" | "int" | "normal"
    seed: int
    # rows the oracle checks when the whole product is too slow for it
    # (None = every output); drawn without replacement from this seed
    row_sample: int | None = None
    row_seed: int | None = None

    @property
    def flop(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        return 4 * (self.M * self.K + self.K * self.N + self.M * self.N)


# The five GEMM shapes the pages' method is measured on (square, ragged, large
# square, the headline 8192^3 and a long-K case) plus the integer variants.
WORKLOADS = {
    "sq256_uniform": Workload("sq256_uniform", 256, 256, 256, "uniform", 1),
    "sq256_int": Workload("sq256_int", 256, 256, 256, "int", 2),
    "ragged_777x1029x513": Workload("ragged_777x1029x513", 777, 1029, 513, "uniform", 3),
    "sq4096_uniform": Workload("sq4096_uniform", 4096, 4096, 4096, "uniform", 4),
    "sq4096_int": Workload("sq4096_int", 4096, 4096, 4096, "int", 5),
    "sq8192_normal": Workload("sq8192_normal", 8192, 8192, 8192, "normal", 6,
                              row_sample=4096, row_seed=1006),
    "longk_2048x2048x16384_normal": Workload("longk_2048x2048x16384_normal", 2048, 2048, 16384,
                                             "normal", 7),
}


def draw(shape, dist: str, gen: torch.Generator) -> torch.Tensor:
    """One float32 CPU tensor of ``shape`` from distribution ``dist``."""
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32).mul_(2.0).sub_(1.0)
    if dist == "int":
        return torch.randint(-2, 3, shape, generator=gen, dtype=torch.int32).to(torch.float32)
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(M: int, N: int, K: int, dist: str, seed: int):
    """(A, B) as contiguous float32 CPU tensors of shapes (M, K) and (K, N)."""
    gen = torch.Generator().manual_seed(seed)
    A = draw((M, K), dist, gen)
    B = draw((K, N), dist, gen)
    return A, B


def workload_inputs(name: str):
    w = WORKLOADS[name]
    return make_inputs(w.M, w.N, w.K, w.dist, w.seed)


def row_order(w: Workload):
    """A seeded random permutation of the output rows of ``w``."""
    gen = torch.Generator().manual_seed(w.row_seed if w.row_seed is not None else 1000 + w.seed)
    return torch.randperm(w.M, generator=gen)


def sample_rows(w: Workload, count: int | None = None):
    """``count`` distinct output rows (default: the workload's row sample),
    uniformly without replacement, seeded, in ascending order."""
    count = w.row_sample if count is None else count
    if count is None or count >= w.M:
        return torch.arange(w.M, dtype=torch.int64)
    return row_order(w)[:count].sort().values
