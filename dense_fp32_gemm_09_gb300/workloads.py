"""Seeded synthetic inputs for the SGEMM workloads.

This module holds no arithmetic of the product itself: it only draws A and B.
Both the CUDA path and the CPU oracle are fed from here, so it imports neither.

Each workload starts a fresh ``torch.Generator('cpu')`` seeded with its seed and
draws A (M x K) first, then B (K x N), as float32:

* uniform[lo, hi):  ``torch.rand(shape) * (hi - lo) + lo``
* standard normal:  ``torch.randn(shape)``

The shapes and distributions stand in for the workloads of the source pages
("기존 작성한 GE_v2 의 regemm 타일드 커널의 1:1 매핑, gemm_tiled_test 작성",
§7: M=N=K=1024 and 2048 with unstated inputs whose printed error magnitudes fit
uniform[0,1)) plus larger, ragged and tall-skinny shapes.
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
    dist: str          # "uniform" or "normal"
    lo: float = 0.0
    hi: float = 1.0
    seed: int = 0

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        return 4 * (self.M * self.K + self.K * self.N + self.M * self.N)


WORKLOADS = {
    w.name: w
    for w in (
        Workload("sgemm_256", 256, 256, 256, "uniform", -1.0, 1.0, seed=0),
        Workload("sgemm_1024", 1024, 1024, 1024, "uniform", 0.0, 1.0, seed=1),
        Workload("sgemm_2048", 2048, 2048, 2048, "uniform", 0.0, 1.0, seed=2),
        Workload("sgemm_4096", 4096, 4096, 4096, "normal", seed=3),
        Workload("sgemm_8192", 8192, 8192, 8192, "normal", seed=3),
        Workload("sgemm_ragged_3001x2047x1999", 3001, 2047, 1999, "uniform", -1.0, 1.0, seed=4),
        Workload("sgemm_tall_16384x64x4096", 16384, 64, 4096, "uniform", -1.0, 1.0, seed=4),
    )
}


def _draw(g: torch.Generator, shape, w: Workload) -> torch.Tensor:
    if w.dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * (w.hi - w.lo) + w.lo
    if w.dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    raise ValueError(f"unknown distribution {w.dist!r}")


def make_inputs(w: Workload | str):
    """(A, B) as contiguous float32 CPU tensors for workload ``w``."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = torch.Generator("cpu")
    g.manual_seed(w.seed)
    A = _draw(g, (w.M, w.K), w)
    B = _draw(g, (w.K, w.N), w)
    return A, B


def random_pair(M: int, N: int, K: int, seed: int, dist: str = "uniform",
                lo: float = -1.0, hi: float = 1.0):
    """(A, B) for an ad-hoc shape, drawn like the named workloads."""
    w = Workload("adhoc", M, N, K, dist, lo, hi, seed)
    return make_inputs(w)


def small_int_pair(M: int, N: int, K: int, seed: int, lim: int = 8):
    """Integer-valued float32 inputs in [-lim, lim]: every partial sum of the
    product is an integer below 2**24 in magnitude for K*lim*lim < 2**24, so any
    summation order gives the same fp32 result."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    A = torch.randint(-lim, lim + 1, (M, K), generator=g).to(torch.float32)
    B = torch.randint(-lim, lim + 1, (K, N), generator=g).to(torch.float32)
    return A, B
