"""Seeded synthetic inputs for the GEMM workloads (shared by tests, oracle and bench).

This module only draws numbers: it holds none of the GEMM's arithmetic, no tiling and
no scheduling.  Both the CUDA path and the CPU oracle consume what it returns, so the
two sides always see the same bf16 bytes.

Recipe (the pages publish no inputs; every workload is synthetic):
* a ``torch.Generator`` on the CPU seeded with the workload's seed draws A first,
  then B (for grouped problems: A_0, B_0, A_1, B_1, ... in group order);
* "uniform" entries are ``torch.rand * 2 - 1`` (float32) rounded to bfloat16 with
  round-to-nearest-even; "normal" entries are ``torch.randn * sigma`` rounded the same
  way;
* grouped row counts are ``128 * ceil(x)`` clipped to [128, 8192], with x drawn from
  ``numpy.random.default_rng(seed).lognormal(mean=2, sigma=1, size=G)``;
* the variable-depth grouped workload draws, from one ``default_rng(5)``, the row counts
  as above and then depths ``K_g = 256 * ceil(x)`` clipped to [256, 16384] from a second
  ``lognormal(2, 1, G)`` draw; N = 4096 for every problem.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    seed: int
    dist: str = "uniform"          # "uniform" in [-1, 1] or "normal"
    sigma: float = 0.02
    bm: int = 128
    bn: int = 256
    cluster: int = 1
    group_m: Tuple[int, ...] = field(default_factory=tuple)   # grouped problems only
    group_k: Tuple[int, ...] = field(default_factory=tuple)   # per-problem depth (else K for all)

    def depths(self) -> Tuple[int, ...]:
        return self.group_k if self.group_k else (self.K,) * len(self.group_m)

    @property
    def flops(self) -> float:
        if self.group_m:
            return 2.0 * self.N * sum(m * k for m, k in zip(self.group_m, self.depths()))
        return 2.0 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> float:
        """Each operand read once and C written once (bf16 in, fp32 out)."""
        if self.group_m:
            return sum(2.0 * (m * k + k * self.N) + 4.0 * m * self.N for m, k in zip(self.group_m, self.depths()))
        return 2.0 * (self.M * self.K + self.K * self.N) + 4.0 * self.M * self.N


def grouped_rows(G: int = 64, seed: int = 4, lo: int = 128, hi: int = 8192) -> Tuple[int, ...]:
    x = np.random.default_rng(seed).lognormal(mean=2.0, sigma=1.0, size=G)
    m = np.clip(128 * np.ceil(x), lo, hi).astype(np.int64)
    return tuple(int(v) for v in m)


TINY = Workload("tiny_384x512x256_t128x128", 384, 512, 256, seed=0, bn=128)
SQUARE = Workload("square_8192x8192x8192", 8192, 8192, 8192, seed=1)


def tail(T: int) -> Workload:
    return Workload(f"tail_T{T}_{128 * T}x256x8192", 128 * T, 256, 8192, seed=2)


TAIL_T = (147, 148, 149, 296, 297)
PAIR = Workload("pair_16384x16384x4096_c2", 16384, 16384, 4096, seed=3, dist="normal",
                cluster=2)


def grouped() -> Workload:
    gm = grouped_rows()
    return Workload("grouped_64x(Mg)x4096x4096", sum(gm), 4096, 4096, seed=4, group_m=gm)


def grouped_varied_depth(G: int = 64, seed: int = 5) -> Workload:
    rng = np.random.default_rng(seed)
    m = np.clip(128 * np.ceil(rng.lognormal(mean=2.0, sigma=1.0, size=G)), 128, 8192).astype(np.int64)
    k = np.clip(256 * np.ceil(rng.lognormal(mean=2.0, sigma=1.0, size=G)), 256, 16384).astype(np.int64)
    gm = tuple(int(v) for v in m)
    gk = tuple(int(v) for v in k)
    return Workload("grouped_varK_64x(Mg)x4096x(Kg)", sum(gm), 4096, max(gk), seed=seed, group_m=gm, group_k=gk)


def _draw(gen: torch.Generator, shape, dist: str, sigma: float) -> torch.Tensor:
    if dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32).mul_(2.0).sub_(1.0)
    elif dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32).mul_(sigma)
    elif dist == "int":
        # integer values in [-4, 4]: exact in bf16 and in fp32 partial sums
        x = torch.randint(-4, 5, shape, generator=gen).to(torch.float32)
    else:
        raise ValueError(dist)
    return x.to(torch.bfloat16)


def make_inputs(w: Workload, dist: Optional[str] = None, pin: bool = False):
    """(A, B) as CPU bfloat16 tensors for a plain workload; for a grouped workload
    (list of A_g, list of B_g)."""
    gen = torch.Generator(device="cpu").manual_seed(w.seed)
    d = dist or w.dist
    if w.group_m:
        As: List[torch.Tensor] = []
        Bs: List[torch.Tensor] = []
        for m, k in zip(w.group_m, w.depths()):
            a = _draw(gen, (m, k), d, w.sigma)
            b = _draw(gen, (k, w.N), d, w.sigma)
            As.append(a.pin_memory() if pin else a)
            Bs.append(b.pin_memory() if pin else b)
        return As, Bs
    a = _draw(gen, (w.M, w.K), d, w.sigma)
    b = _draw(gen, (w.K, w.N), d, w.sigma)
    if pin:
        a, b = a.pin_memory(), b.pin_memory()
    return a, b


def make_matrix(shape, seed: int, dist: str = "uniform", sigma: float = 0.02) -> torch.Tensor:
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return _draw(gen, shape, dist, sigma)
