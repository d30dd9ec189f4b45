"""Seeded synthetic inputs for the all-to-all workloads.

This module only makes input data (shapes, dtypes, value distributions,
seeds).  It holds none of the permutation arithmetic, so both the CUDA path
and the CPU oracle may take their inputs from it.

Recipe (per workload): one ``torch.Generator('cpu')`` seeded with the
workload's seed draws the ranks' inputs one after another in rank order, in
fp32 (``randn`` for N(0,1), ``rand*2a - a`` for U(-a, a)), rounded to the
workload dtype (round-to-nearest-even).  Integer "iota" inputs number every
element: ``rank * base + flat index inside that rank's input``.

Input layout: ``[W][rows][H][D]`` with rows = S*W for a combine input and
rows = S for a dispatch input.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    op: str            # "combine" or "roundtrip" (dispatch, then its inverse)
    W: int
    S: int             # combine: rows per (source, destination) block; dispatch: rows per rank
    H: int
    D: int
    dtype: torch.dtype
    dist: str          # "iota1e6", "normal", "uniform1", "uniform8"
    seed: int
    tile_s: int = 16   # rows per producer/consumer tile
    variants: tuple = ("direct", "pc")

    @property
    def es(self) -> int:
        return torch.empty((), dtype=self.dtype).element_size()

    @property
    def in_rows(self) -> int:
        return self.S * self.W if self.op == "combine" else self.S

    @property
    def numel_per_rank(self) -> int:
        return self.in_rows * self.H * self.D

    @property
    def total_bytes(self) -> int:
        """T: input bytes over all W ranks (the moved tensor)."""
        return self.W * self.numel_per_rank * self.es


# The five workloads: a tiny iota case, a small MoE layer, a DeepSeek-V3-shaped
# combine (hidden 7168, 8 ranks, 2048 tokens per rank pair), a 16-rank
# dispatch/inverse round trip and an unaligned-row (999-element) stress case.
WORKLOADS = {
    "tiny": Workload("tiny", "combine", 2, 4, 2, 8, torch.int32, "iota1e6", 0, tile_s=2),
    "small": Workload("small", "combine", 8, 128, 8, 128, torch.bfloat16, "normal", 1),
    "dsv3": Workload("dsv3", "combine", 8, 2048, 1, 7168, torch.bfloat16, "normal", 2),
    "roundtrip": Workload("roundtrip", "roundtrip", 16, 1024, 4, 128, torch.float16, "uniform1",
                          3, variants=("direct",)),
    "tail": Workload("tail", "combine", 32, 256, 2, 999, torch.float16, "uniform8", 4,
                     tile_s=32),
}


def _draw(g: torch.Generator, shape, dist: str, dtype: torch.dtype) -> torch.Tensor:
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)
    if dist.startswith("uniform"):
        a = float(dist[len("uniform"):])
        return (torch.rand(shape, generator=g, dtype=torch.float32) * (2 * a) - a).to(dtype)
    raise ValueError(dist)


def iota(W: int, rows: int, H: int, D: int, base: int, dtype=torch.int64) -> torch.Tensor:
    """[W][rows][H][D] with value rank*base + flat index inside the rank."""
    per = rows * H * D
    flat = torch.arange(per, dtype=torch.int64)
    out = torch.stack([flat + r * base for r in range(W)]).reshape(W, rows, H, D)
    return out.to(dtype)


def make_input(wl: Workload, out: torch.Tensor | None = None) -> torch.Tensor:
    """The workload's input, [W][rows][H][D] on the CPU (written into ``out``
    when given, e.g. a pinned host buffer)."""
    shape = (wl.W, wl.in_rows, wl.H, wl.D)
    if out is None:
        out = torch.empty(shape, dtype=wl.dtype)
    assert tuple(out.shape) == shape and out.dtype == wl.dtype
    if wl.dist == "iota1e6":
        out.copy_(iota(wl.W, wl.in_rows, wl.H, wl.D, 1_000_000, wl.dtype))
        return out
    g = torch.Generator("cpu")
    g.manual_seed(wl.seed)
    for r in range(wl.W):
        out[r].copy_(_draw(g, shape[1:], wl.dist, wl.dtype))
    return out


def random_bytes(nbytes: int, seed: int) -> torch.Tensor:
    """uint8 noise for primitive tests."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    return torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8)


def moe_counts(W: int, tokens: int, experts: int, topk: int, seed: int,
               skew: float = 1.0) -> torch.Tensor:
    """Rows each PE sends to each PE under synthetic top-k MoE routing.

    Each of the ``tokens`` tokens on PE r picks ``topk`` distinct experts
    (``torch.multinomial`` without replacement) from ``experts`` experts whose
    popularity follows a Zipf law of exponent ``skew`` over a seeded random
    order; expert e lives on PE ``e // (experts // W)``.  A token travels once
    to every PE that hosts at least one of its experts, so ``counts[r, d]`` is
    the number of tokens of PE r with an expert on PE d.  Returns [W, W] int64.
    """
    assert experts % W == 0 and 0 < topk <= experts
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    order = torch.randperm(experts, generator=g)
    weight = torch.empty(experts, dtype=torch.float64)
    weight[order] = 1.0 / torch.arange(1, experts + 1, dtype=torch.float64) ** skew
    counts = torch.zeros(W, W, dtype=torch.int64)
    per_pe = experts // W
    for r in range(W):
        picked = torch.multinomial(weight.expand(tokens, experts), topk, replacement=False,
                                   generator=g)
        hit = torch.zeros(tokens, W, dtype=torch.bool)
        hit.scatter_(1, picked // per_pe, True)
        counts[r] = hit.sum(0)
    return counts


def random_counts(W: int, high: int, seed: int, zero_frac: float = 0.0) -> torch.Tensor:
    """[W, W] int64 counts uniform in [0, high), a ``zero_frac`` share set to 0."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    c = torch.randint(0, high, (W, W), generator=g, dtype=torch.int64)
    if zero_frac > 0:
        c[torch.rand(W, W, generator=g) < zero_frac] = 0
    return c


def ag_matmul_inputs(W: int, m_local: int, k: int, n: int, dtype: torch.dtype, seed: int):
    """Per-rank a [W, m_local, k] and b [W, k, n] of the fused AllGather +
    MatMul, N(0, 1) drawn in fp32 from one seeded generator (a first, then b)
    and rounded to `dtype`."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    a = torch.randn(W, m_local, k, generator=g).to(dtype)
    b = torch.randn(W, k, n, generator=g).to(dtype)
    return a, b
