"""Seeded synthetic GEMM inputs, shared by the tests, the benchmark and smoke().

This module draws random numbers and nothing else: it holds none of the GEMM
arithmetic, imports nothing from the CUDA library or the oracle, and both of
those consume exactly the arrays it returns.

Recipe (every workload is synthetic; no dataset or weights are involved):

* one ``torch.Generator('cpu')`` seeded with the workload's seed draws A first,
  then B, both row-major and contiguous;
* ``uniform``: ``2*rand - 1``, i.i.d. uniform on [-1, 1) in FP32;
* ``int``: ``randint(lo, hi+1)`` converted to the target type (exact);
* ``normal``: ``mu + sigma*randn`` in FP32, then rounded once to BF16
  (round-to-nearest-even) when the path is BF16.

The BF16 rounding happens here, once; the GPU and the oracle then read the
same 16-bit patterns, so the oracle runs on the already-rounded inputs.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Dist:
    """One value distribution: kind in {"uniform", "int", "normal"}."""

    kind: str
    lo: float = -1.0
    hi: float = 1.0
    mu: float = 0.0
    sigma: float = 1.0


UNIFORM = Dist("uniform")
INT4 = Dist("int", lo=-4, hi=4)
INT3 = Dist("int", lo=-3, hi=3)
NORMAL = Dist("normal", mu=0.0, sigma=1.0)
NORMAL_W = Dist("normal", mu=0.0, sigma=0.02)


def _draw(g: torch.Generator, shape, dist: Dist) -> torch.Tensor:
    if dist.kind == "uniform":
        return 2.0 * torch.rand(shape, generator=g, dtype=torch.float32) - 1.0
    if dist.kind == "int":
        return torch.randint(int(dist.lo), int(dist.hi) + 1, shape,
                             generator=g).to(torch.float32)
    if dist.kind == "normal":
        return dist.mu + dist.sigma * torch.randn(shape, generator=g,
                                                  dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist.kind!r}")


def make_pair(M: int, N: int, K: int, seed: int, dist_a: Dist,
              dist_b: Dist | None = None, dtype: torch.dtype = torch.float32):
    """Draw A (M x K) then B (K x N) on the CPU; dtype float32 or bfloat16."""
    if dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("dtype must be float32 or bfloat16")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    a = _draw(g, (M, K), dist_a)
    b = _draw(g, (K, N), dist_b if dist_b is not None else dist_a)
    return a.to(dtype).contiguous(), b.to(dtype).contiguous()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a (CPU, contiguous) BF16 tensor."""
    if t.dtype != torch.bfloat16:
        raise TypeError("bf16_bits takes a bfloat16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def with_leading_dim(t: torch.Tensor, ld: int) -> torch.Tensor:
    """Copy of a 2-D tensor placed in a wider buffer: rows ``ld`` apart.

    The padding columns are filled with a large sentinel so that a reader
    that strays past the row end produces a visibly wrong result.
    """
    rows, cols = t.shape
    if ld < cols:
        raise ValueError("ld must be at least the row length")
    buf = torch.full((rows, ld), 1.0e6, dtype=t.dtype)
    buf[:, :cols] = t
    return buf[:, :cols]
