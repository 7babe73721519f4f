"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers; it holds none of the attention or
quantisation arithmetic, so the CUDA path and the oracle can both be fed from
it without sharing any of the method.

Recipe (one CPU ``torch.Generator`` seeded with ``seed``):
  1. Q, K, V = three successive ``randn(B, H, N, d)`` float32 draws, i.i.d. N(0, 1).
  2. With ``outliers``: three successive ``rand(B, H, N, d) < frac`` draws pick
     the outlier entries of Q, K, V (in that order); those entries are
     multiplied by ``mult`` (default 0.1 % of entries, x20).
  3. Each tensor is rounded to bfloat16.  Layout [B, H, N, d], contiguous.
"""
from __future__ import annotations

import math

import torch


def make_qkv(B: int, H: int, N: int, d: int, seed: int = 0, outliers: bool = False,
             frac: float = 1e-3, mult: float = 20.0):
    """Return bf16 CPU tensors (q, k, v), each [B, H, N, d] contiguous."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if outliers:
        for t in (q, k, v):
            sel = torch.rand(shape, generator=g) < frac
            t[sel] *= mult
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def default_scale(d: int) -> float:
    """1/sqrt(d), the softmax temperature every workload uses."""
    return 1.0 / math.sqrt(d)


def sampled_heads(B: int, H: int, count: int = 4, seed: int = 1):
    """(b, h) heads checked at full size: (0, 0), (B-1, H-1) and the rest drawn
    from a CPU generator seeded ``seed`` (distinct, in draw order)."""
    heads = [(0, 0)]
    if (B - 1, H - 1) not in heads:
        heads.append((B - 1, H - 1))
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    tries = 0
    while len(heads) < min(count, B * H) and tries < 1000:
        idx = int(torch.randint(0, B * H, (1,), generator=g).item())
        bh = (idx // H, idx % H)
        if bh not in heads:
            heads.append(bh)
        tries += 1
    return heads


def sampled_rows(N: int, count: int, seed: int = 2):
    """Query rows checked when a head is too long for every row: the first and
    last rows, rows at tile edges, and the rest drawn uniformly (sorted, distinct)."""
    fixed = {0, 1, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1}
    rows = {r for r in fixed if 0 <= r < N}
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    while len(rows) < min(count, N):
        rows.add(int(torch.randint(0, N, (1,), generator=g).item()))
    return sorted(rows)
