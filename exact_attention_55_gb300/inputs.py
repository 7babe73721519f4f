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

Packed variable-length sequences (``make_packed_qkv``): the same draws with shape
[T, H, d] (T = sum of the lengths), token-major; ``cu`` holds the offsets.
``varlen_lengths`` draws a length mix: uniform integers in [lo, hi] from a CPU
generator, the last length adjusted so the lengths sum to ``total``.

Paged KV cache (``make_paged_cache``): one generator draws q ([B, H, nq, d]), then
the K pool and the V pool ([num_pages, H, page_size, d], num_pages = the pages the
sequences need plus ``spare``), then a permutation of the pages; sequence b takes
the next ceil(L_b / page_size) pages of that permutation, in order.  Unused table
entries are 0.
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


def make_packed_qkv(lengths, H: int, d: int, seed: int = 0, outliers: bool = False,
                    frac: float = 1e-3, mult: float = 20.0):
    """Return bf16 CPU tensors (q, k, v), each [T, H, d], and the int32 offsets cu
    ([len(lengths) + 1], cu[0] = 0, cu[-1] = T)."""
    T = int(sum(int(n) for n in lengths))
    q, k, v = make_qkv(1, 1, T * H, d, seed=seed, outliers=outliers, frac=frac, mult=mult)
    shape = (T, H, d)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor([int(n) for n in lengths], dtype=torch.int64), 0).to(torch.int32)
    return q.reshape(shape), k.reshape(shape), v.reshape(shape), cu


def varlen_lengths(total: int, lo: int, hi: int, seed: int = 3):
    """Sequence lengths drawn uniformly from [lo, hi] until they reach ``total``;
    the last one is cut (or the remainder appended) so the sum is exactly total."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out, acc = [], 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def make_paged_cache(lens, H: int, nq: int, d: int, page_size: int, seed: int = 0, spare: int = 3):
    """Return (q, k_cache, v_cache, page_table int32 [B, max_pages], seq_lens int32 [B])."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    B = len(lens)
    need = [(int(L) + page_size - 1) // page_size for L in lens]
    max_pages = max(1, max(need))
    num_pages = sum(need) + spare
    q = torch.randn((B, H, nq, d), generator=g).to(torch.bfloat16)
    kc = torch.randn((num_pages, H, page_size, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((num_pages, H, page_size, d), generator=g).to(torch.bfloat16)
    perm = torch.randperm(num_pages, generator=g)
    table = torch.zeros((B, max_pages), dtype=torch.int32)
    used = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[used:used + n].to(torch.int32)
        used += n
    return q, kc, vc, table, torch.tensor([int(L) for L in lens], dtype=torch.int32)
