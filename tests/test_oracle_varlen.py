"""Pins for the oracle's packed variable-length attention (CPU only): a library
special case over the whole packed tensor with an explicit block-diagonal mask,
closed forms that show no key crosses a sequence boundary, and edge lengths."""
import math

import numpy as np
import pytest
import torch

import oracle

MODES = [(False, 0), (True, 0), (False, 3), (True, 3)]


def _packed(lengths, H, d, seed):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, cu


def _block_mask(cu, causal, window):
    """Allowed (query token, key token) pairs of the packed tensor, built from the
    definition: same sequence, and the mask rules on positions inside it."""
    T = int(cu[-1])
    seq = np.zeros(T, dtype=np.int64)
    pos = np.zeros(T, dtype=np.int64)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        seq[a:b] = s
        pos[a:b] = np.arange(b - a)
    i, j = pos[:, None], pos[None, :]
    allowed = seq[:, None] == seq[None, :]
    if causal:
        allowed &= j <= i
    if window > 0:
        allowed &= j >= i - window
        if not causal:
            allowed &= j <= i + window
    return torch.from_numpy(allowed)


@pytest.mark.parametrize("causal,window", MODES)
def test_matches_sdpa_with_block_diagonal_mask(causal, window):
    lengths = [5, 1, 17, 0, 9, 33]
    H, d = 3, 8
    q, k, v, cu = _packed(lengths, H, d, seed=1)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attn_varlen_f64(q, k, v, cu, scale, causal=causal, window=window)
    allowed = _block_mask(cu, causal, window)
    # [T, H, d] -> [H, T, d]: every head over all packed tokens, one mask
    tq, tk, tv = (torch.from_numpy(x).transpose(0, 1) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=allowed, scale=scale)
    np.testing.assert_allclose(o, ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
    sc = (tq @ tk.transpose(-1, -2)) * scale
    ref_lse = torch.logsumexp(sc.masked_fill(~allowed, float("-inf")), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


def test_zero_query_averages_only_its_own_sequence():
    lengths = [4, 7, 2]
    H, d = 2, 5
    _, k, v, cu = _packed(lengths, H, d, seed=2)
    q = np.zeros_like(k)
    o, lse = oracle.attn_varlen_f64(q, k, v, cu, 0.5, causal=False)
    for a, b in zip(cu[:-1], cu[1:]):
        for t in range(a, b):
            np.testing.assert_allclose(o[t], v[a:b].mean(axis=0), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[:, t], math.log(b - a), rtol=0, atol=1e-12)


def test_causal_first_token_of_each_sequence_is_its_value():
    lengths = [3, 6, 1, 5]
    H, d = 2, 4
    q, k, v, cu = _packed(lengths, H, d, seed=3)
    o, lse = oracle.attn_varlen_f64(q, k, v, cu, 0.3, causal=True, window=2)
    for a in cu[:-1]:
        np.testing.assert_allclose(o[a], v[a], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, a], 0.3 * (q[a] * k[a]).sum(-1), rtol=0, atol=1e-12)


def test_equal_lengths_match_the_batched_layout():
    B, H, N, d = 3, 2, 11, 4
    rng = np.random.default_rng(4)
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    ob, lb = oracle.attn_f64(q, k, v, 0.2, causal=True)
    pack = lambda x: x.transpose(0, 2, 1, 3).reshape(B * N, H, d)   # [B,H,N,d] -> [B*N,H,d]
    cu = np.arange(B + 1) * N
    ov, lv = oracle.attn_varlen_f64(pack(q), pack(k), pack(v), cu, 0.2, causal=True)
    np.testing.assert_array_equal(ov, pack(ob))
    np.testing.assert_array_equal(lv, lb.transpose(1, 0, 2).reshape(H, B * N))


def test_rejects_bad_offsets():
    q = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.attn_varlen_f64(q, q, q, [0, 3, 2, 4], 1.0)
    with pytest.raises(ValueError):
        oracle.attn_varlen_f64(q, q, q, [0, 3], 1.0)
