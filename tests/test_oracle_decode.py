"""Pins for the oracle's decoding step over a paged KV cache (CPU only): the
prefill definition on the newest rows, float64 SDPA with the end-aligned causal
mask, invariance under page placement, and closed forms."""
import math

import numpy as np
import pytest
import torch

import oracle


def _cache(lens, H, d, ps, seed, shuffle=True):
    """Contiguous per-sequence K/V scattered into a page pool by a (shuffled) table."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    maxp = max((L + ps - 1) // ps for L in lens)
    npages = sum((L + ps - 1) // ps for L in lens) + 3
    order = rng.permutation(npages) if shuffle else np.arange(npages)
    kc = rng.standard_normal((npages, H, ps, d))
    vc = rng.standard_normal((npages, H, ps, d))
    pt = np.full((B, maxp), -1, dtype=np.int64)
    K, V, used = [], [], 0
    for b, L in enumerate(lens):
        n = (L + ps - 1) // ps
        pt[b, :n] = order[used:used + n]
        used += n
        t = np.arange(L)
        K.append(kc[pt[b, t // ps], :, t % ps].transpose(1, 0, 2))   # [H, L, d]
        V.append(vc[pt[b, t // ps], :, t % ps].transpose(1, 0, 2))
    return kc, vc, pt, K, V


@pytest.mark.parametrize("nq", [1, 3])
def test_equals_prefill_definition_on_the_newest_rows(nq):
    lens, H, d, ps = [5, 16, 17, 40], 2, 8, 8
    kc, vc, pt, K, V = _cache(lens, H, d, ps, seed=1)
    rng = np.random.default_rng(2)
    q = rng.standard_normal((len(lens), H, nq, d))
    o, lse = oracle.attn_decode_paged_f64(q, kc, vc, pt, lens, 0.3)
    for b, L in enumerate(lens):
        for h in range(H):
            Q = rng.standard_normal((L, d))
            Q[L - nq:] = q[b, h]                       # the decode queries are the last rows
            rows = list(range(L - nq, L))
            orf, lrf = oracle.attn_rows_f64(Q, K[b][h], V[b][h], rows, 0.3, causal=True)
            np.testing.assert_allclose(o[b, h], orf, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], lrf, rtol=0, atol=1e-12)


def test_matches_sdpa_with_end_aligned_causal_mask():
    lens, H, d, ps, nq = [9, 33], 3, 16, 16, 4
    kc, vc, pt, K, V = _cache(lens, H, d, ps, seed=3)
    q = np.random.default_rng(4).standard_normal((len(lens), H, nq, d))
    o, lse = oracle.attn_decode_paged_f64(q, kc, vc, pt, lens, 0.25)
    for b, L in enumerate(lens):
        i = torch.arange(nq)[:, None] + (L - nq)
        j = torch.arange(L)[None, :]
        mask = j <= i
        tq = torch.from_numpy(q[b])
        tk, tv = torch.from_numpy(K[b]), torch.from_numpy(V[b])
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.25)
        np.testing.assert_allclose(o[b], ref.numpy(), rtol=0, atol=1e-12)
        sc = (tq @ tk.transpose(-1, -2)) * 0.25
        np.testing.assert_allclose(lse[b], torch.logsumexp(sc.masked_fill(~mask, float("-inf")), -1).numpy(),
                                   rtol=0, atol=1e-12)


def test_page_placement_does_not_matter():
    lens, H, d, ps = [30, 7], 2, 4, 4
    q = np.random.default_rng(5).standard_normal((2, H, 1, d))
    a = _cache(lens, H, d, ps, seed=6, shuffle=False)
    # same logical K/V in a shuffled pool
    rng = np.random.default_rng(7)
    perm = rng.permutation(a[0].shape[0])
    kc2, vc2 = np.empty_like(a[0]), np.empty_like(a[1])
    kc2[perm], vc2[perm] = a[0], a[1]
    pt2 = np.where(a[2] >= 0, perm[np.maximum(a[2], 0)], -1)
    o1, l1 = oracle.attn_decode_paged_f64(q, a[0], a[1], a[2], lens, 0.5)
    o2, l2 = oracle.attn_decode_paged_f64(q, kc2, vc2, pt2, lens, 0.5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_closed_forms():
    lens, H, d, ps = [1, 12], 1, 4, 4
    kc, vc, pt, K, V = _cache(lens, H, d, ps, seed=8)
    q = np.zeros((2, H, 1, d))
    o, lse = oracle.attn_decode_paged_f64(q, kc, vc, pt, lens, 1.0)
    # a single cached key returns its value; q = 0 averages all keys
    np.testing.assert_allclose(o[0, 0, 0], V[0][0, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[1, 0, 0], V[1][0].mean(axis=0), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[1, 0, 0], math.log(12), rtol=0, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.attn_decode_paged_f64(np.zeros((2, 1, 2, 4)), kc, vc, pt, lens, 1.0)
