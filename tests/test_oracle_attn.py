"""Pins for the float64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: hand-derived
values, closed forms, invariants, a library routine in a special case, or a
brute-force enumeration.  Mask modes are the (causal, window) pairs the kernel
supports; window <= 0 means no window.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import GOLDEN

MODES = [(False, 0), (True, 0), (False, 5), (True, 5), (True, 1), (False, 1)]


def _rand_head(N, d, seed, dtype=np.float64):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((N, d))
    k = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    return q, k, v


def _allowed_count(i, N, causal, window):
    """|A_i| in closed form."""
    if window <= 0:
        return i + 1 if causal else N
    if causal:
        return min(i, window) + 1
    return min(N - 1, i + window) - max(0, i - window) + 1


def test_golden_two_key_example():
    g = json.load(open(os.path.join(GOLDEN, "two_key_example.json")))
    q, k, v = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "v"))
    for causal, key in ((False, "non_causal"), (True, "causal")):
        o, lse = oracle.attn_f64(q, k, v, g["scale"], causal=causal)
        np.testing.assert_allclose(o, np.array(g[key]["o"]), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, np.array(g[key]["lse"]), rtol=0, atol=1e-12)


def test_mask_matches_printed_band_construction():
    """Non-causal window: the printed construction mask[i, max(0,i-w):i+w+1] = 1."""
    for N in (1, 2, 7, 33, 64):
        for w in (1, 2, 5, 17, 100):
            ref = np.zeros((N, N), dtype=int)
            for i in range(N):
                ref[i, max(0, i - w):i + w + 1] = 1
            got = np.array([[int(oracle.key_allowed(i, j, N, False, w)) for j in range(N)]
                            for i in range(N)])
            np.testing.assert_array_equal(got, ref)
            got_c = np.array([[int(oracle.key_allowed(i, j, N, True, w)) for j in range(N)]
                              for i in range(N)])
            np.testing.assert_array_equal(got_c, np.tril(ref))


def test_mask_golden_and_counts():
    g = json.load(open(os.path.join(GOLDEN, "window_mask_n6_w1.json")))
    N, w = g["N"], g["window"]
    got = [[int(oracle.key_allowed(i, j, N, False, w)) for j in range(N)] for i in range(N)]
    assert got == g["mask"]
    got_c = [[int(oracle.key_allowed(i, j, N, True, w)) for j in range(N)] for i in range(N)]
    assert got_c == g["causal_mask"]
    for N in (1, 5, 64):
        for causal, window in MODES + [(False, 1000), (True, 1000)]:
            for i in range(N):
                cnt = sum(oracle.key_allowed(i, j, N, causal, window) for j in range(N))
                assert cnt == _allowed_count(i, N, causal, window)
    # keys outside [0, N) are never allowed
    assert not oracle.key_allowed(3, -1, 8, False, 0)
    assert not oracle.key_allowed(3, 8, 8, False, 0)


@pytest.mark.parametrize("causal,window", MODES)
def test_zero_query_gives_mean_of_allowed_values(causal, window):
    N, d = 37, 8
    _, k, v = _rand_head(N, d, 1)
    q = np.zeros((N, d))
    o, lse = oracle.attn_f64(q, k, v, 0.37, causal=causal, window=window)
    for i in range(N):
        js = [j for j in range(N) if oracle.key_allowed(i, j, N, causal, window)]
        np.testing.assert_allclose(o[i], v[js].mean(axis=0), rtol=0, atol=1e-12)
        assert abs(lse[i] - math.log(len(js))) < 1e-12


def test_causal_row_zero_is_first_value():
    N, d = 29, 16
    q, k, v = _rand_head(N, d, 2)
    scale = 0.25
    for window in (0, 3):
        o, lse = oracle.attn_f64(q, k, v, scale, causal=True, window=window)
        np.testing.assert_allclose(o[0], v[0], rtol=0, atol=1e-12)
        assert abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-12


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (False, 4)])
def test_one_hot_score_selects_that_value_row(causal, window):
    N, d = 24, 8
    q, k, v = _rand_head(N, d, 3)
    q *= 0.01
    i, jstar = 12, 10
    k[jstar] = 1000.0 * q[i] / float(q[i] @ q[i])   # q_i . k_j* = 1000 >> every other score
    o, _ = oracle.attn_f64(q, k, v, 1.0, causal=causal, window=window)
    np.testing.assert_allclose(o[i], v[jstar], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,window", MODES)
def test_rows_of_p_sum_to_one(causal, window):
    """With every value row equal to 1, O_i = sum_j P_ij must be exactly 1."""
    N, d = 50, 4
    q, k, _ = _rand_head(N, d, 4)
    q *= 3.0
    v = np.ones((N, d))
    o, _ = oracle.attn_f64(q, k, v, 0.9, causal=causal, window=window)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,window", MODES)
def test_matches_torch_sdpa_float64(causal, window):
    """Library special case: torch's scaled_dot_product_attention in float64 with an
    explicit boolean mask, and torch.logsumexp of the masked scores for the LSE."""
    B, H, N, d = 2, 3, 45, 16
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attn_f64(q, k, v, scale, causal=causal, window=window)
    ii = torch.arange(N)[:, None]
    jj = torch.arange(N)[None, :]
    allowed = torch.ones(N, N, dtype=torch.bool)
    if causal:
        allowed &= jj <= ii
    if window > 0:
        allowed &= jj >= ii - window
        if not causal:
            allowed &= jj <= ii + window
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=allowed,
                                                           scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    s = (tq @ tk.transpose(-1, -2)) * scale
    s = s.masked_fill(~allowed, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_rows_api_matches_full_api():
    N, d = 70, 8
    q, k, v = _rand_head(N, d, 6)
    rows = [0, 5, 33, 69]
    for causal, window in MODES:
        o, lse = oracle.attn_f64(q, k, v, 0.3, causal=causal, window=window)
        orow, lrow = oracle.attn_rows_f64(q, k, v, rows, 0.3, causal=causal, window=window)
        np.testing.assert_array_equal(orow, o[rows])
        np.testing.assert_array_equal(lrow, lse[rows])


def test_heads_are_independent():
    """Batching heads gives the per-head result (no cross-head mixing)."""
    B, H, N, d = 2, 2, 20, 4
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    o, lse = oracle.attn_f64(q, k, v, 0.5, causal=True)
    for b in range(B):
        for h in range(H):
            oh, lh = oracle.attn_f64(q[b, h], k[b, h], v[b, h], 0.5, causal=True)
            np.testing.assert_array_equal(o[b, h], oh)
            np.testing.assert_array_equal(lse[b, h], lh)


@pytest.mark.parametrize("causal,window", MODES + [(True, 40), (False, 40)])
@pytest.mark.parametrize("BM,BN", [(16, 16), (32, 64), (64, 32), (128, 128), (16, 128)])
@pytest.mark.parametrize("tau", [0.0, 8.0 * math.log(2.0)])
def test_online_replay_equals_two_pass(causal, window, BM, BN, tau):
    """Tile-by-tile online softmax (with eager or lazy rescaling) equals the
    two-pass definition to 1e-12 on small heads, including a ragged tail."""
    N, d = 203, 16
    q, k, v = _rand_head(N, d, 8)
    q *= 2.0
    scale = 1.0 / math.sqrt(d)
    o2, l2 = oracle.attn_f64(q, k, v, scale, causal=causal, window=window)
    o1, l1 = oracle.online_replay_f64(q, k, v, scale, causal, window, BM, BN, tau)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_bf16_widening_is_exact():
    x = torch.randn(1000).to(torch.bfloat16)
    wide = oracle._f64(x)
    assert np.array_equal(wide.astype(np.float32), x.float().numpy())
