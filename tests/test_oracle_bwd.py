"""Pins for the oracle's backward pass (CPU only): torch autograd through float64
scaled_dot_product_attention with an explicit mask (library special case), central
finite differences of sum(dO * O) on tiny inputs, and closed forms."""
import math

import numpy as np
import pytest
import torch

import oracle

MODES = [(False, 0), (True, 0), (False, 3), (True, 3)]


def _mask(N, causal, window):
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    m = torch.ones(N, N, dtype=torch.bool)
    if causal:
        m &= j <= i
    if window > 0:
        m &= j >= i - window
        if not causal:
            m &= j <= i + window
    return m


@pytest.mark.parametrize("causal,window", MODES)
def test_matches_autograd_through_sdpa(causal, window):
    B, H, N, d = 1, 2, 37, 8
    rng = np.random.default_rng(1)
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    dq, dk, dv = oracle.attn_bwd_f64(q, k, v, do, 0.35, causal=causal, window=window)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=_mask(N, causal, window),
                                                           scale=0.35)
    out.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


def test_central_finite_differences():
    N, d, scale = 6, 3, 0.7
    rng = np.random.default_rng(2)
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    dq, dk, dv = oracle.attn_bwd_f64(q, k, v, do, scale, causal=True)

    def loss(q_, k_, v_):
        o, _ = oracle.attn_f64(q_, k_, v_, scale, causal=True)
        return float((o * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{a + "_": b for a, b in args_p.items()}) -
                        loss(**{a + "_": b for a, b in args_m.items()})) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-7)


def test_closed_forms():
    N, d = 5, 4
    rng = np.random.default_rng(3)
    k, v, do = (rng.standard_normal((N, d)) for _ in range(3))
    q = np.zeros((N, d))
    dq, dk, dv = oracle.attn_bwd_f64(q, k, v, do, 1.0)
    # Q = 0: P is uniform 1/N, so dV_j = mean_i dO_i for every j
    np.testing.assert_allclose(dv, np.tile(do.mean(axis=0), (N, 1)), rtol=0, atol=1e-12)
    # with every value row equal, O does not depend on Q or K: dQ = dK = 0
    vc = np.ones((N, d))
    dq2, dk2, _ = oracle.attn_bwd_f64(rng.standard_normal((N, d)), k, vc, do, 0.5)
    np.testing.assert_allclose(dq2, 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk2, 0.0, rtol=0, atol=1e-12)
    # causal row 0 sees only key 0: its query gets no gradient
    dq3, _, _ = oracle.attn_bwd_f64(rng.standard_normal((N, d)), k, v, do, 0.5, causal=True)
    np.testing.assert_allclose(dq3[0], 0.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,window", MODES)
def test_varlen_matches_autograd_over_the_packed_tensor(causal, window):
    """Library special case: autograd through float64 SDPA over the whole packed tensor
    with the block-diagonal (and causal / window) mask built from the definition."""
    lengths = [5, 1, 17, 0, 9]
    H, d = 2, 4
    rng = np.random.default_rng(21)
    T = sum(lengths)
    q, k, v, do = (rng.standard_normal((T, H, d)) for _ in range(4))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    got = oracle.attn_varlen_bwd_f64(q, k, v, do, cu, 0.4, causal=causal, window=window)
    seq = np.repeat(np.arange(len(lengths)), lengths)
    pos = np.concatenate([np.arange(n) for n in lengths])
    i, j = pos[:, None], pos[None, :]
    allowed = seq[:, None] == seq[None, :]
    if causal:
        allowed &= j <= i
    if window > 0:
        allowed &= j >= i - window
        if not causal:
            allowed &= j <= i + window
    tq, tk, tv = (torch.tensor(x.transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(allowed),
                                                         scale=0.4)
    o.backward(torch.from_numpy(do.transpose(1, 0, 2)))
    for g, t in zip(got, (tq, tk, tv)):
        np.testing.assert_allclose(g, t.grad.numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_varlen_equal_lengths_match_the_batched_layout():
    B, H, N, d = 3, 2, 11, 4
    rng = np.random.default_rng(22)
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    ref = oracle.attn_bwd_f64(q, k, v, do, 0.3, causal=True)
    pack = lambda x: x.transpose(0, 2, 1, 3).reshape(B * N, H, d)
    got = oracle.attn_varlen_bwd_f64(pack(q), pack(k), pack(v), pack(do), np.arange(B + 1) * N, 0.3,
                                     causal=True)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, pack(r))
