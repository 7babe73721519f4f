"""Pins for the oracle's incoherent processing (Walsh-Hadamard rotation before FP8
block quantisation), CPU only.  The rotation is checked against scipy's Sylvester
Hadamard matrix in float64, its algebraic properties, hand-worked values, and the
accuracy effect the pages credit it with."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv

scipy_linalg = pytest.importorskip("scipy.linalg")


def _rot64(d):
    return scipy_linalg.hadamard(d).astype(np.float64) / math.sqrt(d)


def test_hand_worked_d4():
    # butterflies h=1: (1+2, 1-2, 3+4, 3-4) = (3,-1,7,-1); h=2: (10,-2,-4,0); times 1/2
    y = oracle.hadamard_rotate_f32(np.array([[1.0, 2.0, 3.0, 4.0]], dtype=np.float32))
    np.testing.assert_array_equal(y, [[5.0, -1.0, -2.0, 0.0]])


def test_scale_constant():
    assert oracle.hadamard_scale(64) == np.float32(0.125)
    assert oracle.hadamard_scale(256) == np.float32(0.0625)
    assert oracle.hadamard_scale(128) == np.float32(0.08838834764831845)


@pytest.mark.parametrize("d", [2, 8, 64, 128, 256])
def test_matches_sylvester_matrix_within_fp32_bound(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((300, d)).astype(np.float32)
    x[::7, d // 3] *= 40.0  # outliers
    y = oracle.hadamard_rotate_f32(x).astype(np.float64)
    ref = x.astype(np.float64) @ _rot64(d)
    # log2(d) rounded add/sub stages on partial sums bounded by sum|x|, then one
    # rounded multiply by c (itself within 2^-24 of 1/sqrt(d))
    u = 2.0 ** -24
    bound = (math.log2(d) + 3) * u * np.abs(x).astype(np.float64).sum(axis=1, keepdims=True) / math.sqrt(d)
    assert (np.abs(y - ref) <= bound).all()


@pytest.mark.parametrize("d", [64, 128, 256])
def test_rotation_is_its_own_inverse(d):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, d)).astype(np.float32)
    back = oracle.hadamard_rotate_f32(oracle.hadamard_rotate_f32(x))
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-5)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_one_hot_rows_spread_evenly(d):
    x = np.eye(d, dtype=np.float32)
    y = oracle.hadamard_rotate_f32(x)
    c = oracle.hadamard_scale(d)
    j = np.arange(d)
    for k in range(d):
        sign = np.where(np.array([bin(k & jj).count("1") & 1 for jj in j]) == 1, -1.0, 1.0)
        np.testing.assert_array_equal(y[k], (sign * c).astype(np.float32))


def test_bf16_input_widened_exactly():
    x = torch.randn(5, 128).to(torch.bfloat16)
    np.testing.assert_array_equal(oracle.hadamard_rotate_f32(x),
                                  oracle.hadamard_rotate_f32(x.float().numpy()))


def test_rotating_q_and_k_leaves_attention_unchanged():
    rng = np.random.default_rng(2)
    N, d = 70, 64
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    R = _rot64(d)
    for causal, window in [(False, 0), (True, 0), (True, 9)]:
        o1, l1 = oracle.attn_f64(q, k, v, 0.125, causal=causal, window=window)
        o2, l2 = oracle.attn_f64(q @ R, k @ R, v, 0.125, causal=causal, window=window)
        np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


def test_outlier_is_spread_over_the_row():
    d = 128
    x = np.full((1, d), 0.5, dtype=np.float32)
    x[0, 17] = 200.0
    y = oracle.hadamard_rotate_f32(x)
    # the outlier contributes +-200/sqrt(d) to every coordinate
    assert np.abs(y).max() < 200.0 / math.sqrt(d) + 0.5 * math.sqrt(d)
    assert np.abs(y).max() > 200.0 / math.sqrt(d) - 0.5 * math.sqrt(d)


def test_quantize_hadamard_is_rotation_then_block_quantisation():
    q, _, _ = make_qkv(1, 2, 200, 128, seed=4, outliers=True)
    x8, sc = oracle.quantize_fp8_hadamard(q)
    r8, rsc = oracle.quantize_fp8_blockwise(oracle.hadamard_rotate_f32(q))
    np.testing.assert_array_equal(x8, r8)
    np.testing.assert_array_equal(sc, rsc)
    assert sc.shape == (1, 2, 2)


def _rel_rmse(o, ref):
    return float(np.sqrt(np.mean((o - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))


def test_rotation_lowers_error_against_unquantised_attention():
    """On the outlier input distribution, attention on dequantised rotated Q, K (and
    plainly quantised V) is closer to attention on the unquantised inputs than with
    block quantisation alone -- the accuracy effect the pages ascribe to incoherent
    processing.  float64 attention over all rows of two heads."""
    B, H, N, d = 1, 2, 1024, 128
    q, k, v = make_qkv(B, H, N, d, seed=0, outliers=True)
    scale = 1.0 / math.sqrt(d)
    ref, _ = oracle.attn_f64(q, k, v, scale)
    vhat = oracle.dequantize(*oracle.quantize_fp8_blockwise(v))
    qb = oracle.dequantize(*oracle.quantize_fp8_blockwise(q))
    kb = oracle.dequantize(*oracle.quantize_fp8_blockwise(k))
    qr = oracle.dequantize(*oracle.quantize_fp8_hadamard(q))
    kr = oracle.dequantize(*oracle.quantize_fp8_hadamard(k))
    e_block = _rel_rmse(oracle.attn_f64(qb, kb, vhat, scale)[0], ref)
    e_rot = _rel_rmse(oracle.attn_f64(qr, kr, vhat, scale)[0], ref)
    assert e_rot < 0.75 * e_block, (e_rot, e_block)
