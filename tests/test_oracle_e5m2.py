"""Pins for the oracle's E5M2 codec and the E5M2 block quantiser (CPU only): hand-derived
code points, torch's own float8_e5m2 cast as a library special case over every rounding
class of the finite range, all 256 decodes, saturation, and the quantiser's block
invariants."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_points():
    g = json.load(open(os.path.join(GOLDEN, "e5m2_points.json")))
    for e in g["decode"]:
        v = float(oracle.e5m2_decode(np.array([e["code"]]))[0])
        assert v == e["value"] and np.signbit(v) == np.signbit(e["value"]), e
    for c in g["inf_codes"]:
        assert np.isinf(oracle.e5m2_decode(np.array([c]))[0])
    for c in g["nan_codes"]:
        assert np.isnan(oracle.e5m2_decode(np.array([c]))[0])
    for e in g["encode"]:
        assert int(oracle.e5m2_encode(np.array([e["x"]], dtype=np.float32))[0]) == e["code"], e


def test_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e5m2_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float32).numpy()
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def _rounding_classes():
    """Every finite E5M2 value, the midpoints between neighbours and one fp32 ulp on
    either side of each, both signs, below the first value torch would round to inf."""
    finite = oracle.e5m2_decode(np.arange(0, 0x7C, dtype=np.uint8)).astype(np.float64)
    mids = (finite[:-1] + finite[1:]) / 2.0
    pts = np.concatenate([finite, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(-np.inf))
    x = np.concatenate([pts, up, dn, [np.float32(61439.99)]])
    x = x[np.abs(x) < 61440.0]
    return np.concatenate([x, -x]).astype(np.float32)


def test_encode_matches_torch_cast_on_every_rounding_class():
    x = _rounding_classes()
    ours = oracle.e5m2_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_encode_matches_torch_cast_on_random_values():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(1 << 20) * np.exp2(rng.integers(-20, 16, 1 << 20))).astype(np.float32)
    x = x[np.abs(x) < 61440.0]
    ours = oracle.e5m2_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_round_trip_and_saturation():
    codes = np.array([c for c in range(256) if (c & 0x7F) < 0x7C], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e5m2_encode(oracle.e5m2_decode(codes)), codes)
    big = np.array([61440.0, 1e30, np.inf, -np.inf], dtype=np.float32)
    np.testing.assert_array_equal(oracle.e5m2_encode(big), [0x7B, 0x7B, 0x7B, 0xFB])
    assert (oracle.e5m2_encode(np.array([np.nan], dtype=np.float32)) & 0x7F)[0] == 0x7F


def test_block_quantiser_invariants():
    q, _, _ = make_qkv(1, 2, 300, 64, seed=3, outliers=True)   # ragged last block
    x8, sc = oracle.quantize_fp8_blockwise(q, 128, fmt="e5m2")
    qf = q.float().numpy()
    for h in range(2):
        for b in range(3):
            blk = qf[0, h, 128 * b:128 * (b + 1)]
            amax = np.float32(np.abs(blk).max())
            assert sc[0, h, b] == np.float32(amax / np.float32(57344.0))
            codes = x8[0, h, 128 * b:128 * (b + 1)]
            assert (codes & 0x7F).max() == 0x7B          # the amax element is the top code
    deq = oracle.dequantize(x8, sc, 128, fmt="e5m2")
    # normal-range elements are within half an E5M2 step: relative 2^-3
    rows = np.repeat(sc[0], 128, axis=-1)[:, :300].astype(np.float64)
    normal = np.abs(qf[0]) >= (2.0 ** -14) * rows[..., None]
    rel = np.abs(deq[0] - qf[0]) / np.maximum(np.abs(qf[0]), 1e-30)
    assert rel[normal].max() <= 2.0 ** -3


def test_block_quantiser_matches_torch_implementation():
    """Library special case: per-block amax, fp32 division and torch's float8_e5m2 cast."""
    q, _, _ = make_qkv(2, 2, 256, 128, seed=5, outliers=True)
    x8, sc = oracle.quantize_fp8_blockwise(q, 128, fmt="e5m2")
    x = q.float().reshape(2, 2, 2, 128, 128)
    amax = x.abs().amax(dim=(-1, -2))
    scale = torch.where(amax > 0, amax / 57344.0, torch.ones_like(amax))
    codes = (x / scale[..., None, None]).to(torch.float8_e5m2).view(torch.uint8)
    np.testing.assert_array_equal(sc, scale.numpy())
    np.testing.assert_array_equal(x8, codes.reshape(2, 2, 256, 128).numpy())


def test_zero_block_and_e4m3_default_unchanged():
    x = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    x8, sc = oracle.quantize_fp8_blockwise(x, 128, fmt="e5m2")
    assert sc[0, 0, 0] == 1.0 and (x8 == 0).all()
    q, _, _ = make_qkv(1, 1, 256, 64, seed=9)
    a8, asc = oracle.quantize_fp8_blockwise(q, 128)
    b8, bsc = oracle.quantize_fp8_blockwise(q, 128, fmt="e4m3")
    np.testing.assert_array_equal(a8, b8)
    np.testing.assert_array_equal(asc, bsc)


def test_power_of_two_scales():
    """fmt e4m3_pow2: each block's scale is the smallest power of two at or above
    fp32(amax / 448), and the codes are E4M3 of the exact quotient x / scale."""
    q, _, _ = make_qkv(2, 3, 300, 128, seed=11, outliers=True)
    x8, sc = oracle.quantize_fp8_blockwise(q, 128, fmt="e4m3_pow2")
    _, sc448 = oracle.quantize_fp8_blockwise(q, 128)             # fp32(amax / 448)
    m, e = np.frexp(sc)
    assert (m == 0.5).all()                                      # powers of two
    assert (sc >= sc448).all() and (sc < 2 * sc448).all()
    xf = q.float().numpy()
    rows = np.repeat(sc, 128, axis=-1)[..., :300]
    quot = xf / rows[..., None]                                  # exact: power-of-two divisor
    ref = torch.from_numpy(quot.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(x8, ref)
    # the amax element lands in the top binade of E4M3: amax / scale is in (224, 448], which
    # rounds to a code value of at least 224
    dec = np.abs(oracle.e4m3_decode(x8).reshape(2, 3, 300, 128))
    for b in range(3):
        assert dec[:, :, 128 * b:128 * (b + 1)].max(axis=(-1, -2)).min() >= 224.0
    # dequantised values are within half an E4M3 step of the input (relative 2^-4)
    deq = oracle.dequantize(x8, sc, 128, fmt="e4m3_pow2")
    normal = np.abs(xf) >= 2.0 ** -6 * rows[..., None]
    assert (np.abs(deq - xf) / np.maximum(np.abs(xf), 1e-30))[normal].max() <= 2.0 ** -4
