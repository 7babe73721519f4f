"""Pins for the oracle's E4M3 codec and per-block FP8 quantiser (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv
from tests.conftest import GOLDEN


def _rounding_class_patterns():
    """fp32 bit patterns that cover every E4M3 rounding class with |x| <= 464 (below the NaN code):
    all exponents from deep subnormal to 2^8, every value of the 8 leading
    mantissa bits, and low bits below the rounding point that are zero, just
    above zero, just below the midpoint, exactly the midpoint (a tie) and just
    above it, for both signs; plus zero, infinities and NaN."""
    exps = np.arange(100, 136, dtype=np.uint32)          # 2^-27 .. 2^8
    top = np.arange(0, 256, dtype=np.uint32) << np.uint32(15)
    low = np.array([0, 1, 0x3FFF, 0x4000, 0x4001, 0x7FFF, 0x1FFF, 0x2000, 0x2001],
                   dtype=np.uint32)
    bits = (exps[:, None, None] << np.uint32(23)) | top[None, :, None] | low[None, None, :]
    bits = bits.reshape(-1)
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    return bits.view(np.float32)


def test_encode_matches_torch_cast_on_every_rounding_class():
    x = _rounding_class_patterns()
    # torch's cast rounds magnitudes above the 448/480 midpoint (464) to the NaN
    # code; the saturating encoder clamps them to 448 (checked separately below)
    x = x[np.abs(x) <= 464.0]
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_encode_matches_torch_cast_on_random_patterns():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=4_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 464.0)]
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_saturation_and_specials():
    big = np.array([448.0, 464.0, np.nextafter(np.float32(464.0), np.float32(1e9)), 479.9,
                    480.0, 1e6, 3.4e38, np.inf], dtype=np.float32)
    assert (oracle.e4m3_encode(big) == 0x7E).all()
    assert (oracle.e4m3_encode(-big) == 0xFE).all()
    nan = oracle.e4m3_encode(np.array([np.nan], dtype=np.float32))[0]
    assert nan & 0x7F == 0x7F
    assert oracle.e4m3_encode(np.array([-0.0], dtype=np.float32))[0] == 0x80


def test_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])


def test_codec_golden_points():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_points.json")))
    for e in g["decode"]:
        assert float(oracle.e4m3_decode(np.array([e["code"]]))[0]) == e["value"], e
    for c in g["nan_codes"]:
        assert np.isnan(oracle.e4m3_decode(np.array([c]))[0])
    for e in g["encode"]:
        assert int(oracle.e4m3_encode(np.array([e["x"]], dtype=np.float32))[0]) == e["code"], e


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes))
    # +0 and -0 both survive as themselves
    np.testing.assert_array_equal(back, codes)


def _torch_block_quant(x, block):
    """Library special case: per-block amax and fp32 division in torch, then
    torch's own float8_e4m3fn cast (RNE; agrees with satfinite up to 464, and
    x / (amax / 448) never exceeds 448 by more than an fp32 rounding)."""
    B, H, N, d = x.shape
    xf = x.to(torch.float32)
    nblk = (N + block - 1) // block
    x8 = torch.empty(B, H, N, d, dtype=torch.uint8)
    sc = torch.empty(B, H, nblk, dtype=torch.float32)
    for b in range(nblk):
        blk = xf[:, :, b * block:(b + 1) * block]
        amax = blk.abs().amax(dim=(-1, -2))
        s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        q = blk / s[..., None, None]
        x8[:, :, b * block:(b + 1) * block] = q.to(torch.float8_e4m3fn).view(torch.uint8)
        sc[:, :, b] = s
    return x8.numpy(), sc.numpy()


@pytest.mark.parametrize("N", [128, 384, 200])
def test_quantizer_matches_torch_reference(N):
    q, k, v = make_qkv(2, 3, N, 64, seed=11, outliers=True)
    for x in (q, k, v):
        x8, sc = oracle.quantize_fp8_blockwise(x, 128)
        r8, rsc = _torch_block_quant(x, 128)
        np.testing.assert_array_equal(sc, rsc)
        np.testing.assert_array_equal(x8, r8)


def test_quantizer_block_invariants():
    q, _, _ = make_qkv(1, 2, 256, 128, seed=3, outliers=True)
    x = q.float().numpy()
    x8, sc = oracle.quantize_fp8_blockwise(q, 128)
    deq = oracle.dequantize(x8, sc, 128)
    for h in range(2):
        for b in range(2):
            blk = x[0, h, b * 128:(b + 1) * 128]
            amax = np.abs(blk).max()
            assert sc[0, h, b] == np.float32(amax) / np.float32(448.0)
            # the largest element lands on (or next to) the top code 448
            top = np.abs(oracle.e4m3_decode(x8[0, h, b * 128:(b + 1) * 128])).max()
            assert top == 448.0
            # dequantisation error: half an E4M3 step (relative 2^-4) for normals,
            # half the subnormal step 2^-10 * scale below 2^-6 * scale
            err = np.abs(deq[0, h, b * 128:(b + 1) * 128] - blk)
            bound = np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** -10 * float(sc[0, h, b]))
            assert (err <= bound * (1 + 1e-6)).all()


def test_quantizer_zero_block_and_ragged_tail():
    x = torch.zeros(1, 1, 200, 64, dtype=torch.bfloat16)
    x[0, 0, 150, 3] = -2.5
    x8, sc = oracle.quantize_fp8_blockwise(x, 128)
    assert sc.shape == (1, 1, 2)
    assert sc[0, 0, 0] == 1.0 and (x8[0, 0, :128] == 0).all()
    assert sc[0, 0, 1] == np.float32(2.5) / np.float32(448.0)
    assert x8[0, 0, 150, 3] == 0xFE  # -448
    assert (np.delete(x8[0, 0, 128:].reshape(-1), 22 * 64 + 3) == 0).all()


def test_dequantize_is_decode_times_block_scale():
    x8 = np.array([[[[0x38, 0xB8], [0x7E, 0x01]]]], dtype=np.uint8)  # 1, -1, 448, 2^-9
    sc = np.array([[[0.5]]], dtype=np.float32)
    deq = oracle.dequantize(x8, sc, 128)
    np.testing.assert_array_equal(deq, [[[[0.5, -0.5], [224.0, 2.0 ** -10]]]])
