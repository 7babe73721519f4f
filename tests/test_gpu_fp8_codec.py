"""The device's FP8 conversion (cvt.rn.satfinite, as the quantisers use it) against the
oracle's E4M3 and E5M2 encoders, written from the OCP bit layouts, over every one of the
2^32 fp32 bit patterns ("大模型加速-核心网络算子-Flash Attention V3" §1.5: E4M3 and E5M2).
Finite values and infinities must give the same code bit for bit; a NaN input must give
a NaN code of the format (the encoders may differ in which one)."""
import numpy as np
import pytest
import torch

import oracle
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _is_nan_code(codes, fmt):
    if fmt == "e4m3":
        return (codes & 0x7F) == 0x7F
    return ((codes & 0x7C) == 0x7C) & ((codes & 0x03) != 0)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_every_fp32_pattern(fa, fmt):
    encode = oracle.e4m3_encode if fmt == "e4m3" else oracle.e5m2_encode
    buf = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    checked = 0
    for first in range(0, 1 << 32, CHUNK):
        gpu = fa.attn_selftest_fp8_convert(first, CHUNK, fmt, codes=buf).cpu().numpy()
        bits = np.arange(first, first + CHUNK, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        ref = encode(x)
        nan = np.isnan(x)
        mism = np.flatnonzero((gpu != ref) & ~nan)
        assert mism.size == 0, (fmt, hex(int(bits[mism[0]])), int(gpu[mism[0]]), int(ref[mism[0]]))
        assert _is_nan_code(gpu[nan], fmt).all()
        checked += CHUNK
    assert checked == 1 << 32
    assert fa.attn_get_device_status() == fa.ATTN_OK


def test_arguments_are_checked(fa):
    with pytest.raises(fa.AttnError):
        fa.attn_selftest_fp8_convert(0, 12, "e4m3")              # not a multiple of 8
    with pytest.raises(fa.AttnError):
        fa.attn_selftest_fp8_convert((1 << 32) - 8, 16, "e4m3")  # past the last pattern
    with pytest.raises(fa.AttnError):
        fa.attn_selftest_fp8_convert(0, 8, "e4m3_pow2")          # not a conversion format
