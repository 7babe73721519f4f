"""GPU parity of E4M3 with power-of-two block scales: attn_quantize_fp8_blockwise_fmt
('e4m3_pow2') bit for bit against the oracle, and attn_fwd_fp8_fmt with power-of-two V
scales (V's descale applied through P's exponent, O rescaled only when a row max or the
largest V scale grows) against the oracle on the dequantised inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv, sampled_heads, sampled_rows
from tests.attn_check import FP8_REL_RMSE_DEQ, gather, oracle_rows, rel_rmse
from tests.conftest import require_gpu
from tests.test_gpu_fp8 import _rounding_class_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _quant(fa, x, fmt):
    x8, sc = fa.attn_quantize_fp8_blockwise_fmt(x.cuda(), fmt)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    return x8.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("N,d", [(128, 128), (1000, 64), (300, 256), (77, 16)])
def test_quantizer_bit_exact_small(fa, N, d):
    q, k, v = make_qkv(2, 3, N, d, seed=61, outliers=True)
    for x in (q, k, v):
        x8, sc = _quant(fa, x, "e4m3_pow2")
        r8, rsc = oracle.quantize_fp8_blockwise(x, 128, fmt="e4m3_pow2")
        np.testing.assert_array_equal(sc, rsc)
        np.testing.assert_array_equal(x8, r8)


def test_quantizer_every_rounding_class(fa):
    x = _rounding_class_blocks()
    x8, sc = _quant(fa, x, "e4m3_pow2")
    r8, rsc = oracle.quantize_fp8_blockwise(x, 128, fmt="e4m3_pow2")
    np.testing.assert_array_equal(sc, rsc)
    np.testing.assert_array_equal(x8, r8)


def test_quantizer_fp8_workload_v(fa):
    _, _, v = make_qkv(16, 16, 8192, 128, seed=0, outliers=True)
    x8, sc = _quant(fa, v, "e4m3_pow2")
    r8, rsc = oracle.quantize_fp8_blockwise(v, 128, fmt="e4m3_pow2")
    np.testing.assert_array_equal(sc, rsc)
    np.testing.assert_array_equal(x8, r8)


def _case(fa, q, k, v, causal, window, qk_fmt, heads=None, rows=None, v_fmt="e4m3_pow2"):
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d)
    q8, sq = fa.attn_quantize_fp8_blockwise_fmt(q.cuda(), qk_fmt)
    k8, sk = fa.attn_quantize_fp8_blockwise_fmt(k.cuda(), qk_fmt)
    v8, sv = fa.attn_quantize_fp8_blockwise_fmt(v.cuda(), v_fmt)
    o, lse = fa.attn_fwd_fp8_fmt(q8, k8, v8, sq, sk, sv, qk_fmt, v_fmt, scale=scale,
                                 causal=causal, window=window)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    rows = rows if rows is not None else list(range(N))
    deq = [oracle.dequantize(t8.cpu().numpy(), s.cpu().numpy(), 128,
                             fmt="e5m2" if (i < 2 and qk_fmt == "e5m2") else "e4m3")
           for i, (t8, s) in enumerate(((q8, sq), (k8, sk), (v8, sv)))]
    o_deq, lse_deq = oracle_rows(deq[0], deq[1], deq[2], heads, rows, scale, causal, window)
    o_unq, _ = oracle_rows(q, k, v, heads, rows, scale, causal, window)
    o_g = gather(o.cpu(), heads, rows)
    lse_g = gather(lse.cpu(), heads, rows)
    assert np.isfinite(o_g).all() and np.isfinite(lse_g).all()
    return {"vs_deq": rel_rmse(o_g, o_deq), "vs_unq": rel_rmse(o_g, o_unq),
            "lse_max_abs_vs_deq": float(np.abs(lse_g - lse_deq).max())}


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 300), (False, 300)])
@pytest.mark.parametrize("qk_fmt", ["e4m3", "e4m3_pow2"])
def test_pow2_v_attention_small(fa, causal, window, qk_fmt):
    q, k, v = make_qkv(2, 2, 1024, 128, seed=62, outliers=True)
    e = _case(fa, q, k, v, causal, window, qk_fmt)
    print("pow2 V", qk_fmt, causal, window, e)
    assert e["vs_deq"] <= FP8_REL_RMSE_DEQ, e
    assert e["lse_max_abs_vs_deq"] <= 2e-2, e


@pytest.mark.parametrize("direction", [1, -1])
def test_pow2_v_scales_rising_and_falling(fa, direction):
    """V blocks scaled by 2^(3 b) (rising: the reference scale grows every tile and O is
    rescaled) or 2^(-3 b) (falling: every tile's ratio goes into P's exponent, down to
    2^-21), causal and not.  The largest block dominates O, so only ~128 keys carry the
    output and the E4M3 rounding of P averages over fewer terms: the bar is the P-rounding
    bound 2^-4 / sqrt(3), and the error must stay within 1.25x of that of the per-tile
    exact descale path (plain E4M3 V) on the same input."""
    q, k, v = make_qkv(1, 2, 1024, 128, seed=63, outliers=False)
    f = torch.pow(2.0, direction * 3.0 * (torch.arange(1024) // 128).float())
    v = (v.float() * f[None, None, :, None]).to(torch.bfloat16)
    for causal in (False, True):
        e = _case(fa, q, k, v, causal, 0, "e4m3")
        ref = _case(fa, q, k, v, causal, 0, "e4m3", v_fmt="e4m3")
        print("pow2 V ramp", direction, causal, e, "plain E4M3 V:", ref)
        assert e["vs_deq"] <= 2.0 ** -4 / 3.0 ** 0.5, e
        assert e["vs_deq"] <= 1.25 * ref["vs_deq"] + 1e-3, (e, ref)


def test_pow2_v_attention_d256(fa):
    q, k, v = make_qkv(1, 2, 512, 256, seed=64, outliers=True)
    e = _case(fa, q, k, v, False, 0, "e4m3")
    assert e["vs_deq"] <= FP8_REL_RMSE_DEQ, e


@pytest.mark.parametrize("causal", [False, True])
def test_pow2_v_fp8_workload_sampled(fa, causal):
    q, k, v = make_qkv(16, 16, 8192, 128, seed=0, outliers=True)
    e = _case(fa, q, k, v, causal, 0, "e4m3", heads=sampled_heads(16, 16),
              rows=sampled_rows(8192, 96))
    print("pow2 V fp8 workload", causal, e)
    assert e["vs_deq"] <= FP8_REL_RMSE_DEQ, e


def test_bad_v_format_rejected(fa):
    lib = fa.load_library()
    z8 = torch.zeros(1, 1, 128, 128, dtype=torch.uint8, device="cuda")
    sc = torch.ones(1, 1, 1, dtype=torch.float32, device="cuda")
    o = torch.empty(1, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 1, 128, dtype=torch.float32, device="cuda")
    args = [z8.data_ptr(), z8.data_ptr(), z8.data_ptr(), sc.data_ptr(), sc.data_ptr(), sc.data_ptr(),
            o.data_ptr(), lse.data_ptr(), 1, 1, 128, 128, 0.1, 0, 0]
    assert lib.attn_fwd_fp8_fmt(*args, 0, 1, None) == fa.ATTN_ERR_INVALID_ARG   # V in E5M2
    assert lib.attn_fwd_fp8_fmt(*args, 5, 0, None) == fa.ATTN_ERR_INVALID_ARG
