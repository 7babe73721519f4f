"""GPU parity of the second FP8 format: attn_quantize_fp8_blockwise_fmt into E5M2
bit for bit against the oracle's codec and quantiser, and attn_fwd_fp8_fmt with Q, K
in E5M2 (V in E4M3) against the oracle on the dequantised inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv, sampled_heads, sampled_rows
from tests.attn_check import FP8_REL_RMSE_DEQ, gather, oracle_rows, rel_rmse
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _quant_gpu(fa, x, fmt="e5m2"):
    x8, sc = fa.attn_quantize_fp8_blockwise_fmt(x.cuda(), fmt)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    return x8.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("N,d", [(128, 128), (1000, 64), (1000, 128), (300, 256), (77, 16)])
def test_quantizer_bit_exact_small(fa, N, d):
    q, k, v = make_qkv(2, 3, N, d, seed=51, outliers=True)
    for x in (q, k, v):
        x8, sc = _quant_gpu(fa, x)
        r8, rsc = oracle.quantize_fp8_blockwise(x, 128, fmt="e5m2")
        np.testing.assert_array_equal(sc, rsc)
        np.testing.assert_array_equal(x8, r8)


def _rounding_class_blocks():
    """One 128 x 128 block per (amax exponent E, amax mantissa m_a): element 0 is
    amax = (1 + m_a/128) 2^E, then +-(1 + m_x/128) 2^e for every bf16 mantissa m_x and
    e = E-32 .. E, the rest zero.  x / scale runs over every mantissa pair at every
    exponent offset from below the E5M2 subnormals (2^-16 of 57344 is 2^-31.8 of amax)
    up to 57344, so every rounding decision of the quotient and of the conversion is
    exercised."""
    blocks = []
    for E in (-5, 3, 11):
        for ma in range(128):
            amax = (1.0 + ma / 128.0) * 2.0 ** E
            vals = [amax]
            for e in range(E - 32, E + 1):
                for mx in range(128):
                    x = (1.0 + mx / 128.0) * 2.0 ** e
                    if x <= amax:
                        vals += [x, -x]
            blk = np.zeros(128 * 128, dtype=np.float32)
            blk[:len(vals)] = vals
            blocks.append(blk.reshape(128, 128))
    x = torch.from_numpy(np.stack(blocks))[None]
    assert torch.equal(x.to(torch.bfloat16).float(), x)
    return x.to(torch.bfloat16)


def test_quantizer_every_rounding_class(fa):
    x = _rounding_class_blocks()
    x8, sc = _quant_gpu(fa, x)
    r8, rsc = oracle.quantize_fp8_blockwise(x, 128, fmt="e5m2")
    np.testing.assert_array_equal(sc, rsc)
    np.testing.assert_array_equal(x8, r8)


def test_quantizer_zero_block_and_top_code(fa):
    x = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16)
    x[0, 0, 200, 5] = -3.0
    x8, sc = _quant_gpu(fa, x)
    assert sc[0, 0, 0] == 1.0 and (x8[0, 0, :128] == 0).all()
    assert sc[0, 0, 1] == np.float32(3.0) / np.float32(57344.0)
    assert x8[0, 0, 200, 5] == 0xFB                        # -57344


def test_quantizer_bit_exact_fp8_workload(fa):
    """FP8 workload tensors (B=16, H=16, N=8192, d=128, 0.1% outliers x20), Q and K."""
    q, k, _ = make_qkv(16, 16, 8192, 128, seed=0, outliers=True)
    for x in (q, k):
        x8, sc = _quant_gpu(fa, x)
        r8, rsc = oracle.quantize_fp8_blockwise(x, 128, fmt="e5m2")
        np.testing.assert_array_equal(sc, rsc)
        np.testing.assert_array_equal(x8, r8)


def test_e4m3_format_is_the_plain_entry(fa):
    q, k, v = make_qkv(1, 2, 512, 128, seed=52, outliers=True)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    a8, asc = fa.attn_quantize_fp8_blockwise(qd)
    b8, bsc = fa.attn_quantize_fp8_blockwise_fmt(qd, "e4m3")
    assert torch.equal(a8, b8) and torch.equal(asc, bsc)
    qs = [fa.attn_quantize_fp8_blockwise(t) for t in (qd, kd, vd)]
    o1, l1 = fa.attn_fwd_fp8(qs[0][0], qs[1][0], qs[2][0], qs[0][1], qs[1][1], qs[2][1], causal=True)
    o2, l2 = fa.attn_fwd_fp8_fmt(qs[0][0], qs[1][0], qs[2][0], qs[0][1], qs[1][1], qs[2][1], "e4m3",
                                 causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bad_format_rejected(fa):
    x = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.attn_quantize_fp8_blockwise_fmt(x, "e3m4")
    lib = fa.load_library()
    x8 = torch.empty(1, 1, 128, 128, dtype=torch.uint8, device="cuda")
    sc = torch.empty(1, 1, 1, dtype=torch.float32, device="cuda")
    st = lib.attn_quantize_fp8_blockwise_fmt(x.data_ptr(), x8.data_ptr(), sc.data_ptr(), 1, 1, 128,
                                             128, 128, 7, None)
    assert st == fa.ATTN_ERR_INVALID_ARG


def _mixed_case(fa, B, H, N, d, causal, window, seed, heads=None, rows=None):
    q, k, v = make_qkv(B, H, N, d, seed=seed, outliers=True)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    rows = rows if rows is not None else list(range(N))
    v8, sv = fa.attn_quantize_fp8_blockwise(vd)
    vdeq = oracle.dequantize(v8.cpu().numpy(), sv.cpu().numpy(), 128)
    o_unq, _ = oracle_rows(q, k, v, heads, rows, scale, causal, window)
    out = {}
    for fmt in ("e4m3", "e5m2"):
        q8, sq = fa.attn_quantize_fp8_blockwise_fmt(qd, fmt)
        k8, sk = fa.attn_quantize_fp8_blockwise_fmt(kd, fmt)
        o, lse = fa.attn_fwd_fp8_fmt(q8, k8, v8, sq, sk, sv, fmt, scale=scale, causal=causal,
                                     window=window)
        assert fa.attn_get_device_status() == fa.ATTN_OK
        qdeq = oracle.dequantize(q8.cpu().numpy(), sq.cpu().numpy(), 128, fmt=fmt)
        kdeq = oracle.dequantize(k8.cpu().numpy(), sk.cpu().numpy(), 128, fmt=fmt)
        o_deq, lse_deq = oracle_rows(qdeq, kdeq, vdeq, heads, rows, scale, causal, window)
        o_g = gather(o.cpu(), heads, rows)
        lse_g = gather(lse.cpu(), heads, rows)
        assert np.isfinite(o_g).all() and np.isfinite(lse_g).all()
        out[fmt] = {"vs_deq": rel_rmse(o_g, o_deq), "vs_unq": rel_rmse(o_g, o_unq),
                    "lse_max_abs_vs_deq": float(np.abs(lse_g - lse_deq).max())}
    return out


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 300), (False, 300)])
def test_qk_e5m2_attention_small(fa, causal, window):
    e = _mixed_case(fa, 2, 2, 1024, 128, causal, window, seed=53)
    print("qk e5m2 small", causal, window, e)
    assert e["e5m2"]["vs_deq"] <= FP8_REL_RMSE_DEQ, e
    assert e["e5m2"]["lse_max_abs_vs_deq"] <= 2e-2, e


def test_qk_e5m2_attention_d256(fa):
    e = _mixed_case(fa, 1, 2, 512, 256, False, 0, seed=54)
    assert e["e5m2"]["vs_deq"] <= FP8_REL_RMSE_DEQ, e


@pytest.mark.parametrize("causal", [False, True])
def test_qk_e5m2_fp8_workload_sampled(fa, causal):
    """FP8 workload (B=16, H=16, N=8192, d=128, outliers): 4 heads x 96 rows."""
    e = _mixed_case(fa, 16, 16, 8192, 128, causal, 0, seed=0, heads=sampled_heads(16, 16),
                    rows=sampled_rows(8192, 96))
    print("qk e5m2 fp8 workload", causal, e)
    assert e["e5m2"]["vs_deq"] <= FP8_REL_RMSE_DEQ, e
