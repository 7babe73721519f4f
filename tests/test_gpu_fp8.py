"""GPU parity of the FP8 path: the block quantiser bit for bit against the oracle's
quantiser, and attn_fwd_fp8 against the oracle on the dequantised inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv, sampled_heads
from tests.attn_check import (FP8_P_ROUNDING_BOUND, FP8_REL_RMSE_DEQ, fp8_lse_bound, gather,
                              oracle_rows, rel_rmse)
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _quant_gpu(fa, x):
    x8, sc = fa.attn_quantize_fp8_blockwise(x.cuda())
    assert fa.attn_get_device_status() == fa.ATTN_OK
    return x8.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("N,d", [(128, 128), (1000, 64), (1000, 128), (300, 256), (77, 16)])
def test_quantizer_bit_exact_small(fa, N, d):
    q, k, v = make_qkv(2, 3, N, d, seed=21, outliers=True)
    for x in (q, k, v):
        x8, sc = _quant_gpu(fa, x)
        r8, rsc = oracle.quantize_fp8_blockwise(x, 128)
        np.testing.assert_array_equal(sc, rsc)
        np.testing.assert_array_equal(x8, r8)


def _rounding_class_blocks():
    """One 128 x 128 block per (amax exponent E, amax mantissa m_a): element 0 is
    amax = (1 + m_a/128) 2^E, then +-(1 + m_x/128) 2^e for every bf16 mantissa m_x
    and e = E-20 .. E (not above amax), the rest zero.  x / scale then runs over
    every mantissa pair at every exponent offset, from the E4M3 subnormal range
    (and below it) up to 448, so every rounding decision of the quotient and of
    the E4M3 conversion is exercised."""
    blocks = []
    for E in (-3, 2, 9):
        for ma in range(128):
            amax = (1.0 + ma / 128.0) * 2.0 ** E
            vals = [amax]
            for e in range(E - 20, E + 1):
                for mx in range(128):
                    x = (1.0 + mx / 128.0) * 2.0 ** e
                    if x <= amax:
                        vals += [x, -x]
            blk = np.zeros(128 * 128, dtype=np.float32)
            blk[:len(vals)] = vals
            blocks.append(blk.reshape(128, 128))
    x = torch.from_numpy(np.stack(blocks))[None]          # [1, 384, 128, 128]
    assert torch.equal(x.to(torch.bfloat16).float(), x)   # every value is a bf16
    return x.to(torch.bfloat16)


def test_quantizer_every_rounding_class(fa):
    """The GPU quotient (reciprocal plus one FMA residual correction) and E4M3
    conversion match the oracle's IEEE division bit for bit on every pair of
    bf16 mantissas."""
    x = _rounding_class_blocks()
    x8, sc = _quant_gpu(fa, x)
    r8, rsc = oracle.quantize_fp8_blockwise(x, 128)
    np.testing.assert_array_equal(sc, rsc)
    np.testing.assert_array_equal(x8, r8)


def test_quantizer_zero_block(fa):
    x = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16)
    x[0, 0, 200, 5] = 3.0
    x8, sc = _quant_gpu(fa, x)
    r8, rsc = oracle.quantize_fp8_blockwise(x, 128)
    np.testing.assert_array_equal(sc, rsc)
    np.testing.assert_array_equal(x8, r8)
    assert sc[0, 0, 0] == 1.0


def test_quantizer_bit_exact_headline(fa):
    """FP8 workload tensors: B=16, H=16, N=8192, d=128, 0.1% outliers x20."""
    q, k, v = make_qkv(16, 16, 8192, 128, seed=0, outliers=True)
    for x in (q, k, v):
        x8, sc = _quant_gpu(fa, x)
        r8, rsc = oracle.quantize_fp8_blockwise(x, 128)
        np.testing.assert_array_equal(sc, rsc)
        np.testing.assert_array_equal(x8, r8)


def _fp8_case(fa, B, H, N, d, causal, window, seed, heads=None, rows=None, outliers=True):
    q, k, v = make_qkv(B, H, N, d, seed=seed, outliers=outliers)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    q8, sq = fa.attn_quantize_fp8_blockwise(qd)
    k8, sk = fa.attn_quantize_fp8_blockwise(kd)
    v8, sv = fa.attn_quantize_fp8_blockwise(vd)
    o, lse = fa.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, scale=scale, causal=causal, window=window)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    o = o.cpu()
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    rows = rows if rows is not None else list(range(N))
    # oracle (ii): the dequantised FP8 inputs the kernel actually consumed (only the
    # checked heads are dequantised; the dict is indexed by (b, h) like the tensors)
    deq = []
    for t8, s in ((q8, sq), (k8, sk), (v8, sv)):
        t8c, sc = t8.cpu().numpy(), s.cpu().numpy()
        deq.append({(b, h): oracle.dequantize(t8c[b, h], sc[b, h], 128) for (b, h) in heads})
    o_deq, lse_deq = oracle_rows(deq[0], deq[1], deq[2], heads, rows, scale, causal, window)
    # oracle (i): the unquantised bf16 inputs
    o_unq, _ = oracle_rows(q, k, v, heads, rows, scale, causal, window)
    o_g = gather(o, heads, rows)
    lse_g = gather(lse.cpu(), heads, rows)
    assert np.isfinite(o_g).all() and np.isfinite(lse_g).all()
    return {
        "vs_deq": rel_rmse(o_g, o_deq),
        "vs_unq": rel_rmse(o_g, o_unq),
        "oracle_deq_vs_unq": rel_rmse(o_deq, o_unq),
        "lse_max_abs_vs_deq": float(np.abs(lse_g - lse_deq).max()),
        "lse_bound_ratio": float((np.abs(lse_g - lse_deq) / fp8_lse_bound(lse_deq)).max()),
        "rows_checked": int(len(heads) * len(rows)),
    }


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 300), (False, 300)])
def test_fp8_attention_small(fa, causal, window):
    e = _fp8_case(fa, 2, 2, 1024, 128, causal, window, seed=31)
    assert e["vs_deq"] <= FP8_REL_RMSE_DEQ, e
    # the rest of the error against the unquantised inputs is the quantiser's
    assert e["vs_unq"] <= e["oracle_deq_vs_unq"] + FP8_REL_RMSE_DEQ, e
    assert e["lse_bound_ratio"] <= 1.0, e


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_attention_d256(fa, causal):
    """d = 256 on the FP8 workload's distribution at N = 512 (measured 0.73 % non-causal,
    1.03 % causal over all rows: a causal row i averages P's E4M3 rounding over only i + 1
    keys), so the bound here is that rounding's RMS."""
    e = _fp8_case(fa, 1, 2, 512, 256, causal, 0, seed=32)
    print(f"fp8 d256 causal={causal}:", e)
    assert e["vs_deq"] <= FP8_P_ROUNDING_BOUND, e
    assert e["vs_unq"] <= e["oracle_deq_vs_unq"] + FP8_P_ROUNDING_BOUND, e
    assert e["lse_bound_ratio"] <= 1.0, e


def test_fp8_attention_without_outliers(fa):
    """Spread attention (no outliers, not one of the FP8 workload's cases): O averages many
    V rows and is small, so P's E4M3 rounding (up to 2^-4 relative per element) shows in the
    relative error almost undiminished; the bound is that rounding's RMS."""
    e = _fp8_case(fa, 1, 4, 1024, 128, False, 0, seed=33, outliers=False)
    print("fp8 without outliers:", e)
    assert e["vs_deq"] <= FP8_P_ROUNDING_BOUND, e


def test_fp8_closed_form_zero_query(fa):
    """Q = 0: every allowed key gets the same weight, so O is the mean of the
    dequantised V rows and P = 1 is exact in E4M3."""
    B, H, N, d = 1, 2, 512, 128
    _, k, v = make_qkv(B, H, N, d, seed=34, outliers=True)
    q = torch.zeros_like(k)
    qs = [fa.attn_quantize_fp8_blockwise(t.cuda()) for t in (q, k, v)]
    o, lse = fa.attn_fwd_fp8(qs[0][0], qs[1][0], qs[2][0], qs[0][1], qs[1][1], qs[2][1],
                             scale=0.1, causal=True)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    vdeq = oracle.dequantize(qs[2][0].cpu().numpy(), qs[2][1].cpu().numpy(), 128)
    o = o.cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    for i in (0, 1, 127, 128, 300, 511):
        ref = vdeq[:, :, :i + 1].mean(axis=2)
        assert np.abs(o[:, :, i] - ref).max() <= 1e-2 * max(1.0, np.abs(ref).max())
        assert np.abs(lse[:, :, i] - math.log(i + 1)).max() <= 1e-5


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_attention_headline_all_rows_of_sampled_heads(fa, causal):
    """FP8 workload: B=16, H=16, N=8192, d=128 with outliers; every row of four seeded
    heads against the oracle on the dequantised inputs (O and LSE) and, reported, on
    the unquantised inputs."""
    heads = sampled_heads(16, 16)
    e = _fp8_case(fa, 16, 16, 8192, 128, causal, 0, seed=0, heads=heads, rows=list(range(8192)))
    print(f"fp8 headline causal={causal}:", e)
    assert e["rows_checked"] == 4 * 8192
    assert e["vs_deq"] <= FP8_REL_RMSE_DEQ, e
    assert e["vs_unq"] <= e["oracle_deq_vs_unq"] + FP8_REL_RMSE_DEQ, e
    assert e["lse_bound_ratio"] <= 1.0, e
