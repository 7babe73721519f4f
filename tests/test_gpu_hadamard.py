"""GPU parity of incoherent processing (attn_quantize_fp8_hadamard): codes and
scales bit for bit against the oracle's fp32 rotation + block quantiser, and the
FP8 forward pass on rotated Q, K against the oracle on the dequantised inputs."""
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


def _rot_gpu(fa, x):
    x8, sc = fa.attn_quantize_fp8_hadamard(x.cuda())
    assert fa.attn_get_device_status() == fa.ATTN_OK
    return x8.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("N,d", [(128, 128), (1000, 64), (1000, 128), (200, 256), (77, 64)])
def test_bit_exact_small(fa, N, d):
    q, k, _ = make_qkv(2, 3, N, d, seed=41, outliers=True)
    for x in (q, k):
        x8, sc = _rot_gpu(fa, x)
        r8, rsc = oracle.quantize_fp8_hadamard(x, 128)
        np.testing.assert_array_equal(sc, rsc)
        np.testing.assert_array_equal(x8, r8)


def test_wide_dynamic_range(fa):
    """Rows mixing magnitudes 2^-20 .. 2^12, so sums in the butterflies round."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(1, 2, 384, 128, generator=g)
    x = x * torch.pow(2.0, torch.randint(-20, 13, x.shape, generator=g).float())
    x = x.to(torch.bfloat16)
    x8, sc = _rot_gpu(fa, x)
    r8, rsc = oracle.quantize_fp8_hadamard(x, 128)
    np.testing.assert_array_equal(sc, rsc)
    np.testing.assert_array_equal(x8, r8)


def test_zero_and_one_hot_rows(fa):
    """A zero block keeps scale 1 and zero codes.  In a block of one-hot rows every
    rotated value is +-1/sqrt(d), the block amax, so every code is +-448 with the
    sign pattern of the Hadamard matrix row."""
    d = 128
    x = torch.zeros(1, 1, 256, d, dtype=torch.bfloat16)
    for r in range(128, 256):
        x[0, 0, r, r - 128] = 1.0
    x8, sc = _rot_gpu(fa, x)
    assert sc[0, 0, 0] == 1.0 and (x8[0, 0, :128] == 0).all()
    assert sc[0, 0, 1] == np.float32(oracle.hadamard_scale(d)) / np.float32(448.0)
    k = np.arange(d)[:, None]
    j = np.arange(d)[None, :]
    neg = np.vectorize(lambda a: bin(a).count("1") & 1)(k & j).astype(bool)
    np.testing.assert_array_equal(x8[0, 0, 128:], np.where(neg, 0xFE, 0x7E).astype(np.uint8))


def test_bit_exact_fp8_workload_sampled_heads(fa):
    """FP8 workload tensors (B=16, H=16, N=8192, d=128, 0.1% outliers x20), rotated on
    the GPU in full; four seeded heads compared with the oracle."""
    q, k, _ = make_qkv(16, 16, 8192, 128, seed=0, outliers=True)
    heads = sampled_heads(16, 16)
    for x in (q, k):
        x8, sc = _rot_gpu(fa, x)
        for (b, h) in heads:
            r8, rsc = oracle.quantize_fp8_hadamard(x[b, h][None], 128)
            np.testing.assert_array_equal(sc[b, h], rsc[0])
            np.testing.assert_array_equal(x8[b, h], r8[0])


def _rotated_case(fa, B, H, N, d, causal, window, seed, heads=None, rows=None):
    q, k, v = make_qkv(B, H, N, d, seed=seed, outliers=True)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    rows = rows if rows is not None else list(range(N))
    o_unq, _ = oracle_rows(q, k, v, heads, rows, scale, causal, window)
    v8, sv = fa.attn_quantize_fp8_blockwise(vd)
    vdeq = oracle.dequantize(v8.cpu().numpy(), sv.cpu().numpy(), 128)
    out = {}
    for name, quant in (("block", fa.attn_quantize_fp8_blockwise),
                        ("hadamard", fa.attn_quantize_fp8_hadamard)):
        q8, sq = quant(qd)
        k8, sk = quant(kd)
        o, lse = fa.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, scale=scale, causal=causal,
                                 window=window)
        assert fa.attn_get_device_status() == fa.ATTN_OK
        qdeq = oracle.dequantize(q8.cpu().numpy(), sq.cpu().numpy(), 128)
        kdeq = oracle.dequantize(k8.cpu().numpy(), sk.cpu().numpy(), 128)
        o_deq, lse_deq = oracle_rows(qdeq, kdeq, vdeq, heads, rows, scale, causal, window)
        o_g = gather(o.cpu(), heads, rows)
        lse_g = gather(lse.cpu(), heads, rows)
        assert np.isfinite(o_g).all() and np.isfinite(lse_g).all()
        out[name] = {"vs_deq": rel_rmse(o_g, o_deq), "vs_unq": rel_rmse(o_g, o_unq),
                     "lse_max_abs_vs_deq": float(np.abs(lse_g - lse_deq).max())}
    return out


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 300)])
def test_fp8_attention_on_rotated_inputs(fa, causal, window):
    e = _rotated_case(fa, 2, 2, 1024, 128, causal, window, seed=43)
    print("rotated small", causal, window, e)
    assert e["hadamard"]["vs_deq"] <= FP8_REL_RMSE_DEQ, e
    assert e["hadamard"]["lse_max_abs_vs_deq"] <= 2e-2, e
    # incoherent processing lowers the error against the unquantised inputs
    assert e["hadamard"]["vs_unq"] < 0.8 * e["block"]["vs_unq"], e


def test_fp8_attention_rotated_d256(fa):
    e = _rotated_case(fa, 1, 2, 512, 256, False, 0, seed=44)
    assert e["hadamard"]["vs_deq"] <= 2.0 ** -4 / 3.0 ** 0.5, e
    assert e["hadamard"]["vs_unq"] < e["block"]["vs_unq"], e


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_workload_rotated_sampled(fa, causal):
    """FP8 workload (B=16, H=16, N=8192, d=128, outliers): 4 heads x 96 rows."""
    e = _rotated_case(fa, 16, 16, 8192, 128, causal, 0, seed=0, heads=sampled_heads(16, 16),
                      rows=sampled_rows(8192, 96))
    print("rotated fp8 workload", causal, e)
    assert e["hadamard"]["vs_deq"] <= FP8_REL_RMSE_DEQ, e
    assert e["hadamard"]["vs_unq"] < 0.8 * e["block"]["vs_unq"], e
