"""GPU parity of head-dim-aware FP8 scaling: the quantiser at 64-row blocks bit for bit
against the oracle, and the FP8 forward (attn_fwd_fp8_blocks, d = 64 included) against
the oracle on the dequantised inputs.

"Warp Group Cluster 优化：Flash Attention V3 在 H100 上的 FP8 融合计算实践" §3 (头维度感知
量化): Q and K scale blocks of min(d, 128) rows, V blocks of 128 rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv, sampled_heads
from tests.attn_check import FP8_REL_RMSE_DEQ, LSE_MAX_ABS, gather, oracle_rows, rel_rmse
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

MASKS = [(False, 0), (True, 0), (True, 300), (False, 300)]


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def test_library_rule_matches_the_oracle(fa):
    for d in (64, 128, 256):
        assert fa.attn_fp8_qk_block_rows(d) == oracle.fp8_block_rows(d, "q") == \
            oracle.fp8_block_rows(d, "k")


@pytest.mark.parametrize("N,d", [(64, 64), (1000, 64), (300, 128), (77, 16), (1024, 256)])
def test_quantizer_64_row_blocks_bit_exact(fa, N, d):
    q, k, v = make_qkv(2, 3, N, d, seed=61, outliers=True)
    for x in (q, k, v):
        x8, sc = fa.attn_quantize_fp8_blockwise(x.cuda(), block=64)
        assert fa.attn_get_device_status() == fa.ATTN_OK
        r8, rsc = oracle.quantize_fp8_blockwise(x, 64)
        np.testing.assert_array_equal(sc.cpu().numpy(), rsc)
        np.testing.assert_array_equal(x8.cpu().numpy(), r8)


@pytest.mark.parametrize("fmt", ["e5m2", "e4m3_pow2"])
def test_quantizer_64_row_blocks_other_formats(fa, fmt):
    q, _, _ = make_qkv(1, 4, 640, 64, seed=62, outliers=True)
    x8, sc = fa.attn_quantize_fp8_blockwise_fmt(q.cuda(), fmt, block=64)
    r8, rsc = oracle.quantize_fp8_blockwise(q, 64, fmt=fmt)
    np.testing.assert_array_equal(sc.cpu().numpy(), rsc)
    np.testing.assert_array_equal(x8.cpu().numpy(), r8)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_rotated_quantizer_64_row_blocks(fa, d):
    q, _, _ = make_qkv(1, 3, 500, d, seed=63, outliers=True)
    x8, sc = fa.attn_quantize_fp8_hadamard(q.cuda(), block=64)
    r8, rsc = oracle.quantize_fp8_hadamard(q, 64)
    np.testing.assert_array_equal(sc.cpu().numpy(), rsc)
    np.testing.assert_array_equal(x8.cpu().numpy(), r8)


def _case(fa, B, H, N, d, causal, window, seed, qk_block, heads=None, rows=None):
    """Quantise Q, K with qk_block-row blocks and V with 128-row blocks, run the FP8
    forward, and compare with the oracle on the dequantised (and the unquantised) inputs."""
    q, k, v = make_qkv(B, H, N, d, seed=seed, outliers=True)
    scale = 1.0 / math.sqrt(d)
    q8, sq = fa.attn_quantize_fp8_blockwise(q.cuda(), block=qk_block)
    k8, sk = fa.attn_quantize_fp8_blockwise(k.cuda(), block=qk_block)
    v8, sv = fa.attn_quantize_fp8_blockwise(v.cuda(), block=128)
    o, lse = fa.attn_fwd_fp8_blocks(q8, k8, v8, sq, sk, sv, qk_block=qk_block, scale=scale,
                                    causal=causal, window=window)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    rows = rows if rows is not None else list(range(N))
    deq = []
    for t8, s, blk in ((q8, sq, qk_block), (k8, sk, qk_block), (v8, sv, 128)):
        t8c, sc = t8.cpu().numpy(), s.cpu().numpy()
        deq.append({(b, h): oracle.dequantize(t8c[b, h], sc[b, h], blk) for (b, h) in heads})
    o_deq, lse_deq = oracle_rows(deq[0], deq[1], deq[2], heads, rows, scale, causal, window)
    o_unq, _ = oracle_rows(q, k, v, heads, rows, scale, causal, window)
    o_g = gather(o.cpu(), heads, rows)
    lse_g = gather(lse.cpu(), heads, rows)
    assert np.isfinite(o_g).all() and np.isfinite(lse_g).all()
    return {"vs_deq": rel_rmse(o_g, o_deq), "vs_unq": rel_rmse(o_g, o_unq),
            "oracle_deq_vs_unq": rel_rmse(o_deq, o_unq),
            "lse_max_abs_vs_deq": float(np.abs(lse_g - lse_deq).max())}


@pytest.mark.parametrize("causal,window", MASKS)
@pytest.mark.parametrize("d,qk_block", [(64, 64), (64, 128), (128, 64), (256, 64)])
def test_forward_against_dequantised_oracle(fa, d, qk_block, causal, window):
    e = _case(fa, 2, 2, 1024, d, causal, window, seed=64, qk_block=qk_block)
    print(f"d={d} qk_block={qk_block} c={causal} w={window}:", e)
    assert e["vs_deq"] <= FP8_REL_RMSE_DEQ, e
    assert e["vs_unq"] <= e["oracle_deq_vs_unq"] + FP8_REL_RMSE_DEQ, e
    assert e["lse_max_abs_vs_deq"] <= LSE_MAX_ABS, e


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_workload_at_d64_all_rows_of_sampled_heads(fa, causal):
    """The FP8 workload's distribution at head dim 64 (B=16, H=16, N=8192, d=64), with
    head-dim-aware blocks: every row of four seeded heads."""
    heads = sampled_heads(16, 16)
    e = _case(fa, 16, 16, 8192, 64, causal, 0, seed=0, qk_block=64, heads=heads)
    print(f"fp8 d64 workload causal={causal}:", e)
    assert e["vs_deq"] <= FP8_REL_RMSE_DEQ, e
    assert e["vs_unq"] <= e["oracle_deq_vs_unq"] + FP8_REL_RMSE_DEQ, e
    assert e["lse_max_abs_vs_deq"] <= LSE_MAX_ABS, e


def test_head_dim_aware_blocks_lower_the_error_at_d64(fa):
    """Through the GPU path: at d = 64 on the FP8 workload's distribution, 64-row Q/K
    blocks give a lower error against unquantised attention than 128-row blocks."""
    e64 = _case(fa, 1, 8, 2048, 64, False, 0, seed=0, qk_block=64)
    e128 = _case(fa, 1, 8, 2048, 64, False, 0, seed=0, qk_block=128)
    print("d=64 vs unquantised: 64-row Q/K blocks", e64["vs_unq"], "128-row", e128["vs_unq"])
    assert e64["vs_unq"] < e128["vs_unq"]


def test_block_128_is_the_plain_fp8_forward(fa):
    """qk_block = 128 reproduces attn_fwd_fp8 bit for bit (the same kernel with equal
    descales for both 64-key halves of a tile)."""
    q, k, v = make_qkv(2, 2, 1024, 128, seed=65, outliers=True)
    qs = [fa.attn_quantize_fp8_blockwise(t.cuda()) for t in (q, k, v)]
    args = (qs[0][0], qs[1][0], qs[2][0], qs[0][1], qs[1][1], qs[2][1])
    for causal in (False, True):
        o1, l1 = fa.attn_fwd_fp8(*args, causal=causal)
        o2, l2 = fa.attn_fwd_fp8_blocks(*args, qk_block=128, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_descale_shapes_are_checked(fa):
    q, k, v = make_qkv(1, 1, 256, 64, seed=66)
    q8, sq = fa.attn_quantize_fp8_blockwise(q.cuda(), block=128)   # 2 blocks, 4 expected
    with pytest.raises(TypeError):
        fa.attn_fwd_fp8_blocks(q8, q8, q8, sq, sq, sq, qk_block=64)
