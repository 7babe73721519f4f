"""GPU parity of attn_fwd_bf16 (through the C ABI) against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv, sampled_heads, sampled_rows
from tests.attn_check import assert_bf16_close, gather, oracle_rows
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

MASKS = [(False, 0), (True, 0), (False, 100), (True, 100)]


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _run(fa, q, k, v, scale, causal, window):
    o, lse = fa.attn_fwd_bf16(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal,
                              window=window)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    return o.cpu(), lse.cpu()


def _full_check(fa, q, k, v, scale, causal, window, label):
    o, lse = _run(fa, q, k, v, scale, causal, window)
    o_ref, lse_ref = oracle.attn_f64(q, k, v, scale, causal=causal, window=window)
    return assert_bf16_close(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref, label)


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(fa, causal):
    """B=1, H=2, N=128, d=64, seed 0, scale 1/8: every output against the oracle."""
    q, k, v = make_qkv(1, 2, 128, 64, seed=0)
    _full_check(fa, q, k, v, 1.0 / 8.0, causal, 0, f"tiny causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal,window", MASKS)
def test_multi_tile_ragged(fa, d, causal, window):
    """Several query blocks and key tiles with a ragged tail (N = 1000)."""
    q, k, v = make_qkv(2, 2, 1000, d, seed=3)
    _full_check(fa, q, k, v, 1.0 / math.sqrt(d), causal, window, f"d={d} c={causal} w={window}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", [1, 31, 32, 33, 127, 129])
def test_narrow_windows(fa, d, window):
    """Windows around the 32-key chunk and the 128-key tile: the edge tiles' chunks are
    allowed for every row of a warp, masked for every row, or mixed, in every combination;
    N = 600 leaves a ragged last tile.  V is scaled by 1/4 (exact in bf16): with a window of
    a few keys O is nearly one V row, and the absolute bf16 bars assume O averages many rows;
    a masking error still moves O by the size of a V row."""
    q, k, v = make_qkv(1, 2, 600, d, seed=40 + window)
    v = v * 0.25
    for causal in (False, True):
        _full_check(fa, q, k, v, 1.0 / math.sqrt(d), causal, window, f"d={d} w={window} c={causal}")


@pytest.mark.parametrize("N", [1, 7, 129, 255, 257, 513])
def test_small_and_odd_lengths(fa, N):
    q, k, v = make_qkv(1, 3, N, 128, seed=N)
    for causal, window in MASKS:
        _full_check(fa, q, k, v, 0.09, causal, window, f"N={N} c={causal} w={window}")


def test_zero_query_gives_mean_of_values(fa):
    B, H, N, d = 1, 2, 300, 128
    _, k, v = make_qkv(B, H, N, d, seed=5)
    q = torch.zeros_like(k)
    for causal, window in MASKS:
        o, lse = _run(fa, q, k, v, 0.1, causal, window)
        vv = v.double()
        for i in (0, 1, 150, 299):
            js = [j for j in range(N) if oracle.key_allowed(i, j, N, causal, window)]
            ref = vv[:, :, js].mean(dim=2)
            assert (o[:, :, i].double() - ref).abs().max() <= 1e-2
            assert (lse[:, :, i].double() - math.log(len(js))).abs().max() <= 1e-5


def test_causal_row_zero_is_exactly_first_value_row(fa):
    q, k, v = make_qkv(2, 2, 640, 64, seed=6)
    for window in (0, 37):
        o, lse = _run(fa, q, k, v, 0.125, True, window)
        assert torch.equal(o[:, :, 0], v[:, :, 0])
        ref = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) * 0.125
        assert (lse[:, :, 0].double() - ref).abs().max() <= 1e-4


@pytest.mark.parametrize("causal", [False, True])
def test_config_n2048_sampled_heads(fa, causal):
    """B=16, H=16, N=2048, d=128: all rows of four seeded heads."""
    B, H, N, d = 16, 16, 2048, 128
    q, k, v = make_qkv(B, H, N, d, seed=0)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, scale, causal, 0)
    heads = sampled_heads(B, H)
    rows = list(range(N))
    o_ref, lse_ref = oracle_rows(q, k, v, heads, rows, scale, causal, 0)
    assert_bf16_close(gather(o, heads, rows), gather(lse, heads, rows), o_ref, lse_ref,
                      f"N2048 causal={causal}")
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True])
def test_headline_n8192_all_rows_of_sampled_heads(fa, causal):
    """B=16, H=16, N=8192, d=128: every row of four seeded heads ((0,0), (15,15) and
    two drawn from Generator(1)) against the oracle."""
    B, H, N, d = 16, 16, 8192, 128
    q, k, v = make_qkv(B, H, N, d, seed=0)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, scale, causal, 0)
    heads = sampled_heads(B, H)
    rows = list(range(N))
    o_ref, lse_ref = oracle_rows(q, k, v, heads, rows, scale, causal, 0)
    e = assert_bf16_close(gather(o, heads, rows), gather(lse, heads, rows), o_ref, lse_ref,
                          f"N8192 causal={causal}")
    print(f"headline bf16 causal={causal} ({len(heads)} heads x {N} rows):", e)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


SWEEP = [(d, N) for d in (64, 128, 256) for N in (512, 1024, 2048, 4096, 8192, 16384)]


@pytest.mark.parametrize("d,N", SWEEP)
def test_sweep(fa, d, N):
    """B*N = 16384 tokens, H = 2048/d; non-causal, causal, causal window 1024.
    From N = 2048 on, every row of head (0, 0) is checked, plus 48 sampled rows of a
    second seeded head; shorter points check every row of both heads."""
    B, H = 16384 // N, 2048 // d
    q, k, v = make_qkv(B, H, N, d, seed=7)
    scale = 1.0 / math.sqrt(d)
    heads = sampled_heads(B, H, count=2)
    full = list(range(N))
    plan = [([heads[0]], full), ([heads[1]], full if N < 2048 else sampled_rows(N, 48))]
    for causal, window in [(False, 0), (True, 0), (True, 1024)]:
        o, lse = _run(fa, q, k, v, scale, causal, window)
        for hs, rows in plan:
            o_ref, lse_ref = oracle_rows(q, k, v, hs, rows, scale, causal, window)
            assert_bf16_close(gather(o, hs, rows), gather(lse, hs, rows), o_ref, lse_ref,
                              f"sweep d={d} N={N} c={causal} w={window} heads={hs} rows={len(rows)}")
        assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("d,H", [(128, 16), (256, 8)])
def test_result_does_not_depend_on_the_walk(fa, d, H):
    """B2 at N = 8192 has 512 query-block pairs, which the CTAs walk as single units; each
    batch alone (256 pairs) is walked as pairs.  A unit's result depends only on its inputs,
    so the two launches agree bit for bit."""
    q, k, v = make_qkv(2, H, 8192, d, seed=11)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / math.sqrt(d)
    o2, l2 = fa.attn_fwd_bf16(qd, kd, vd, scale=scale)
    for b in range(2):
        o1, l1 = fa.attn_fwd_bf16(qd[b:b + 1].contiguous(), kd[b:b + 1].contiguous(),
                                  vd[b:b + 1].contiguous(), scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(o1[0], o2[b]) and torch.equal(l1[0], l2[b])
    assert fa.attn_get_device_status() == fa.ATTN_OK


def test_repeated_calls_are_deterministic(fa):
    q, k, v = make_qkv(2, 4, 1024, 128, seed=9)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fa.attn_fwd_bf16(qd, kd, vd, causal=True)
    o2, l2 = fa.attn_fwd_bf16(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_runs_on_a_side_stream(fa):
    q, k, v = make_qkv(1, 2, 512, 64, seed=10)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o, lse = fa.attn_fwd_bf16(qd, kd, vd, stream=s)
    s.synchronize()
    o_ref, lse_ref = oracle.attn_f64(q, k, v, 0.125)
    assert_bf16_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref)
