"""GPU parity of attn_fwd_bf16_varlen (packed variable-length sequences) against the
float64 oracle, and against the batched kernel when every length is equal."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import (make_packed_qkv, make_qkv, sampled_rows,
                                             varlen_lengths)
from tests.attn_check import assert_bf16_close
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

MASKS = [(False, 0), (True, 0), (False, 100), (True, 100)]


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _run(fa, q, k, v, cu, scale, causal, window, max_len=None):
    lens = (cu[1:] - cu[:-1]).tolist()
    max_len = max(lens) if max_len is None else max_len
    o, lse = fa.attn_fwd_bf16_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max_len, scale=scale,
                                     causal=causal, window=window)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal,window", MASKS)
def test_ragged_lengths_all_rows(fa, d, causal, window):
    lengths = [300, 1, 0, 129, 1000, 128, 127, 255, 2]
    q, k, v, cu = make_packed_qkv(lengths, 3, d, seed=51)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, cu, scale, causal, window)
    o_ref, lse_ref = oracle.attn_varlen_f64(q, k, v, cu.numpy(), scale, causal=causal, window=window)
    assert_bf16_close(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref,
                      f"varlen d={d} c={causal} w={window}")


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_bit_identical_to_batched(fa, causal):
    """Same tiles, same arithmetic: the packed call reproduces the batched one bit for bit."""
    B, H, N, d = 3, 4, 1000, 128
    q, k, v = make_qkv(B, H, N, d, seed=52)
    ob, lb = fa.attn_fwd_bf16(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    pack = lambda x: x.permute(0, 2, 1, 3).reshape(B * N, H, d).contiguous()
    cu = torch.arange(B + 1, dtype=torch.int32) * N
    ov, lv = _run(fa, pack(q), pack(k), pack(v), cu, 1.0 / math.sqrt(d), causal, 0)
    assert torch.equal(ov, pack(ob.cpu()))
    assert torch.equal(lv, lb.cpu().permute(1, 0, 2).reshape(H, B * N))


def test_larger_max_seqlen_and_empty_sequences(fa):
    lengths = [0, 0, 200, 0, 17]
    q, k, v, cu = make_packed_qkv(lengths, 2, 128, seed=53)
    o, lse = _run(fa, q, k, v, cu, 0.1, True, 0, max_len=217)  # more slots than needed
    o_ref, lse_ref = oracle.attn_varlen_f64(q, k, v, cu.numpy(), 0.1, causal=True)
    assert_bf16_close(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref, "empty seqs")


def test_zero_tokens_and_bad_arguments(fa):
    e = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    cu0 = torch.zeros(2, dtype=torch.int32, device="cuda")
    o, lse = fa.attn_fwd_bf16_varlen(e, e, e, cu0, 0)
    assert o.shape == (0, 2, 64) and lse.shape == (2, 0)
    q, k, v, cu = make_packed_qkv([5, 6], 2, 64, seed=54)
    with pytest.raises(fa.AttnError):   # max_seqlen > T is rejected before any launch
        fa.attn_fwd_bf16_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), 100)


@pytest.mark.parametrize("causal", [False, True])
def test_mixed_lengths_at_headline_token_count(fa, causal):
    """131072 tokens (the headline's B*N) as lengths uniform in [512, 16384], H=16, d=128;
    four sequences x all heads' sampled rows against the oracle."""
    lengths = varlen_lengths(16 * 8192, 512, 16384, seed=3)
    H, d = 16, 128
    q, k, v, cu = make_packed_qkv(lengths, H, d, seed=0)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(fa, q, k, v, cu, scale, causal, 0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    seqs = [0, len(lengths) - 1, int(np.argmax(lengths)), len(lengths) // 2]
    for s in seqs:
        a, b = int(cu[s]), int(cu[s + 1])
        n = b - a
        rows = sampled_rows(n, 48)
        for h in (0, H - 1, 7):
            o_ref, l_ref = oracle.attn_rows_f64(q[a:b, h], k[a:b, h], v[a:b, h], rows, scale,
                                                causal=causal)
            o_g = o[a:b, h][rows].double().numpy()
            l_g = lse[h, a:b][rows].double().numpy()
            assert_bf16_close(o_g, l_g, o_ref, l_ref, f"seq {s} (n={n}) head {h}")


@pytest.mark.parametrize("causal", [False, True])
def test_more_sequences_than_the_schedule_table(fa, causal):
    """Up to 220 sequences are scheduled longest first from a table each CTA sorts; more
    fall back to the round-robin over pair slots.  Both paths against the oracle, and
    both bit-identical to a call on the same sequences one at a time."""
    g = torch.Generator().manual_seed(55)
    for count in (219, 221, 300):
        lengths = torch.randint(0, 300, (count,), generator=g).tolist()
        lengths[count // 2] = 700                  # one long sequence among short ones
        q, k, v, cu = make_packed_qkv(lengths, 2, 64, seed=56)
        o, lse = _run(fa, q, k, v, cu, 0.125, causal, 0)
        o_ref, lse_ref = oracle.attn_varlen_f64(q, k, v, cu.numpy(), 0.125, causal=causal)
        assert_bf16_close(o.double().numpy(), lse.double().numpy(), o_ref, lse_ref,
                          f"{count} sequences causal={causal}")
        s = count // 2
        a, b = int(cu[s]), int(cu[s + 1])
        one = torch.tensor([0, b - a], dtype=torch.int32)
        o1, l1 = _run(fa, q[a:b].contiguous(), k[a:b].contiguous(), v[a:b].contiguous(), one,
                      0.125, causal, 0)
        assert torch.equal(o[a:b], o1) and torch.equal(lse[:, a:b], l1)
