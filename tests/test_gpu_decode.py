"""GPU parity of attn_decode_bf16_paged (a decoding step over a paged KV cache)
against the float64 oracle, with automatic and forced key splits."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_paged_cache
from tests.attn_check import assert_bf16_close
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _check(fa, lens, H, nq, d, ps, splits, seed, label):
    q, kc, vc, pt, sl = make_paged_cache(lens, H, nq, d, ps, seed=seed)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.attn_decode_bf16_paged(q.cuda(), kc.cuda(), vc.cuda(), pt.cuda(), sl.cuda(),
                                       scale=scale, num_splits=splits)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    o_ref, l_ref = oracle.attn_decode_paged_f64(q, kc, vc, pt.numpy(), sl.numpy(), scale)
    return assert_bf16_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, l_ref, label)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("nq", [1, 3, 8])
@pytest.mark.parametrize("ps", [16, 64])
def test_small_against_oracle(fa, d, nq, ps):
    lens = [max(nq, n) for n in (1, 17, 64, 65, 300, 1000)]
    for splits in (0, 1, 3):
        _check(fa, lens, 2, nq, d, ps, splits, seed=80 + nq, label=f"d={d} nq={nq} ps={ps} s={splits}")


def test_full_size_step(fa):
    """B=16, H=16, every sequence 8192 tokens in 64-token pages, d=128, one new token."""
    _check(fa, [8192] * 16, 16, 1, 128, 64, 0, seed=0, label="B16 H16 L8192")


@pytest.mark.parametrize("nq", [2, 4, 8])
def test_full_size_multi_query_step(fa, nq):
    """B=16, H=16, 8192 cached tokens each in 64-token pages, d=128, nq new tokens (the
    tensor-core kernel): every output against the oracle."""
    _check(fa, [8192] * 16, 16, nq, 128, 64, 0, seed=nq, label=f"B16 H16 L8192 nq{nq}")


@pytest.mark.parametrize("ps", [8, 128, 256])
def test_multi_query_page_sizes(fa, ps):
    """Pages smaller than, equal to and larger than a 128-key tile, lengths that end inside
    a tile and inside a page, d = 64 and 128, automatic and forced splits."""
    lens = [1, 7, 127, 128, 129, 300, 1000, 2049]
    for d in (64, 128):
        for splits in (0, 1, 3):
            _check(fa, [max(4, n) for n in lens], 2, 4, d, ps, splits, seed=ps + d,
                   label=f"nq4 d={d} ps={ps} s={splits}")


def test_mixed_lengths_many_splits(fa):
    lens = [2, 5000, 129, 8192, 7, 2048]
    _check(fa, lens, 4, 2, 128, 32, 0, seed=81, label="mixed auto")
    _check(fa, lens, 4, 2, 128, 32, 64, seed=81, label="mixed 64 splits")


def test_workspace_rules(fa):
    lens = [4096, 4096]
    q, kc, vc, pt, sl = make_paged_cache(lens, 2, 1, 128, 64, seed=82)
    args = [t.cuda() for t in (q, kc, vc, pt, sl)]
    need = fa.attn_decode_workspace_bytes(2, 2, 1, 128, 64, pt.shape[1], 8)
    assert need == 2 * 2 * 8 * 1 * 129 * 4
    small = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(fa.AttnError):          # forced splits that do not fit
        fa.attn_decode_bf16_paged(*args, num_splits=8, workspace=small)
    # automatic plan with too small a workspace falls back to fewer splits, same result
    o1, l1 = fa.attn_decode_bf16_paged(*args, num_splits=0, workspace=small)
    o2, l2 = fa.attn_decode_bf16_paged(*args, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_sequence_shorter_than_queries(fa):
    """L = 2 with nq = 4: queries 0, 1 see no key (O = 0, LSE = -inf); 2, 3 see 1 and 2 keys."""
    q, kc, vc, pt, sl = make_paged_cache([2], 1, 4, 64, 16, seed=83)
    o, lse = fa.attn_decode_bf16_paged(q.cuda(), kc.cuda(), vc.cuda(), pt.cuda(), sl.cuda(), scale=0.2)
    o, lse = o.cpu(), lse.cpu()
    assert torch.all(o[0, 0, :2] == 0) and torch.all(torch.isinf(lse[0, 0, :2]))
    page = int(pt[0, 0])
    k0, v0 = kc[page, 0, 0].double(), vc[page, 0, 0].double()
    assert (o[0, 0, 2].double() - v0).abs().max() <= 1e-2      # one key: its value
    assert abs(float(lse[0, 0, 2]) - 0.2 * float((q[0, 0, 2].double() * k0).sum())) <= 1e-3
