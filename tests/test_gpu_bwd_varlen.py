"""GPU parity of attn_bwd_bf16_varlen (backward over packed variable-length sequences)
against the oracle's per-sequence float64 gradients, and bit-identity with the batched
backward when every sequence has the same length."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_packed_qkv, make_qkv
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

LENGTHS = [300, 1, 0, 129, 1000, 128, 127, 255, 2]
MASKS = [(False, 0), (True, 0), (False, 100), (True, 100)]


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _run(fa, lengths, H, d, causal, window, seed):
    q, k, v, cu = make_packed_qkv(lengths, H, d, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod, cud = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu.cuda()
    o, lse = fa.attn_fwd_bf16_varlen(qd, kd, vd, cud, max(lengths), scale=scale, causal=causal,
                                     window=window)
    dq, dk, dv = fa.attn_bwd_bf16_varlen(qd, kd, vd, o, dod, lse, cud, max(lengths), scale=scale,
                                         causal=causal, window=window)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    return (q, k, v, do, cu, scale), (dq.cpu(), dk.cpu(), dv.cpu())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", MASKS)
def test_ragged_packs_against_the_oracle(fa, d, causal, window):
    (q, k, v, do, cu, scale), got = _run(fa, LENGTHS, 2, d, causal, window, seed=71)
    ref = oracle.attn_varlen_bwd_f64(q, k, v, do, cu.numpy(), scale, causal=causal, window=window)
    for name, gv, r in zip(("dq", "dk", "dv"), got, ref):
        gv = gv.double().numpy()
        assert np.isfinite(gv).all()
        rel = float(np.sqrt(np.mean((gv - r) ** 2)) / np.sqrt(np.mean(r ** 2)))
        mx = float(np.abs(gv - r).max() / np.abs(r).max())
        print(name, d, causal, window, rel, mx)
        assert rel <= 1e-2 and mx <= 5e-2, (name, rel, mx)
    # single-token sequences: one key, so dQ = dK = 0 and dV = dO
    a = int(cu[1])
    np.testing.assert_allclose(got[0][a].double().numpy(), 0.0, atol=1e-3)
    np.testing.assert_allclose(got[2][a].double().numpy(), do[a].double().numpy(), atol=2e-2)


def test_equal_lengths_match_the_batched_backward(fa):
    B, H, N, d = 3, 2, 256, 128
    q, k, v = make_qkv(B, H, N, d, seed=72)
    g = torch.Generator().manual_seed(73)
    do = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)
    pack = lambda x: x.transpose(1, 2).reshape(B * N, H, d).contiguous()
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    for causal in (False, True):
        o, lse = fa.attn_fwd_bf16(qd, kd, vd, causal=causal)
        ref = fa.attn_bwd_bf16(qd, kd, vd, o, dod, lse, causal=causal)
        cu = (torch.arange(B + 1, dtype=torch.int32) * N).cuda()
        lse_p = lse.permute(1, 0, 2).reshape(H, B * N).contiguous()   # [H, T]
        got = fa.attn_bwd_bf16_varlen(pack(qd), pack(kd), pack(vd), pack(o), pack(dod), lse_p, cu, N,
                                      causal=causal)
        assert fa.attn_get_device_status() == fa.ATTN_OK
        for gp, r in zip(got, ref):
            assert torch.equal(gp, pack(r)), causal


def test_zero_tokens_and_argument_errors(fa):
    H, d = 2, 64
    e = torch.empty((0, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((H, 0), dtype=torch.float32, device="cuda")
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    fa.attn_bwd_bf16_varlen(e, e, e, e, e, lse, cu, 0)   # nothing to do, no error
    q, k, v, cu = make_packed_qkv([10, 20], H, 256, seed=74)
    qd = q.cuda()
    lse2 = torch.empty((H, 30), dtype=torch.float32, device="cuda")
    with pytest.raises(fa.AttnError):                     # d = 256 is not supported
        fa.attn_bwd_bf16_varlen(qd, qd, qd, qd, qd, lse2, cu.cuda(), 20)
