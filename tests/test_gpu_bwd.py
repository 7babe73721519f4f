"""GPU parity of attn_bwd_bf16 against the float64 oracle's gradients.

Tolerance: the kernel rounds dS and P to bf16 for the tensor-core products
(relative 2^-9 per element), reads the bf16 forward output O for D = dO . O, and
rounds dQ, dK, dV to bf16; each of these is a relative error of a few 1e-3 RMS,
so the bar is RMSE / RMS <= 1e-2 per gradient (and max |d| <= 5 % of max |ref|)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_55_gb300.inputs import make_qkv
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

MASKS = [(False, 0), (True, 0), (False, 100), (True, 100)]


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _case(fa, B, H, N, d, causal, window, seed, heads=None):
    q, k, v = make_qkv(B, H, N, d, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    do = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attn_fwd_bf16(qd, kd, vd, scale=scale, causal=causal, window=window)
    dq, dk, dv = fa.attn_bwd_bf16(qd, kd, vd, o, dod, lse, scale=scale, causal=causal, window=window)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    out = {}
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        out[name] = got.cpu()
    errs = {}
    for (b, h) in heads:
        ref = oracle.attn_bwd_f64(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal=causal, window=window)
        for name, r in zip(("dq", "dk", "dv"), ref):
            gv = out[name][b, h].double().numpy()
            assert np.isfinite(gv).all()
            if np.abs(r).max() < 1e-9:
                # an identically zero gradient (e.g. dQ with a single key: dS = dP - D = 0)
                assert np.abs(gv).max() <= 1e-3, f"{name} head {(b, h)}: {np.abs(gv).max()}"
                continue
            rel = float(np.sqrt(np.mean((gv - r) ** 2)) / np.sqrt(np.mean(r ** 2)))
            mx = float(np.abs(gv - r).max() / np.abs(r).max())
            errs[name] = max(errs.get(name, 0.0), rel)
            assert rel <= 1e-2 and mx <= 5e-2, f"{name} head {(b, h)} rel {rel} max {mx}"
    return errs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", MASKS)
def test_ragged(fa, d, causal, window):
    _case(fa, 1, 2, 300, d, causal, window, seed=100)


@pytest.mark.parametrize("N", [1, 128, 129, 1000])
def test_lengths(fa, N):
    for causal in (False, True):
        _case(fa, 2, 2, N, 128, causal, 0, seed=101 + N)


@pytest.mark.parametrize("causal", [False, True])
def test_n2048_sampled_heads(fa, causal):
    e = _case(fa, 2, 8, 2048, 128, causal, 0, seed=102, heads=[(0, 0), (1, 7), (0, 5)])
    print("bwd N2048", causal, e)
