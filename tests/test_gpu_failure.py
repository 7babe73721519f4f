"""Failure detection on the GPU without a fault: a bounded wait that runs out
records ATTN_ERR_TIMEOUT, the host reads it, and the context keeps working -- first
in a standalone waiting kernel, then in the forward, quantiser and backward kernels
themselves with one of their loads withheld."""
import numpy as np
import pytest

import oracle
from exact_attention_55_gb300.inputs import make_qkv
from tests.attn_check import assert_bf16_close
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def test_wait_that_runs_out_reports_timeout_and_context_survives(fa):
    assert fa.attn_get_device_status() == fa.ATTN_OK          # clears any earlier state
    fa.attn_selftest_wait_timeout(50_000_000)                 # 50 ms, nobody arrives
    assert fa.attn_get_device_status() == fa.ATTN_ERR_TIMEOUT
    assert fa.attn_get_device_status() == fa.ATTN_OK          # reading cleared it
    q, k, v = make_qkv(1, 2, 256, 64, seed=40)
    o, lse = fa.attn_fwd_bf16(q.cuda(), k.cuda(), v.cuda(), scale=0.125, causal=True)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    o_ref, lse_ref = oracle.attn_f64(q, k, v, 0.125, causal=True)
    assert_bf16_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref)


def test_selftest_rejects_bad_limits(fa):
    with pytest.raises(fa.AttnError):
        fa.attn_selftest_wait_timeout(0)
    with pytest.raises(fa.AttnError):
        fa.attn_selftest_wait_timeout(10 ** 10)


# The production kernels' own abort path: one load is never issued, so the bounded
# waits on it run out (20 ms here), the CTA raises its abort flag, waits for the copies
# and MMAs it already issued, frees its tensor memory and exits.  The status word then
# reads ATTN_ERR_TIMEOUT, and a normal call afterwards reproduces, bit for bit, the
# result of the same call made before the aborted one.

def test_forward_kernel_aborts_on_a_withheld_load(fa):
    import math
    import torch
    q, k, v = make_qkv(1, 2, 1024, 128, seed=41)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1.0 / math.sqrt(128)
    o1, l1 = fa.attn_fwd_bf16(qd, kd, vd, scale=scale)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    o_bad, l_bad = torch.empty_like(qd), torch.empty_like(l1)
    # load 2 of each CTA is the K tile of the second key step; the ring has room for
    # three more loads behind it, which are in flight or landed when the CTA aborts
    fa.attn_selftest_fwd_withheld_load(qd, kd, vd, o_bad, l_bad, withheld=2, timeout_ns=20_000_000)
    assert fa.attn_get_device_status() == fa.ATTN_ERR_TIMEOUT
    o2, l2 = fa.attn_fwd_bf16(qd, kd, vd, scale=scale)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, lse_ref = oracle.attn_f64(q, k, v, scale)
    assert_bf16_close(o2.cpu().double().numpy(), l2.cpu().double().numpy(), o_ref, lse_ref)


def test_forward_kernel_aborts_on_a_withheld_load_causal_d64(fa):
    import torch
    q, k, v = make_qkv(2, 2, 2048, 64, seed=42)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fa.attn_fwd_bf16(qd, kd, vd, scale=0.125, causal=True)
    o_bad, l_bad = torch.empty_like(qd), torch.empty_like(l1)
    fa.attn_selftest_fwd_withheld_load(qd, kd, vd, o_bad, l_bad, causal=True, withheld=5,
                                       timeout_ns=20_000_000)
    assert fa.attn_get_device_status() == fa.ATTN_ERR_TIMEOUT
    o2, l2 = fa.attn_fwd_bf16(qd, kd, vd, scale=0.125, causal=True)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_quantizer_aborts_on_a_withheld_load(fa):
    import torch
    # 1024 blocks over at most 2 CTAs per SM: several blocks per CTA, so the loads of
    # the following iterations are in flight when the second one never arrives
    x = make_qkv(1, 16, 8192, 128, seed=43, outliers=True)[0].cuda()
    x8a, sa = fa.attn_quantize_fp8_blockwise(x)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    x8b, sb = torch.empty_like(x8a), torch.empty_like(sa)
    fa.attn_selftest_quant_withheld_load(x, x8b, sb, withheld=1, timeout_ns=20_000_000)
    assert fa.attn_get_device_status() == fa.ATTN_ERR_TIMEOUT
    x8c, sc = fa.attn_quantize_fp8_blockwise(x)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    assert torch.equal(x8a, x8c) and torch.equal(sa, sc)
    r8, rsc = oracle.quantize_fp8_blockwise(x.cpu(), 128)
    np.testing.assert_array_equal(x8c.cpu().numpy(), r8)
    np.testing.assert_array_equal(sc.cpu().numpy(), rsc)


def test_backward_kernels_abort_on_a_withheld_load(fa):
    import torch
    q, k, v = make_qkv(1, 2, 512, 128, seed=44)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.attn_fwd_bf16(qd, kd, vd, scale=1.0 / 128 ** 0.5)
    g = torch.Generator(device="cuda")
    g.manual_seed(45)
    dout = torch.randn(qd.shape, generator=g, device="cuda").to(torch.bfloat16)
    ref = fa.attn_bwd_bf16(qd, kd, vd, o, dout, lse, scale=1.0 / 128 ** 0.5)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    bad = [torch.empty_like(qd) for _ in range(3)]
    ws = torch.empty((1, 2, 512), dtype=torch.float32, device="cuda")
    fa.attn_selftest_bwd_withheld_load(qd, kd, vd, o, dout, lse, *bad, ws, withheld=2,
                                       timeout_ns=20_000_000)
    assert fa.attn_get_device_status() == fa.ATTN_ERR_TIMEOUT
    again = fa.attn_bwd_bf16(qd, kd, vd, o, dout, lse, scale=1.0 / 128 ** 0.5)
    assert fa.attn_get_device_status() == fa.ATTN_OK
    for a, b in zip(ref, again):
        assert torch.equal(a, b)
