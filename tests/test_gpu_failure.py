"""Failure detection on the GPU without a fault: a bounded wait that runs out
records ATTN_ERR_TIMEOUT, the host reads it, and the context keeps working."""
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
