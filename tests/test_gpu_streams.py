"""Independent calls on concurrent streams give their sequential results bit for
bit: the entry points share no state besides the status word (and the no-alloc
decode scratch, which is documented as ordered-only and not used here)."""
import pytest
import torch

from exact_attention_55_gb300.inputs import make_packed_qkv, make_paged_cache, make_qkv
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu


def test_concurrent_streams_match_sequential():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    q, k, v = (t.cuda() for t in make_qkv(2, 4, 2048, 128, seed=90))
    q8i = [t.cuda() for t in make_qkv(1, 4, 1024, 128, seed=91, outliers=True)]
    qp, kp, vp, cu = (t.cuda() for t in make_packed_qkv([700, 1, 1300], 4, 64, seed=92))
    dq, dkc, dvc, dpt, dsl = (t.cuda() for t in make_paged_cache([3000, 17, 9000], 4, 2, 128, 32, seed=93))

    def run_all():
        o1, l1 = fa.attn_fwd_bf16(q, k, v, causal=True)
        qs = [fa.attn_quantize_fp8_hadamard(q8i[0]), fa.attn_quantize_fp8_hadamard(q8i[1]),
              fa.attn_quantize_fp8_blockwise(q8i[2])]
        o2, l2 = fa.attn_fwd_fp8(qs[0][0], qs[1][0], qs[2][0], qs[0][1], qs[1][1], qs[2][1])
        o3, l3 = fa.attn_fwd_bf16_varlen(qp, kp, vp, cu, 1300, window=100)
        o4, l4 = fa.attn_decode_bf16_paged(dq, dkc, dvc, dpt, dsl)
        return [o1, l1, o2, l2, o3, l3, o4, l4]

    ref = run_all()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(4)]
    outs = [None] * 4
    torch.cuda.synchronize()
    for rep in range(3):
        for n, s in enumerate(streams):
            with torch.cuda.stream(s):
                if n == 0:
                    outs[0] = fa.attn_fwd_bf16(q, k, v, causal=True)
                elif n == 1:
                    qs = [fa.attn_quantize_fp8_hadamard(q8i[0]), fa.attn_quantize_fp8_hadamard(q8i[1]),
                          fa.attn_quantize_fp8_blockwise(q8i[2])]
                    outs[1] = fa.attn_fwd_fp8(qs[0][0], qs[1][0], qs[2][0], qs[0][1], qs[1][1], qs[2][1])
                elif n == 2:
                    outs[2] = fa.attn_fwd_bf16_varlen(qp, kp, vp, cu, 1300, window=100)
                else:
                    outs[3] = fa.attn_decode_bf16_paged(dq, dkc, dvc, dpt, dsl)
        torch.cuda.synchronize()
        assert fa.attn_get_device_status() == fa.ATTN_OK
        got = [t for pair in outs for t in pair]
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
