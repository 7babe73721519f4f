"""The C-ABI calls can be captured in a CUDA graph: a replay gives the eager
result bit for bit and follows new contents of the captured input buffers."""
import pytest
import torch

from exact_attention_55_gb300.inputs import make_qkv
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def test_bf16_forward_in_a_graph(fa):
    q, k, v = make_qkv(2, 4, 1024, 128, seed=70)
    q2, _, _ = make_qkv(2, 4, 1024, 128, seed=71)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((2, 4, 1024), dtype=torch.float32, device="cuda")
    fa.attn_fwd_bf16(qd, kd, vd, causal=True, o=o, lse=lse)   # eager first (device set-up)
    torch.cuda.synchronize()
    ref_o, ref_l = o.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.attn_fwd_bf16(qd, kd, vd, causal=True, o=o, lse=lse)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
    qd.copy_(q2.cuda())
    g.replay()
    o2, l2 = fa.attn_fwd_bf16(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert fa.attn_get_device_status() == fa.ATTN_OK
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_fp8_chain_in_a_graph(fa):
    """Three quantisations (Q, K rotated) and the FP8 forward as one graph."""
    q, k, v = make_qkv(1, 4, 1024, 128, seed=72, outliers=True)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()

    def chain():
        q8, sq = fa.attn_quantize_fp8_hadamard(qd, x8=bufs[0][0], scales=bufs[0][1])
        k8, sk = fa.attn_quantize_fp8_hadamard(kd, x8=bufs[1][0], scales=bufs[1][1])
        v8, sv = fa.attn_quantize_fp8_blockwise(vd, x8=bufs[2][0], scales=bufs[2][1])
        fa.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o=o, lse=lse)

    bufs = [(torch.empty(qd.shape, dtype=torch.uint8, device="cuda"),
             torch.empty((1, 4, 8), dtype=torch.float32, device="cuda")) for _ in range(3)]
    o = torch.empty_like(qd)
    lse = torch.empty((1, 4, 1024), dtype=torch.float32, device="cuda")
    chain()
    torch.cuda.synchronize()
    ref_o, ref_l = o.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fa.attn_get_device_status() == fa.ATTN_OK
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
