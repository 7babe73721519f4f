"""attn_decode_bf16_paged_noalloc: the decoding step that allocates nothing.

Some callers cannot allocate device memory at the moment they decode: an engine that
planned every byte of the GPU when it started and hands a kernel only the tensors it
computes on, or a latency-bound loop where cudaMalloc would synchronise the device
and stall the other streams.  For them the split partials live in a fixed 16 MiB
array that the library keeps on each device.  These tests call that entry point
directly through the C ABI (ctypes, raw device pointers, outputs allocated by the
test beforehand) and compare it bit for bit with attn_decode_bf16_paged given a
workspace and the same split plan.

The file is named so that pytest collects it last: a run that stops at the first
failure has run every other test before it.  It passes on its own in a fresh
process as well as after the rest of the suite.
"""
import math

import pytest
import torch

from exact_attention_55_gb300.inputs import make_paged_cache
from tests.conftest import require_gpu

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20   # the library's per-device scratch for this entry point


@pytest.fixture(scope="module")
def fa():
    require_gpu()
    import exact_attention_55_gb300 as fa
    fa.load_library()
    return fa


def _noalloc(fa, q, kc, vc, pt, sl, o, lse, splits, stream=None):
    """One call of the C entry point; returns its status code."""
    B, H, nq, d = q.shape
    num_pages, _, page_size, _ = kc.shape
    s = torch.cuda.current_stream() if stream is None else stream
    return fa.load_library().attn_decode_bf16_paged_noalloc(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), pt.data_ptr(), sl.data_ptr(), o.data_ptr(),
        lse.data_ptr(), B, H, nq, d, page_size, num_pages, pt.shape[1], 1.0 / math.sqrt(d),
        splits, s.cuda_stream)


def _outputs(q):
    B, H, nq, _ = q.shape
    return torch.empty_like(q), torch.empty((B, H, nq), dtype=torch.float32, device=q.device)


def _reference(fa, q, kc, vc, pt, sl, splits):
    """The workspace entry point (caller-owned workspace) with the same plan."""
    return fa.attn_decode_bf16_paged(q, kc, vc, pt, sl, scale=1.0 / math.sqrt(q.shape[-1]),
                                     num_splits=splits)


def _device_case(lens, H, nq, d, ps, seed):
    return tuple(t.cuda() for t in make_paged_cache(lens, H, nq, d, ps, seed=seed))


CASES = [
    # lens, H, nq, d, page size, splits (0: automatic plan)
    ([8192] * 16, 16, 1, 128, 64, 0),          # the decode workload, many splits
    ([2, 5000, 129, 3000], 4, 3, 64, 32, 5),   # ragged lengths, forced splits
    ([700, 33, 4096], 2, 8, 256, 16, 0),       # largest head dim and query count
]


def test_two_calls_in_a_row_match_the_workspace_entry(fa):
    """Two consecutive calls, each with a different shape, so the second one runs on
    whatever the first left in the shared scratch; both equal the workspace entry."""
    assert fa.attn_get_device_status() == fa.ATTN_OK
    for seed, (lens, H, nq, d, ps, splits) in enumerate(CASES[:2]):
        args = _device_case(lens, H, nq, d, ps, seed=90 + seed)
        o_ref, l_ref = _reference(fa, *args, splits)
        o, lse = _outputs(args[0])
        assert _noalloc(fa, *args, o, lse, splits) == fa.ATTN_OK
        torch.cuda.synchronize()
        assert fa.attn_get_device_status() == fa.ATTN_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), (lens, H, nq, d, ps, splits)


def test_ordered_calls_on_one_stream_reuse_the_scratch(fa):
    """Several calls of different shapes queued back to back on one stream, without a
    host synchronisation between them: each call's partials are merged before the
    next call overwrites them, so every output equals the workspace entry's."""
    cases = [_device_case(lens, H, nq, d, ps, seed=100 + i)
             for i, (lens, H, nq, d, ps, _) in enumerate(CASES)]
    refs = [_reference(fa, *args, c[-1]) for args, c in zip(cases, CASES)]
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    outs = [_outputs(args[0]) for args in cases]
    torch.cuda.synchronize()
    for _ in range(2):
        for args, (o, lse), c in zip(cases, outs, CASES):
            assert _noalloc(fa, *args, o, lse, c[-1], stream=stream) == fa.ATTN_OK
    stream.synchronize()
    assert fa.attn_get_device_status() == fa.ATTN_OK
    for (o, lse), (o_ref, l_ref) in zip(outs, refs):
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_automatic_plan_shrinks_to_the_scratch(fa):
    """B=32, H=16, nq=8, d=256, 4096 cached tokens: the automatic plan wants about
    eight splits (4.2 MB of partials each), more than the 16 MiB scratch holds, so the
    entry point falls back to the 3 splits that fit and gives the workspace entry's
    3-split result bit for bit."""
    B, H, nq, d, ps, L = 32, 16, 8, 256, 64, 4096
    per_split = B * H * nq * (d + 1) * 4
    assert SCRATCH_BYTES // per_split == 3
    assert fa.attn_decode_workspace_bytes(B, H, nq, d, ps, L // ps, 0) > SCRATCH_BYTES
    g = torch.Generator(device="cuda")
    g.manual_seed(95)
    pages = B * (L // ps)
    q = torch.randn((B, H, nq, d), generator=g, device="cuda").to(torch.bfloat16)
    kc = torch.randn((pages, H, ps, d), generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn((pages, H, ps, d), generator=g, device="cuda").to(torch.bfloat16)
    pt = torch.randperm(pages, generator=g, device="cuda").to(torch.int32).reshape(B, L // ps)
    sl = torch.full((B,), L, dtype=torch.int32, device="cuda")
    sl[::3] = L - 77                            # some sequences end inside a page
    o_ref, l_ref = _reference(fa, q, kc, vc, pt, sl, 3)
    o, lse = _outputs(q)
    for _ in range(2):
        assert _noalloc(fa, q, kc, vc, pt, sl, o, lse, 0) == fa.ATTN_OK
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert fa.attn_get_device_status() == fa.ATTN_OK


def test_a_forced_plan_larger_than_the_scratch_is_refused(fa):
    """num_splits = 8 at B=64, H=32, nq=8, d=256 needs 134 MB of partials: refused
    with ATTN_ERR_INVALID_ARG before anything is launched."""
    B, H, nq, d = 64, 32, 8, 256
    q = torch.zeros((B, H, nq, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((8, H, 16, d), dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros((B, 8), dtype=torch.int32, device="cuda")
    sl = torch.full((B,), 100, dtype=torch.int32, device="cuda")
    o, lse = _outputs(q)
    assert _noalloc(fa, q, kc, kc, pt, sl, o, lse, 8) == fa.ATTN_ERR_INVALID_ARG
    assert fa.attn_get_device_status() == fa.ATTN_OK
