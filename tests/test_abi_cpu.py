"""CPU checks of the C ABI: the library loads, exports every function include/attn.h
declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "attn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_55_gb300 import build
    path = build.build()
    import exact_attention_55_gb300 as fa
    return fa.load_library(path)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("attn_fwd_bf16", "attn_fwd_bf16_varlen", "attn_decode_bf16_paged",
              "attn_decode_workspace_bytes", "attn_quantize_fp8_blockwise",
              "attn_quantize_fp8_hadamard", "attn_fwd_fp8", "attn_status_string",
              "attn_get_device_status", "attn_selftest_wait_timeout"):
        assert n in names


def test_header_is_plain_c():
    """The boundary header compiles on its own as C (no C++ or CUDA types leak in)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} is declared in attn.h but not exported"


def test_binding_names_match_header():
    import exact_attention_55_gb300 as fa
    for name in _declared_functions():
        assert callable(getattr(fa, name)), name


def test_status_strings(lib):
    for code in range(6):
        assert lib.attn_status_string(code)
    assert lib.attn_status_string(99) == b"unknown status"


P = 0x10000  # a 16-byte aligned fake device address; no call below reaches the GPU


@pytest.mark.parametrize("args,expected", [
    ((0, P, P, P, P, 1, 1, 128, 128, 0.1, 0, 0), 1),          # null q
    ((P, P, P, P, 0, 1, 1, 128, 128, 0.1, 0, 0), 1),          # null lse
    ((P, P, P, P, P, 0, 1, 128, 128, 0.1, 0, 0), 1),          # B = 0
    ((P, P, P, P, P, 1, 1, 0, 128, 0.1, 0, 0), 1),            # N = 0
    ((P, P, P, P, P, 1, 1, 128, 128, 0.0, 0, 0), 1),          # scale = 0
    ((P, P, P, P, P, 1, 1, 128, 128, float("nan"), 0, 0), 1),  # scale = nan
    ((P, P, P, P, P, 1, 1, 128, 128, float("inf"), 0, 0), 1),  # scale = inf
    ((P, P, P, P, P, 1, 1, 128, 96, 0.1, 0, 0), 2),           # d = 96
    ((P, P, P, P, P, 1, 1, 128, 32, 0.1, 0, 0), 2),           # d = 32
    ((P + 8, P, P, P, P, 1, 1, 128, 128, 0.1, 0, 0), 3),      # q misaligned
    ((P, P, P, P + 2, P, 1, 1, 128, 128, 0.1, 0, 0), 3),      # o misaligned
    ((P, P, P, P, P + 2, 1, 1, 128, 128, 0.1, 0, 0), 3),      # lse misaligned
])
def test_bf16_argument_errors(lib, args, expected):
    assert lib.attn_fwd_bf16(*args, None) == expected


@pytest.mark.parametrize("args,expected", [
    ((0, P, P, 1, 1, 128, 128, 128), 1),
    ((P, P, P, 1, 1, 128, 128, 32), 2),      # block not 64 or 128
    ((P, P, P, 1, 1, 128, 128, 256), 2),
    ((P, P, P, 1, 1, 128, 120, 128), 2),     # d % 16 != 0
    ((P, P, P, 1, 1, 128, 512, 128), 2),     # d > 256
    ((P + 4, P, P, 1, 1, 128, 128, 128), 3),
    ((P, P, P + 2, 1, 1, 128, 128, 128), 3),
])
def test_quantizer_argument_errors(lib, args, expected):
    assert lib.attn_quantize_fp8_blockwise(*args, None) == expected


@pytest.mark.parametrize("args,expected", [
    ((P, P, P, 0, P, P, P, P, 1, 1, 256, 128, 0.1, 0, 0), 1),   # null descale
    ((P, P, P, P, P, P, P, P, 1, 1, 200, 128, 0.1, 0, 0), 2),   # N % 128
    ((P, P, P, P, P, P, P, P, 1, 1, 256, 32, 0.1, 0, 0), 2),    # d = 32
    ((P, P, P + 1, P, P, P, P, P, 1, 1, 256, 128, 0.1, 0, 0), 3),
])
def test_fp8_argument_errors(lib, args, expected):
    assert lib.attn_fwd_fp8(*args, None) == expected


def test_selftest_rejects_bad_limits_before_any_launch(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == 1
    assert lib.attn_selftest_wait_timeout(3_000_000_000, None) == 1
    fwd = (P, P, P, P, P, 1, 1, 256, 128, 0)
    assert lib.attn_selftest_fwd_withheld_load(*fwd, -1, 1_000_000, None) == 1
    assert lib.attn_selftest_fwd_withheld_load(*fwd, 2, 0, None) == 1
    assert lib.attn_selftest_fwd_withheld_load(*fwd, 2, 3_000_000_000, None) == 1
    assert lib.attn_selftest_quant_withheld_load(P, P, P, 1, 1, 256, 128, -1, 1_000_000, None) == 1
    assert lib.attn_selftest_quant_withheld_load(P, P, P, 1, 1, 256, 128, 0, 0, None) == 1
    bwd = (P, P, P, P, P, P, P, P, P, P, 4096, 1, 1, 256, 128, 0)
    assert lib.attn_selftest_bwd_withheld_load(*bwd, -1, 1_000_000, None) == 1
    assert lib.attn_selftest_bwd_withheld_load(*bwd, 1, 0, None) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    import exact_attention_55_gb300 as fa
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fa.attn_fwd_bf16(q, q, q)


def test_missing_library_fails_loudly(tmp_path):
    import exact_attention_55_gb300 as fa
    saved = fa._lib
    fa._lib = None
    try:
        with pytest.raises(RuntimeError):
            fa.load_library(str(tmp_path / "nope.so"))
    finally:
        fa._lib = saved


@pytest.mark.parametrize("args,expected", [
    ((P, P, P, 1, 1, 128, 128, 128, 3), 1),       # unknown format
    ((P, P, P, 1, 1, 128, 128, 128, -1), 1),
    ((P, P, P, 1, 1, 128, 128, 96, 1), 2),        # E5M2, block not 64 or 128
    ((P + 4, P, P, 1, 1, 128, 128, 128, 2), 3),   # power-of-two scales, x misaligned
])
def test_quantizer_fmt_argument_errors(lib, args, expected):
    assert lib.attn_quantize_fp8_blockwise_fmt(*args, None) == expected


@pytest.mark.parametrize("fmts,shape,expected", [
    ((3, 0), (256, 128), 1),      # unknown Q/K format
    ((0, 1), (256, 128), 1),      # V in E5M2 is not a V format
    ((1, 3), (256, 128), 1),
    ((1, 0), (200, 128), 2),      # E5M2 Q/K, N % 128
    ((0, 2), (256, 96), 2),       # power-of-two V, d = 96
])
def test_fp8_fmt_argument_errors(lib, fmts, shape, expected):
    N, d = shape
    args = (P, P, P, P, P, P, P, P, 1, 1, N, d, 0.1, 0, 0)
    assert lib.attn_fwd_fp8_fmt(*args, *fmts, None) == expected


@pytest.mark.parametrize("qk_block,shape,expected", [
    (32, (256, 64), 2),           # block height not 64 or 128
    (256, (256, 128), 2),
    (64, (200, 64), 2),           # N % 128
    (64, (256, 48), 2),           # head dim
])
def test_fp8_blocks_argument_errors(lib, qk_block, shape, expected):
    N, d = shape
    args = (P, P, P, P, P, P, P, P, 1, 1, N, d, 0.1, 0, 0, 0, 0, qk_block)
    assert lib.attn_fwd_fp8_blocks(*args, None) == expected


def test_head_dim_aware_block_rows(lib):
    assert [lib.attn_fp8_qk_block_rows(d) for d in (64, 128, 256, 0)] == [64, 128, 128, 0]


def test_bwd_workspace_size(lib):
    assert lib.attn_bwd_workspace_bytes(2, 3, 100) == 2 * 3 * 100 * 4


@pytest.mark.parametrize("change,expected", [
    ({0: 0}, 1),                  # null q
    ({9: 0}, 1),                  # null workspace
    ({10: 4}, 1),                 # workspace too small
    ({14: 256}, 2),               # d = 256
    ({14: 96}, 2),
    ({11: 0}, 1),                 # B = 0
    ({15: 0.0}, 1),               # scale = 0
    ({3: P + 2}, 3),              # o misaligned
    ({5: P + 2}, 3),              # lse misaligned
])
def test_bwd_argument_errors(lib, change, expected):
    # q, k, v, o, dout, lse, dq, dk, dv, workspace, ws_bytes, B, H, N, d, scale, causal, window
    args = [P, P, P, P, P, P, P, P, P, P, 1 * 1 * 256 * 4, 1, 1, 256, 128, 0.1, 0, 0]
    for i, v in change.items():
        args[i] = v
    assert lib.attn_bwd_bf16(*args, None) == expected


@pytest.mark.parametrize("change,expected", [
    ({14: 0, 13: 0}, 0),          # zero tokens: nothing to do
    ({12: 0}, 1),                 # num_seqs = 0
    ({0: 0}, 1),                  # null q
    ({11: 0}, 1),                 # null cu_seqlens
    ({10: 4}, 1),                 # workspace too small
    ({16: 256}, 2),               # d = 256
    ({13: 300}, 1),               # max_seqlen > T
    ({11: P + 2}, 3),             # cu_seqlens misaligned
])
def test_bwd_varlen_argument_errors(lib, change, expected):
    # q, k, v, o, dout, lse, dq, dk, dv, ws, ws_bytes, cu, S, max_seqlen, T, H, d, scale, causal, window
    args = [P, P, P, P, P, P, P, P, P, P, 2 * 256 * 4, P, 2, 128, 256, 2, 128, 0.1, 0, 0]
    for i, v in change.items():
        args[i] = v
    assert lib.attn_bwd_bf16_varlen(*args, None) == expected
