"""GB300 (sm_103a) fused exact-attention forward: thin Python binding of the C ABI.

The functions below carry the C entry points' names (``include/attn.h``) and do
argument marshalling only: every arithmetic step runs in the CUDA library
``_build/libgb300attn.so``.  PyTorch supplies device memory and the stream.
There is no fallback: if the library is missing or fails to load, every call
raises.

    import exact_attention_55_gb300 as fa
    o, lse = fa.attn_fwd_bf16(q, k, v, causal=True)          # q, k, v: cuda bf16 [B,H,N,d]
    q8, sq = fa.attn_quantize_fp8_blockwise(q)               # E4M3 codes + per-block scales
    o8, lse8 = fa.attn_fwd_fp8(q8, k8, v8, sq, sk, sv)
    q8h, sqh = fa.attn_quantize_fp8_hadamard(q)              # rotate rows, then quantise (Q, K)
    o, lse = fa.attn_fwd_bf16_varlen(qp, kp, vp, cu, max_len) # packed [T, H, d], int32 offsets
    o, lse = fa.attn_decode_bf16_paged(q1, kc, vc, table, lens) # decoding step, paged KV cache
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

__all__ = [
    "AttnError", "ATTN_OK", "ATTN_ERR_TIMEOUT", "load_library", "attn_fwd_bf16",
    "attn_bwd_bf16", "attn_bwd_workspace_bytes", "attn_bwd_bf16_varlen",
    "attn_fwd_bf16_varlen", "attn_decode_bf16_paged", "attn_decode_bf16_paged_noalloc",
    "attn_decode_workspace_bytes",
    "attn_quantize_fp8_blockwise", "attn_quantize_fp8_hadamard", "attn_fwd_fp8",
    "attn_quantize_fp8_blockwise_fmt", "attn_fwd_fp8_fmt", "attn_fwd_fp8_blocks",
    "attn_fp8_qk_block_rows", "attn_fwd_schedule", "ATTN_FP8_E4M3", "ATTN_FP8_E5M2",
    "ATTN_FP8_E4M3_POW2",
    "attn_status_string", "attn_get_device_status", "attn_selftest_wait_timeout",
    "attn_selftest_fwd_withheld_load", "attn_selftest_quant_withheld_load",
    "attn_selftest_bwd_withheld_load", "attn_selftest_fp8_convert", "EXPORTED_SYMBOLS",
]

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5

ATTN_FP8_E4M3 = 0
ATTN_FP8_E5M2 = 1
ATTN_FP8_E4M3_POW2 = 2   # E4M3 codes, power-of-two block scales
_FP8_FORMATS = {"e4m3": ATTN_FP8_E4M3, "e5m2": ATTN_FP8_E5M2, "e4m3_pow2": ATTN_FP8_E4M3_POW2,
                ATTN_FP8_E4M3: ATTN_FP8_E4M3, ATTN_FP8_E5M2: ATTN_FP8_E5M2,
                ATTN_FP8_E4M3_POW2: ATTN_FP8_E4M3_POW2}

EXPORTED_SYMBOLS = (
    "attn_fwd_bf16", "attn_bwd_bf16", "attn_bwd_workspace_bytes", "attn_bwd_bf16_varlen",
    "attn_fwd_bf16_varlen",
    "attn_decode_bf16_paged",
    "attn_decode_bf16_paged_noalloc", "attn_decode_workspace_bytes",
    "attn_quantize_fp8_blockwise", "attn_quantize_fp8_blockwise_fmt",
    "attn_quantize_fp8_hadamard",
    "attn_fwd_fp8", "attn_fwd_fp8_fmt", "attn_fwd_fp8_blocks", "attn_fp8_qk_block_rows",
    "attn_fwd_schedule", "attn_status_string", "attn_get_device_status",
    "attn_selftest_wait_timeout", "attn_selftest_fwd_withheld_load",
    "attn_selftest_quant_withheld_load", "attn_selftest_bwd_withheld_load",
    "attn_selftest_fp8_convert",
)

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of the CUDA library.  Raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library not built: {path} is missing (run exact_attention_55_gb300.build.build())")
        lib = ctypes.CDLL(path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd_bf16.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.attn_fwd_bf16.restype = i
        lib.attn_fwd_bf16_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
        lib.attn_fwd_bf16_varlen.restype = i
        lib.attn_bwd_workspace_bytes.argtypes = [i, i, i]
        lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_bwd_bf16.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i,
                                      i, i, f, i, i, vp]
        lib.attn_bwd_bf16.restype = i
        lib.attn_bwd_bf16_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                             vp, i, i, i, i, i, f, i, i, vp]
        lib.attn_bwd_bf16_varlen.restype = i
        lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_decode_bf16_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f,
                                               i, vp, ctypes.c_size_t, vp]
        lib.attn_decode_bf16_paged.restype = i
        lib.attn_decode_bf16_paged_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                                       i, i, f, i, vp]
        lib.attn_decode_bf16_paged_noalloc.restype = i
        lib.attn_quantize_fp8_blockwise.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
        lib.attn_quantize_fp8_blockwise.restype = i
        lib.attn_quantize_fp8_hadamard.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
        lib.attn_quantize_fp8_hadamard.restype = i
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.attn_fwd_fp8.restype = i
        lib.attn_quantize_fp8_blockwise_fmt.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp]
        lib.attn_quantize_fp8_blockwise_fmt.restype = i
        lib.attn_fwd_fp8_fmt.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, i, vp]
        lib.attn_fwd_fp8_fmt.restype = i
        lib.attn_fwd_fp8_blocks.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i,
                                            i, i, vp]
        lib.attn_fwd_fp8_blocks.restype = i
        lib.attn_fp8_qk_block_rows.argtypes = [i]
        lib.attn_fp8_qk_block_rows.restype = i
        lib.attn_fwd_schedule.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
        lib.attn_fwd_schedule.restype = i
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_get_device_status.argtypes = [vp]
        lib.attn_get_device_status.restype = i
        lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
        lib.attn_selftest_wait_timeout.restype = i
        u64 = ctypes.c_ulonglong
        lib.attn_selftest_fwd_withheld_load.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, u64, vp]
        lib.attn_selftest_fwd_withheld_load.restype = i
        lib.attn_selftest_quant_withheld_load.argtypes = [vp, vp, vp, i, i, i, i, i, u64, vp]
        lib.attn_selftest_quant_withheld_load.restype = i
        lib.attn_selftest_bwd_withheld_load.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                        ctypes.c_size_t, i, i, i, i, i, i, u64, vp]
        lib.attn_selftest_bwd_withheld_load.restype = i
        lib.attn_selftest_fp8_convert.argtypes = [ctypes.c_uint, ctypes.c_size_t, i, vp, vp]
        lib.attn_selftest_fp8_convert.restype = i
        _lib = lib
        return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_bhnd(name, t, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")


def _check_out(t, shape, dtype, device, name):
    if (not isinstance(t, torch.Tensor) or t.dtype != dtype or tuple(t.shape) != tuple(shape)
            or t.device != device or not t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")


def _raise_if(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def attn_fwd_bf16(q, k, v, scale: float | None = None, causal: bool = False, window: int = 0,
                  o=None, lse=None, stream=None):
    """O = softmax(scale * Q K^T + mask) V and the natural-log LSE; bf16 in and out."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_bhnd(n, t, torch.bfloat16)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_bhnd("o", o, torch.bfloat16)
    _check_out(o, q.shape, torch.bfloat16, q.device, "o")
    _check_out(lse, (B, H, N), torch.float32, q.device, "lse")
    st = load_library().attn_fwd_bf16(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, N, d, float(scale), int(bool(causal)),
                                      int(window), _stream_handle(stream))
    _raise_if(st, "attn_fwd_bf16")
    return o, lse


def attn_bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    """Workspace bytes attn_bwd_bf16 needs (the per-row D = dO . O)."""
    return int(load_library().attn_bwd_workspace_bytes(B, H, N))


def attn_bwd_bf16(q, k, v, o, dout, lse, scale: float | None = None, causal: bool = False,
                  window: int = 0, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward pass: returns (dQ, dK, dV) bf16 [B, H, N, d] for the upstream gradient dout,
    given the forward's o and lse (same scale / mask)."""
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_bhnd(n, t, torch.bfloat16)
        if t.shape != q.shape:
            raise ValueError(f"{n} must have q's shape")
    B, H, N, d = q.shape
    _check_out(lse, (B, H, N), torch.float32, q.device, "lse")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_out(t, (B, H, N, d), torch.bfloat16, q.device, n)
    if workspace is None:
        workspace = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    st = load_library().attn_bwd_bf16(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), B, H, N, d, float(scale),
        int(bool(causal)), int(window), _stream_handle(stream))
    _raise_if(st, "attn_bwd_bf16")
    return dq, dk, dv


def attn_bwd_bf16_varlen(q, k, v, o, dout, lse, cu_seqlens, max_seqlen: int,
                         scale: float | None = None, causal: bool = False, window: int = 0,
                         dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward over packed sequences: returns (dQ, dK, dV) bf16 [T, H, d] for the upstream
    gradient dout, given attn_fwd_bf16_varlen's o and lse ([H, T]) with the same offsets."""
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous bf16 CUDA tensor [T, H, d]")
        if t.shape != q.shape:
            raise ValueError(f"{n} must have q's shape")
    T, H, d = q.shape
    _check_out(lse, (H, T), torch.float32, q.device, "lse")
    if (not cu_seqlens.is_cuda or cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1
            or not cu_seqlens.is_contiguous()):
        raise TypeError("cu_seqlens must be a contiguous int32 CUDA tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_out(t, (T, H, d), torch.bfloat16, q.device, n)
    if workspace is None:
        workspace = torch.empty((H, max(T, 1)), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    st = load_library().attn_bwd_bf16_varlen(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), cu_seqlens.data_ptr(),
        cu_seqlens.numel() - 1, int(max_seqlen), T, H, d, float(scale), int(bool(causal)),
        int(window), _stream_handle(stream))
    _raise_if(st, "attn_bwd_bf16_varlen")
    return dq, dk, dv


def attn_fwd_bf16_varlen(q, k, v, cu_seqlens, max_seqlen: int, scale: float | None = None,
                         causal: bool = False, window: int = 0, o=None, lse=None, stream=None):
    """Packed variable-length sequences: q, k, v bf16 [T, H, d]; cu_seqlens int32 [S + 1]
    on the same device (sequence s = tokens cu[s] .. cu[s+1]-1); max_seqlen >= every
    length.  Returns O [T, H, d] and the natural-log LSE [H, T]."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError(f"{n} must be a CUDA bf16 tensor")
        if t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous [T, H, d] tensor")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    if (not isinstance(cu_seqlens, torch.Tensor) or cu_seqlens.dtype != torch.int32
            or cu_seqlens.device != q.device or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2
            or not cu_seqlens.is_contiguous()):
        raise TypeError("cu_seqlens must be a contiguous int32 [S + 1] tensor on q's device")
    T, H, d = q.shape
    S = cu_seqlens.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    _check_out(o, (T, H, d), torch.bfloat16, q.device, "o")
    _check_out(lse, (H, T), torch.float32, q.device, "lse")
    st = load_library().attn_fwd_bf16_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                             lse.data_ptr(), cu_seqlens.data_ptr(), S,
                                             int(max_seqlen), T, H, d, float(scale),
                                             int(bool(causal)), int(window), _stream_handle(stream))
    _raise_if(st, "attn_fwd_bf16_varlen")
    return o, lse


def attn_decode_workspace_bytes(B: int, H: int, nq: int, d: int, page_size: int, max_pages: int,
                                num_splits: int = 0) -> int:
    """Workspace bytes attn_decode_bf16_paged needs for that plan (0: one split)."""
    return int(load_library().attn_decode_workspace_bytes(B, H, nq, d, page_size, max_pages,
                                                          num_splits))


def _decode_args(q, k_cache, v_cache, page_table, seq_lens, scale, o, lse):
    _check_bhnd("q", q, torch.bfloat16)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check_bhnd(n, t, torch.bfloat16)
    if v_cache.shape != k_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    B, H, nq, d = q.shape
    num_pages, Hc, page_size, dc = k_cache.shape
    if Hc != H or dc != d:
        raise ValueError("cache heads / head dim must match q")
    for n, t in (("page_table", page_table), ("seq_lens", seq_lens)):
        if (not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or t.device != q.device
                or not t.is_contiguous()):
            raise TypeError(f"{n} must be a contiguous int32 tensor on q's device")
    if page_table.dim() != 2 or page_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("page_table must be [B, max_pages] and seq_lens [B]")
    max_pages = page_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, nq), dtype=torch.float32, device=q.device)
    _check_out(o, (B, H, nq, d), torch.bfloat16, q.device, "o")
    _check_out(lse, (B, H, nq), torch.float32, q.device, "lse")
    return B, H, nq, d, num_pages, page_size, max_pages, scale, o, lse


def attn_decode_bf16_paged(q, k_cache, v_cache, page_table, seq_lens, scale: float | None = None,
                           num_splits: int = 0, workspace=None, o=None, lse=None, stream=None):
    """One decoding step over a paged KV cache.  q: bf16 [B, H, nq, d] (the nq newest
    tokens, nq <= 8); k_cache, v_cache: bf16 [num_pages, H, page_size, d]; page_table:
    int32 [B, max_pages]; seq_lens: int32 [B] (cached lengths, the new tokens included).
    Returns O [B, H, nq, d] and the natural-log LSE [B, H, nq].  A workspace of
    attn_decode_workspace_bytes(...) is allocated when none is given."""
    B, H, nq, d, num_pages, page_size, max_pages, scale, o, lse = _decode_args(
        q, k_cache, v_cache, page_table, seq_lens, scale, o, lse)
    if workspace is None:
        nbytes = attn_decode_workspace_bytes(B, H, nq, d, page_size, max_pages, num_splits)
        workspace = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=q.device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    st = load_library().attn_decode_bf16_paged(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), page_table.data_ptr(),
        seq_lens.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, nq, d, page_size, num_pages,
        max_pages, float(scale), int(num_splits), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _raise_if(st, "attn_decode_bf16_paged")
    return o, lse


def attn_decode_bf16_paged_noalloc(q, k_cache, v_cache, page_table, seq_lens,
                                   scale: float | None = None, num_splits: int = 0, o=None,
                                   lse=None, stream=None):
    """attn_decode_bf16_paged for callers that cannot allocate device memory when they
    decode: the split partials go to the library's own 16 MiB device scratch (no
    workspace).  Calls on one device must be ordered (they share the scratch); a
    forced num_splits whose partials exceed 16 MiB raises AttnError.  This wrapper
    allocates o and lse when they are not given; pass them to allocate nothing."""
    B, H, nq, d, num_pages, page_size, max_pages, scale, o, lse = _decode_args(
        q, k_cache, v_cache, page_table, seq_lens, scale, o, lse)
    st = load_library().attn_decode_bf16_paged_noalloc(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), page_table.data_ptr(),
        seq_lens.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, nq, d, page_size, num_pages,
        max_pages, float(scale), int(num_splits), _stream_handle(stream))
    _raise_if(st, "attn_decode_bf16_paged_noalloc")
    return o, lse


def _quant_outputs(x, block, x8, scales):
    B, H, N, d = x.shape
    nblk = (N + block - 1) // block
    if x8 is None:
        x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    elif (x8.dtype != torch.uint8 or tuple(x8.shape) != (B, H, N, d) or x8.device != x.device
          or not x8.is_contiguous()):
        raise TypeError(f"x8 must be a contiguous uint8 tensor of shape {(B, H, N, d)} on {x.device}")
    if scales is None:
        scales = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    elif (scales.dtype != torch.float32 or tuple(scales.shape) != (B, H, nblk)
          or scales.device != x.device or not scales.is_contiguous()):
        raise TypeError(f"scales must be a contiguous float32 tensor of shape {(B, H, nblk)} on {x.device}")
    return x8, scales


def attn_quantize_fp8_blockwise(x, block: int = 128, x8=None, scales=None, stream=None):
    """Per-(head, block of `block` rows) E4M3 quantisation, block = 128 or 64 (the
    head-dim-aware Q / K block at d = 64); returns (x8 uint8 codes, fp32 scales)."""
    _check_bhnd("x", x, torch.bfloat16)
    B, H, N, d = x.shape
    x8, scales = _quant_outputs(x, block, x8, scales)
    st = load_library().attn_quantize_fp8_blockwise(x.data_ptr(), x8.data_ptr(),
                                                    scales.data_ptr(), B, H, N, d, int(block),
                                                    _stream_handle(stream))
    _raise_if(st, "attn_quantize_fp8_blockwise")
    return x8, scales


def _fp8_format(fmt) -> int:
    if fmt not in _FP8_FORMATS:
        raise ValueError(f"unknown FP8 format {fmt!r} (use 'e4m3', 'e5m2' or 'e4m3_pow2')")
    return _FP8_FORMATS[fmt]


def attn_quantize_fp8_blockwise_fmt(x, fmt, block: int = 128, x8=None, scales=None, stream=None):
    """Per-(head, 128-row block) quantisation into E4M3 ('e4m3': scale = amax/448), E5M2
    ('e5m2': scale = amax/57344) or E4M3 with power-of-two scales ('e4m3_pow2': the smallest
    2^k >= amax/448); returns (x8 uint8 codes, fp32 scales)."""
    _check_bhnd("x", x, torch.bfloat16)
    B, H, N, d = x.shape
    x8, scales = _quant_outputs(x, block, x8, scales)
    st = load_library().attn_quantize_fp8_blockwise_fmt(x.data_ptr(), x8.data_ptr(),
                                                        scales.data_ptr(), B, H, N, d, int(block),
                                                        _fp8_format(fmt), _stream_handle(stream))
    _raise_if(st, "attn_quantize_fp8_blockwise_fmt")
    return x8, scales


def attn_quantize_fp8_hadamard(x, block: int = 128, x8=None, scales=None, stream=None):
    """Rows of x times the orthonormal Walsh-Hadamard matrix, then per-block E4M3
    quantisation (for Q and K); returns (x8 uint8 codes, fp32 scales)."""
    _check_bhnd("x", x, torch.bfloat16)
    B, H, N, d = x.shape
    x8, scales = _quant_outputs(x, block, x8, scales)
    st = load_library().attn_quantize_fp8_hadamard(x.data_ptr(), x8.data_ptr(),
                                                   scales.data_ptr(), B, H, N, d, int(block),
                                                   _stream_handle(stream))
    _raise_if(st, "attn_quantize_fp8_hadamard")
    return x8, scales


def attn_fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, scale: float | None = None,
                 causal: bool = False, window: int = 0, o=None, lse=None, stream=None):
    """Forward pass on E4M3 operands (uint8 codes or float8_e4m3fn) with per-block descales."""
    return _fwd_fp8("attn_fwd_fp8", None, q8, k8, v8, descale_q, descale_k, descale_v, scale,
                    causal, window, o, lse, stream)


def attn_fwd_fp8_fmt(q8, k8, v8, descale_q, descale_k, descale_v, qk_fmt, v_fmt="e4m3",
                     scale: float | None = None, causal: bool = False, window: int = 0, o=None,
                     lse=None, stream=None):
    """attn_fwd_fp8 with Q and K both in qk_fmt ('e4m3', 'e5m2' or 'e4m3_pow2', from
    attn_quantize_fp8_blockwise_fmt) and V in v_fmt ('e4m3' or 'e4m3_pow2': power-of-two
    block scales, applied through P's exponent)."""
    return _fwd_fp8("attn_fwd_fp8_fmt", (_fp8_format(qk_fmt), _fp8_format(v_fmt)), q8, k8, v8,
                    descale_q, descale_k, descale_v, scale, causal, window, o, lse, stream)


def attn_fwd_fp8_blocks(q8, k8, v8, descale_q, descale_k, descale_v, qk_block: int | None = None,
                        qk_fmt="e4m3", v_fmt="e4m3", scale: float | None = None,
                        causal: bool = False, window: int = 0, o=None, lse=None, stream=None):
    """attn_fwd_fp8_fmt with Q and K scaled per block of qk_block rows (64 or 128; V per 128
    rows).  The default is the head-dim-aware block, attn_fp8_qk_block_rows(d): 64 rows at
    d = 64, 128 above.  Quantise Q and K with attn_quantize_fp8_blockwise(x, block=qk_block)."""
    d = q8.shape[-1]
    if qk_block is None:
        qk_block = attn_fp8_qk_block_rows(d)
    return _fwd_fp8("attn_fwd_fp8_blocks", (_fp8_format(qk_fmt), _fp8_format(v_fmt), int(qk_block)),
                    q8, k8, v8, descale_q, descale_k, descale_v, scale, causal, window, o, lse,
                    stream, qk_block=int(qk_block))


def attn_fp8_qk_block_rows(d: int) -> int:
    """Rows per Q / K scale block under head-dim-aware scaling: min(d, 128)."""
    return int(load_library().attn_fp8_qk_block_rows(int(d)))


def attn_fwd_schedule(B: int, H: int, N: int, d: int, causal: bool = False, window: int = 0,
                      sm_count: int = 152) -> dict:
    """How a batched forward call would spread its work over sm_count SMs (no device is
    touched): the walk (0 pairs, 1 single units with a plain stride, 2 rotated), the grid,
    the number of sub-units, the walk's constants and the query blocks per head."""
    out = (ctypes.c_int * 8)()
    st = load_library().attn_fwd_schedule(int(B), int(H), int(N), int(d), int(bool(causal)),
                                          int(window), int(sm_count), out)
    _raise_if(st, "attn_fwd_schedule")
    keys = ("walk", "grid", "subs", "first", "a", "m", "step", "num_qblk")
    return dict(zip(keys, (int(x) for x in out)))


def _fwd_fp8(entry, qk_fmt, q8, k8, v8, descale_q, descale_k, descale_v, scale, causal, window,
             o, lse, stream, qk_block=128):
    views = []
    for n, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
            t = t.view(torch.uint8)
        _check_bhnd(n, t, torch.uint8)
        views.append(t)
    q8, k8, v8 = views
    if k8.shape != q8.shape or v8.shape != q8.shape:
        raise ValueError("q8, k8, v8 must have the same shape")
    B, H, N, d = q8.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    _check_out(o, (B, H, N, d), torch.bfloat16, q8.device, "o")
    _check_out(lse, (B, H, N), torch.float32, q8.device, "lse")
    nqk = (N + qk_block - 1) // qk_block
    for n, t, nb in (("descale_q", descale_q, nqk), ("descale_k", descale_k, nqk),
                     ("descale_v", descale_v, (N + 127) // 128)):
        _check_out(t, (B, H, nb), torch.float32, q8.device, n)
    args = [q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), descale_q.data_ptr(), descale_k.data_ptr(),
            descale_v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, float(scale),
            int(bool(causal)), int(window)]
    if qk_fmt is not None:
        args.extend(qk_fmt)
    st = getattr(load_library(), entry)(*args, _stream_handle(stream))
    _raise_if(st, entry)
    return o, lse


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load_library().attn_get_device_status(_stream_handle(stream)))


def attn_selftest_wait_timeout(timeout_ns: int = 50_000_000, stream=None) -> None:
    """Run the bounded-wait self-test kernel (it records ATTN_ERR_TIMEOUT on purpose)."""
    st = load_library().attn_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream))
    _raise_if(st, "attn_selftest_wait_timeout")


def attn_selftest_fwd_withheld_load(q, k, v, o, lse, causal: bool = False, withheld: int = 2,
                                    timeout_ns: int = 20_000_000, stream=None) -> None:
    """Run the bf16 forward kernel with K/V load `withheld` of every CTA never issued and
    every wait bounded by timeout_ns: the kernel aborts and records ATTN_ERR_TIMEOUT
    (read it with attn_get_device_status); o and lse are left unspecified."""
    B, H, N, d = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_bhnd(n, t, torch.bfloat16)
    st = load_library().attn_selftest_fwd_withheld_load(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
        int(bool(causal)), int(withheld), int(timeout_ns), _stream_handle(stream))
    _raise_if(st, "attn_selftest_fwd_withheld_load")


def attn_selftest_quant_withheld_load(x, x8, scales, withheld: int = 1,
                                      timeout_ns: int = 20_000_000, stream=None) -> None:
    """Run the E4M3 block quantiser with block load `withheld` of every CTA never issued
    and every wait bounded by timeout_ns (it records ATTN_ERR_TIMEOUT)."""
    B, H, N, d = x.shape
    _check_bhnd("x", x, torch.bfloat16)
    st = load_library().attn_selftest_quant_withheld_load(
        x.data_ptr(), x8.data_ptr(), scales.data_ptr(), B, H, N, d, int(withheld),
        int(timeout_ns), _stream_handle(stream))
    _raise_if(st, "attn_selftest_quant_withheld_load")


def attn_selftest_bwd_withheld_load(q, k, v, o, dout, lse, dq, dk, dv, workspace,
                                    causal: bool = False, withheld: int = 2,
                                    timeout_ns: int = 20_000_000, stream=None) -> None:
    """Run the backward kernels with ring load `withheld` of every CTA never issued and
    every wait bounded by timeout_ns (they record ATTN_ERR_TIMEOUT)."""
    B, H, N, d = q.shape
    st = load_library().attn_selftest_bwd_withheld_load(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), B, H, N, d, int(bool(causal)),
        int(withheld), int(timeout_ns), _stream_handle(stream))
    _raise_if(st, "attn_selftest_bwd_withheld_load")


def attn_selftest_fp8_convert(first: int, count: int, fmt="e4m3", codes=None, stream=None):
    """Device FP8 codes (the quantisers' conversion) of the fp32 bit patterns first ..
    first + count - 1; returns a uint8 CUDA tensor of count codes."""
    if codes is None:
        codes = torch.empty(int(count), dtype=torch.uint8, device="cuda")
    st = load_library().attn_selftest_fp8_convert(int(first), int(count), _fp8_format(fmt),
                                                  codes.data_ptr(), _stream_handle(stream))
    _raise_if(st, "attn_selftest_fp8_convert")
    return codes

