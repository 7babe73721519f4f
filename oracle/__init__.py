"""Float64 CPU oracle for the fused exact-attention forward pass.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product path (the
CUDA library and its Python binding) never imports, links or runs it, and it
shares no code with them; the two meet only through the seeded input
generators, which hold none of the method's arithmetic.

The arithmetic lives in ``attn_oracle.c`` (plain C, float64, OpenMP over rows);
this module builds it with gcc and marshals numpy arrays into it.

Pages cited (titles as published):
  [WGC] "Warp Group Cluster 优化：Flash Attention V3 在 H100 上的 FP8 融合计算实践"
  [JJ]  "大模型加速-核心网络算子-Flash Attention V3"
  [YT]  "FlashAttention V3：优化框架吞吐量的关键技术实践"

Functions and the passage each follows:
  attn_f64 / attn_rows_f64   standard attention, the exact result the method
                             reaches ([WGC] §背景; [YT] §1.2 fused softmax+mask+matmul)
  online_replay_f64          block-wise online softmax ([WGC] §2 GEMM-Softmax 融合流水线)
  key_allowed                mask sets ([YT] §2.1.2 稀疏性感知的Mask优化)
  e4m3_encode / e4m3_decode  E4M3 format ([JJ] §1.5 低精度FP8)
  e5m2_encode / e5m2_decode  E5M2 format, the wider-range one ([JJ] §1.5; [WGC] §3 lists
                             both formats)
  quantize_fp8_blockwise     per-block scaling ([WGC] §3 FP8 量化与精度保持), into E4M3
                             (fmt="e4m3", scale = amax/448), E5M2 (fmt="e5m2",
                             scale = amax/57344), or E4M3 with a power-of-two scale per
                             block (fmt="e4m3_pow2": the smallest 2^k >= amax/448)
  fp8_block_rows             head-dim-aware scaling ([WGC] §3 头维度感知量化: the scaling
                             is tuned separately for head dims 64 and 128 so that small head
                             dims lose no precision): rows per scale block of Q, K and V
  dequantize                 x ~= x8 * scale for the block, the inverse map
  hadamard_rotate_f32        incoherent processing before quantisation ([JJ] §1
                             item 3, 块量化和无相关处理): orthonormal Walsh-Hadamard
                             rotation of each row, in fp32 in a fixed butterfly order
  quantize_fp8_hadamard      the rotation followed by quantize_fp8_blockwise
  attn_varlen_f64            variable-length sequences packed without padding ([YT]
                             §1.1 可变序列长度): each sequence attends only within
                             itself, masks relative to its own first token
  attn_bwd_f64               gradients of the forward pass (the backward pass the pages
                             mention for training: [YT] §2.3.2 流水线并行, forward and
                             backward of micro-batches; [JJ] §2.3-2.4 call their
                             kernel the forward pass): dQ, dK, dV of sum(dO * O)
  attn_varlen_bwd_f64        the backward pass over packed variable-length sequences
                             (attn_bwd_f64 of each sequence on its own)
  attn_decode_paged_f64      a decoding step against a paged KV cache ([JJ] §3 总结:
                             tokens generated one at a time over cached K/V; [WGC]
                             §局限性与后续方向 item 2: PagedAttention KV-cache management)
Every function is pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

E4M3_MAX = 448.0


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``oracle/_build/liboracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lp = ctypes.POINTER(ctypes.c_long)
        L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
        lib.oracle_key_allowed.argtypes = [L, L, L, I, L]
        lib.oracle_key_allowed.restype = I
        lib.oracle_attn_rows_f64.argtypes = [dp, dp, dp, L, L, D, I, L, lp, L, dp, dp, I]
        lib.oracle_attn_rows_f64.restype = I
        lib.oracle_attn_f64.argtypes = [dp, dp, dp, L, L, L, D, I, L, dp, dp, I]
        lib.oracle_attn_f64.restype = I
        lib.oracle_online_replay_f64.argtypes = [dp, dp, dp, L, L, D, I, L, L, L, D, dp, dp]
        lib.oracle_online_replay_f64.restype = None
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_float
        lib.oracle_e4m3_encode_array.argtypes = [fp, u8p, L]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_quantize_fp8_blockwise.argtypes = [fp, u8p, fp, L, L, L, L]
        lib.oracle_quantize_fp8_blockwise.restype = None
        lib.oracle_e5m2_encode.argtypes = [ctypes.c_float]
        lib.oracle_e5m2_encode.restype = ctypes.c_uint8
        lib.oracle_e5m2_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e5m2_decode.restype = ctypes.c_float
        lib.oracle_e5m2_encode_array.argtypes = [fp, u8p, L]
        lib.oracle_e5m2_encode_array.restype = None
        lib.oracle_quantize_fp8_blockwise_fmt.argtypes = [fp, u8p, fp, L, L, L, L, I]
        lib.oracle_quantize_fp8_blockwise_fmt.restype = None
        lib.oracle_hadamard_rotate_f32.argtypes = [fp, fp, L, L, ctypes.c_float]
        lib.oracle_hadamard_rotate_f32.restype = None
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    """Exact widening to contiguous float64 (bf16 and fp32 values are representable)."""
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def key_allowed(i: int, j: int, N: int, causal: bool, window: int) -> bool:
    return bool(_load().oracle_key_allowed(i, j, N, int(causal), int(window)))


def attn_f64(q, k, v, scale: float, causal: bool = False, window: int = 0,
             nthreads: int = 0):
    """All rows of every head.  q, k, v: [..., N, d] -> (O [..., N, d], LSE [..., N])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    shape = q.shape
    N, d = shape[-2], shape[-1]
    BH = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    o = np.empty(shape, dtype=np.float64)
    lse = np.empty(shape[:-1], dtype=np.float64)
    _load().oracle_attn_f64(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                            _ptr(v, ctypes.c_double), BH, N, d, float(scale), int(causal),
                            int(window), _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                            int(nthreads))
    return o, lse


def attn_rows_f64(q, k, v, rows, scale: float, causal: bool = False, window: int = 0,
                  nthreads: int = 0, return_threads: bool = False):
    """Selected query rows of ONE head.  q, k, v: [N, d]; rows: R indices.

    Returns (O [R, d], LSE [R]) (and the thread count when ``return_threads``).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise ValueError("row index out of range")
    R = rows.size
    o = np.empty((R, d), dtype=np.float64)
    lse = np.empty((R,), dtype=np.float64)
    nt = _load().oracle_attn_rows_f64(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double), N, d,
        float(scale), int(causal), int(window), _ptr(rows, ctypes.c_long), R,
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double), int(nthreads))
    if return_threads:
        return o, lse, nt
    return o, lse


def attn_varlen_f64(q, k, v, cu_seqlens, scale: float, causal: bool = False, window: int = 0):
    """Packed variable-length sequences.  q, k, v: [T, H, d] (bf16 or float values),
    cu_seqlens: S + 1 non-decreasing token offsets with cu[0] = 0 and cu[S] = T;
    sequence s is tokens [cu[s], cu[s+1]).  Returns (O [T, H, d], LSE [H, T]) float64:
    attn_f64 of each sequence on its own (its rows, its keys, its mask)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    T, H, d = q.shape
    if cu[0] != 0 or cu[-1] != T or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must rise from 0 to T")
    o = np.zeros((T, H, d))
    lse = np.zeros((H, T))
    for a, b in zip(cu, cu[1:]):
        if b == a:
            continue
        # [n, H, d] -> [H, n, d] for the per-head definition
        oh, lh = attn_f64(q[a:b].transpose(1, 0, 2), k[a:b].transpose(1, 0, 2),
                          v[a:b].transpose(1, 0, 2), scale, causal=causal, window=window)
        o[a:b] = oh.transpose(1, 0, 2)
        lse[:, a:b] = lh
    return o, lse


def attn_varlen_bwd_f64(q, k, v, do, cu_seqlens, scale: float, causal: bool = False,
                        window: int = 0):
    """Backward pass over packed variable-length sequences ([T, H, d] tensors and
    cu_seqlens as attn_varlen_f64): attn_bwd_f64 of each sequence on its own.  Returns
    (dQ, dK, dV) float64 [T, H, d]."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    T = q.shape[0]
    if cu[0] != 0 or cu[-1] != T or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must rise from 0 to T")
    out = [np.zeros_like(q) for _ in range(3)]
    for a, b in zip(cu, cu[1:]):
        if b == a:
            continue
        g = attn_bwd_f64(*(x[a:b].transpose(1, 0, 2) for x in (q, k, v, do)), scale,
                         causal=causal, window=window)
        for o_, g_ in zip(out, g):
            o_[a:b] = g_.transpose(1, 0, 2)
    return tuple(out)


def attn_bwd_f64(q, k, v, do, scale: float, causal: bool = False, window: int = 0):
    """Gradients of O = softmax(scale * Q K^T + mask) V for the upstream gradient dO.
    q, k, v, do: [..., N, d].  With P the masked softmax (two-pass, as attn_f64):
        dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij (= dO_i . O_i),
        dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.
    Returns (dQ, dK, dV) float64, shaped like q."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    N = q.shape[-2]
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    allowed = np.ones((N, N), dtype=bool)
    if causal:
        allowed &= j <= i
    if window > 0:
        allowed &= j >= i - window
        if not causal:
            allowed &= j <= i + window
    s = scale * (q @ np.swapaxes(k, -1, -2))
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.where(allowed, np.exp(s - m), 0.0)
    p = e / e.sum(axis=-1, keepdims=True)
    dv = np.swapaxes(p, -1, -2) @ do
    dp = do @ np.swapaxes(v, -1, -2)
    dd = (p * dp).sum(axis=-1, keepdims=True)
    ds = p * (dp - dd)
    dq = scale * (ds @ k)
    dk = scale * (np.swapaxes(ds, -1, -2) @ q)
    return dq, dk, dv


def attn_decode_paged_f64(q, k_cache, v_cache, page_table, seq_lens, scale: float):
    """One decoding step over a paged KV cache.
    q: [B, H, nq, d], the nq newest tokens of each sequence; k_cache, v_cache:
    [num_pages, H, page_size, d]; page_table: [B, max_pages] page numbers in order;
    seq_lens: [B] cached lengths L_b >= nq (the new tokens' keys included).  Key t of
    sequence b is row t % page_size of page page_table[b][t // page_size]; query i
    sits at position L_b - nq + i and sees keys 0 .. L_b - nq + i.
    Returns (O [B, H, nq, d], LSE [B, H, nq]) float64."""
    q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
    pt = np.asarray(page_table, dtype=np.int64)
    lens = [int(x) for x in np.asarray(seq_lens).reshape(-1)]
    B, H, nq, d = q.shape
    ps = kc.shape[2]
    o = np.zeros((B, H, nq, d))
    lse = np.zeros((B, H, nq))
    for b in range(B):
        L = lens[b]
        if L < nq:
            raise ValueError("seq_lens must be >= nq")
        t = np.arange(L)
        pages = pt[b, t // ps]
        rows = t % ps
        for h in range(H):
            K = kc[pages, h, rows]          # [L, d], keys in sequence order
            V = vc[pages, h, rows]
            s = scale * (q[b, h] @ K.T)     # [nq, L]
            for i in range(nq):
                last = L - nq + i           # causal, aligned to the end of the sequence
                si = s[i, :last + 1]
                m = si.max()
                e = np.exp(si - m)
                o[b, h, i] = (e @ V[:last + 1]) / e.sum()
                lse[b, h, i] = m + np.log(e.sum())
    return o, lse


def online_replay_f64(q, k, v, scale: float, causal: bool, window: int, BM: int, BN: int,
                      tau: float = 0.0):
    """Tile-by-tile online-softmax replay of ONE head.  q, k, v: [N, d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    o = np.empty((N, d), dtype=np.float64)
    lse = np.empty((N,), dtype=np.float64)
    _load().oracle_online_replay_f64(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double), N, d,
        float(scale), int(causal), int(window), int(BM), int(BN), float(tau),
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    return o, lse


def e4m3_encode(x) -> np.ndarray:
    """float32 array -> uint8 E4M3 codes (RNE, saturating to +-448)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint8),
                                     x.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    """uint8 E4M3 codes -> float32 values (exact)."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float32)
    return table[np.asarray(codes, dtype=np.uint8)]


def e5m2_encode(x) -> np.ndarray:
    """float32 array -> uint8 E5M2 codes (RNE, saturating to +-57344)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e5m2_encode_array(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint8),
                                     x.size)
    return out


def e5m2_decode(codes) -> np.ndarray:
    """uint8 E5M2 codes -> float32 values (exact; exponent field 31 gives inf / NaN)."""
    lib = _load()
    table = np.array([lib.oracle_e5m2_decode(c) for c in range(256)], dtype=np.float32)
    return table[np.asarray(codes, dtype=np.uint8)]


FP8_FORMATS = {"e4m3": 0, "e5m2": 1, "e4m3_pow2": 2}


def quantize_fp8_blockwise(x, block: int = 128, fmt: str = "e4m3"):
    """x: [..., N, d] (bf16 values) -> (x8 uint8 [..., N, d], scales float32 [..., ceil(N/block)]).
    fmt "e4m3" (scale = amax/448), "e5m2" (scale = amax/57344) or "e4m3_pow2" (E4M3 codes,
    scale = the smallest power of two >= amax/448)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu").to(torch.float32).numpy()
    x = np.ascontiguousarray(x, dtype=np.float32)
    shape = x.shape
    N, d = shape[-2], shape[-1]
    BH = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    nblk = (N + block - 1) // block
    x8 = np.empty(shape, dtype=np.uint8)
    scales = np.empty(shape[:-2] + (nblk,), dtype=np.float32)
    if fmt == "e4m3":
        _load().oracle_quantize_fp8_blockwise(_ptr(x, ctypes.c_float), _ptr(x8, ctypes.c_uint8),
                                              _ptr(scales, ctypes.c_float), BH, N, d, int(block))
    else:
        _load().oracle_quantize_fp8_blockwise_fmt(_ptr(x, ctypes.c_float), _ptr(x8, ctypes.c_uint8),
                                                  _ptr(scales, ctypes.c_float), BH, N, d, int(block),
                                                  FP8_FORMATS[fmt])
    return x8, scales


def hadamard_scale(d: int) -> np.float32:
    """c = fp32(1 / sqrt(d)): the double value rounded once to fp32."""
    return np.float32(1.0 / np.sqrt(np.float64(d)))


def hadamard_rotate_f32(x) -> np.ndarray:
    """Rows of x ([..., d], bf16 or fp32 values; d a power of two) times H_d / sqrt(d),
    computed in fp32 by the radix-2 butterfly sweep h = 1, 2, ..., d/2 and a final
    multiply by hadamard_scale(d)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu").to(torch.float32).numpy()
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = x.shape[-1]
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    y = np.empty_like(x)
    _load().oracle_hadamard_rotate_f32(_ptr(x, ctypes.c_float), _ptr(y, ctypes.c_float),
                                       x.size // d, d, hadamard_scale(d))
    return y


def quantize_fp8_hadamard(x, block: int = 128):
    """Incoherent processing then per-block quantisation: quantize_fp8_blockwise of
    hadamard_rotate_f32(x).  Dequantised values approximate x @ H_d / sqrt(d)."""
    return quantize_fp8_blockwise(hadamard_rotate_f32(x), block)


def fp8_block_rows(d: int, operand: str) -> int:
    """Rows per FP8 scale block under head-dim-aware scaling.

    [WGC] §3 FP8 量化与精度保持 says the scaling strategy is tuned separately for head
    dims 64 and 128 so that small head dims do not lose precision, and gives no rule.
    Reading: Q and K, whose products with each other run over the d entries of a row,
    are scaled per block of min(d, 128) rows -- a d x d block at d = 64, the 128-row
    block at d >= 128 (the FP8 workload's block); V, whose error in O averages over keys
    rather than over d, keeps 128-row blocks at every d."""
    if operand not in ("q", "k", "v"):
        raise ValueError("operand must be 'q', 'k' or 'v'")
    if d < 1:
        raise ValueError("head dim must be positive")
    return 128 if operand == "v" else min(int(d), 128)


def dequantize(x8, scales, block: int = 128, fmt: str = "e4m3") -> np.ndarray:
    """x_hat = decode(x8) * scale of its row block, in float64 (exact products)."""
    x8 = np.asarray(x8, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.float32)
    vals = (e5m2_decode(x8) if fmt == "e5m2" else e4m3_decode(x8)).astype(np.float64)
    N = x8.shape[-2]
    row_scale = np.repeat(scales.astype(np.float64), block, axis=-1)[..., :N]
    return vals * row_scale[..., None]
