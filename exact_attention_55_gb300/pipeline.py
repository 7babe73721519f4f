"""Attention on host-resident tensors with copies overlapped with the kernel.

For callers whose Q, K, V live in (pinned) host memory and who want O and LSE
back in host memory.  The batch is cut into chunks; while the kernel runs on
chunk c, chunk c+1 is copied to the device and chunk c-1's O and LSE are copied
back, on five CUDA streams (one upload stream per input tensor, one for the
kernel, one for the copies back) with two device buffers per tensor.  The arithmetic
is the C-ABI call `attn_fwd_bf16` on each chunk; this module only moves memory
and orders streams.
"""
from __future__ import annotations

import math

import torch

from . import attn_fwd_bf16


class HostAttention:
    """Reusable pipeline for bf16 [B, H, N, d] host tensors on one CUDA device.

    Allocates two device buffers per tensor for one chunk of `B / chunks`
    batches (torch allocates them once, at construction).  Call it with pinned
    host tensors; it enqueues all copies and kernels and makes the caller's
    current stream wait for the last copy back, without synchronising the host.
    """

    def __init__(self, B: int, H: int, N: int, d: int, chunks: int = 4, device=None):
        if B % chunks != 0:
            raise ValueError("B must be a multiple of chunks")
        self.B, self.H, self.N, self.d, self.chunks = B, H, N, d, chunks
        self.bc = B // chunks
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        shape = (self.bc, H, N, d)
        self.qd = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.kd = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.vd = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.od = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.ld = [torch.empty((self.bc, H, N), dtype=torch.float32, device=dev) for _ in range(2)]
        # one input stream per tensor, so the three uploads can use separate copy engines
        self.s_ins = [torch.cuda.Stream(device=dev) for _ in range(3)]
        self.s_comp = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        # buffer-slot state carried across calls: the chunk counter picks the slot, and
        # the last compute / copy-back that used each slot gates its next reuse
        self._chunk = 0
        self._done_comp = [None, None]  # compute finished with slot -> inputs may be overwritten
        self._done_out = [None, None]   # copy-back finished with slot -> outputs may be overwritten

    def h2d_bytes(self) -> int:
        return 3 * self.B * self.H * self.N * self.d * 2

    def d2h_bytes(self) -> int:
        return self.B * self.H * self.N * (self.d * 2 + 4)

    def __call__(self, qh, kh, vh, oh, lseh, scale: float | None = None, causal: bool = False,
                 window: int = 0, wait_caller: bool = True) -> None:
        """Enqueue one pass.  With wait_caller (the default) the copies start only after
        the work already queued on the caller's stream, so inputs written there (for
        instance the outputs of a previous call) are seen.  With wait_caller=False the
        inputs must already be in host memory (written by the CPU): the uploads of this
        call may then overlap the previous call's last kernels and copies back."""
        for n, t in (("q", qh), ("k", kh), ("v", vh), ("o", oh)):
            if t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != (
                    self.B, self.H, self.N, self.d):
                raise TypeError(f"{n} must be a host bf16 tensor of shape {(self.B, self.H, self.N, self.d)}")
        if lseh.is_cuda or lseh.dtype != torch.float32 or tuple(lseh.shape) != (self.B, self.H, self.N):
            raise TypeError(f"lse must be a host float32 tensor of shape {(self.B, self.H, self.N)}")
        if scale is None:
            scale = 1.0 / math.sqrt(self.d)
        caller = torch.cuda.current_stream()
        if wait_caller:
            for st in self.s_ins:
                st.wait_stream(caller)
        self.s_out.wait_stream(caller)
        done_comp, done_out = self._done_comp, self._done_out
        last = None
        for c in range(self.chunks):
            slot = self._chunk & 1
            self._chunk += 1
            b0, b1 = c * self.bc, (c + 1) * self.bc
            evs_in = []
            for st, dst, src in zip(self.s_ins, (self.qd, self.kd, self.vd), (qh, kh, vh)):
                with torch.cuda.stream(st):
                    if done_comp[slot] is not None:
                        st.wait_event(done_comp[slot])
                    dst[slot].copy_(src[b0:b1], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(st)
                    evs_in.append(ev)
            with torch.cuda.stream(self.s_comp):
                for ev in evs_in:
                    self.s_comp.wait_event(ev)
                if done_out[slot] is not None:
                    self.s_comp.wait_event(done_out[slot])
                attn_fwd_bf16(self.qd[slot], self.kd[slot], self.vd[slot], scale=scale,
                              causal=causal, window=window, o=self.od[slot], lse=self.ld[slot],
                              stream=self.s_comp)
                ev_c = torch.cuda.Event()
                ev_c.record(self.s_comp)
                done_comp[slot] = ev_c
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_c)
                oh[b0:b1].copy_(self.od[slot], non_blocking=True)
                lseh[b0:b1].copy_(self.ld[slot], non_blocking=True)
                ev_o = torch.cuda.Event()
                ev_o.record(self.s_out)
                done_out[slot] = ev_o
                last = ev_o
        caller.wait_event(last)
        caller.wait_stream(self.s_comp)
