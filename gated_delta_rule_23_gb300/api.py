"""Tensor-level binding of the C ABI (argument marshalling only).

``kda_fwd`` mirrors the argument list of flash_kda.fwd in the FlashKDA README
mirror (ai-feeds.com, section "内核 API"): the caller passes CUDA tensors and a
pre-allocated ``out`` (and ``final_state``); every step of the computation runs in
libkda.so.  PyTorch is used only to hold device memory and to name the stream.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _native
from ._native import KDA_DTYPE_BF16, KDA_DTYPE_FP32, KDA_DTYPE_NONE, KDA_OK, KDAError

D = 128


def _check(t: torch.Tensor, name: str, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def kda_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
            scale: float, out: torch.Tensor, A_log: torch.Tensor, dt_bias: torch.Tensor, lower_bound: float,
            initial_state: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
            cu_seqlens: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
            workspace: Optional[torch.Tensor] = None, stage_events=None, noalloc: bool = False,
            recurrent: bool = False) -> None:
    """KDA chunked forward on CUDA tensors; writes ``out`` and ``final_state`` in place.

    q, k, v, g: bf16 [B, T, H, 128]; beta: bf16 [B, T, H]; out: bf16 [B, T, H, 128];
    A_log: fp32 [H]; dt_bias: fp32 [H, 128]; states: bf16 or fp32 [N, H, 128, 128] (same dtype
    when both are given); cu_seqlens: int64 [N + 1] with B = 1.  Runs asynchronously on
    ``stream`` (default: the current stream).  ``workspace``: optional uint8 CUDA tensor of at
    least ``workspace_size(...)`` bytes (kda_fwd_ws); without it the library's pool provides one.
    ``stage_events``: optional three recorded-once torch.cuda.Event objects marking the start of
    the prep kernel, the prep/recurrence boundary and the end (kda_fwd_ws_profiled; needs
    ``workspace``).  ``noalloc``: use the library's static workspace (kda_fwd_noalloc).
    ``recurrent``: evaluate token by token (kda_fwd_recurrent; decode and short sequences, no
    workspace).
    """
    lib = _native.load()
    if q.dim() != 4 or q.shape[-1] != D:
        raise ValueError("q must be [B, T, H, 128]")
    B, T, H, _ = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_fwd needs CUDA tensors (use KDAHostRunner for host data)")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("out", out)):
        _check(t, name, torch.bfloat16, (B, T, H, D), dev)
    _check(beta, "beta", torch.bfloat16, (B, T, H), dev)
    _check(A_log, "A_log", torch.float32, (H,), dev)
    _check(dt_bias, "dt_bias", torch.float32, (H, D), dev)
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be int64 [N + 1]")
        N = cu_seqlens.numel() - 1
        _check(cu_seqlens, "cu_seqlens", torch.int64, (N + 1,), dev)
    else:
        N = B
    sd = None
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        if t is None:
            continue
        if sd is None:
            sd = t.dtype
        if t.dtype not in (torch.bfloat16, torch.float32) or t.dtype != sd:
            raise TypeError("states must both be bf16 or both fp32")
        _check(t, name, sd, (N, H, D, D), dev)
    state_dtype = KDA_DTYPE_NONE if sd is None else (KDA_DTYPE_BF16 if sd == torch.bfloat16 else KDA_DTYPE_FP32)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out), _ptr(A_log), _ptr(dt_bias),
            float(lower_bound), _ptr(initial_state), _ptr(final_state), state_dtype, _ptr(cu_seqlens), int(N),
            int(T), int(H))
    if workspace is not None:
        if workspace.dtype != torch.uint8 or workspace.device != dev or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
        wsz = workspace.numel()
    elif stage_events is not None:
        raise ValueError("stage_events needs a workspace")
    if (noalloc or recurrent) and (workspace is not None or stage_events is not None):
        raise ValueError("noalloc and recurrent take no workspace or stage events")
    if noalloc and recurrent:
        raise ValueError("noalloc and recurrent are exclusive")
    with torch.cuda.device(dev):
        if recurrent:
            rc = lib.kda_fwd_recurrent(*args, s.cuda_stream)
        elif noalloc:
            rc = lib.kda_fwd_noalloc(*args, s.cuda_stream)
        elif workspace is None:
            rc = lib.kda_fwd(*args, s.cuda_stream)
        elif stage_events is None:
            rc = lib.kda_fwd_ws(*args, _ptr(workspace), wsz, s.cuda_stream)
        else:
            ev = (ctypes.c_void_p * 3)(*[e.cuda_event if e is not None else None for e in stage_events])
            rc = lib.kda_fwd_ws_profiled(*args, _ptr(workspace), wsz, ev, s.cuda_stream)
    if rc != KDA_OK:
        raise KDAError(rc)


def kda_fwd_recurrent(*args, **kwargs) -> None:
    """kda_fwd evaluated token by token (the C entry point kda_fwd_recurrent): same arguments
    as kda_fwd without ``workspace``, ``stage_events`` and ``noalloc``."""
    kda_fwd(*args, recurrent=True, **kwargs)


def workspace_size(N: int, T: int, H: int, varlen: bool) -> int:
    """Bytes of workspace kda_fwd needs for N sequences, T tokens, H heads (kda_fwd_workspace_size)."""
    return int(_native.load().kda_fwd_workspace_size(int(N), int(T), int(H), int(bool(varlen))))


def device_status(stream: Optional[torch.cuda.Stream] = None) -> None:
    """Synchronise `stream` and raise KDAError if a kernel gave up a bounded device wait."""
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _native.load().kda_device_status(s.cuda_stream)
    if rc != KDA_OK:
        raise KDAError(rc)


class KDAHostRunner:
    """Runs kda_fwd on host (pinned) tensors: copies inputs in, computes, copies results out.

    Device buffers for one problem shape are allocated once at construction; ``run``
    then issues, on one stream, the host-to-device copies of the step's inputs, the
    forward kernel, and the device-to-host copies of ``out`` and ``final_state``.
    """

    def __init__(self, B: int, T: int, H: int, N: Optional[int] = None, state_dtype=None,
                 has_initial: bool = True, want_final: bool = True, device="cuda"):
        self.device = torch.device(device)
        self.N = B if N is None else N
        self.shape = (B, T, H, D)
        z = lambda shape, dt: torch.empty(shape, dtype=dt, device=self.device)
        self.q, self.k, self.v, self.g, self.out = (z(self.shape, torch.bfloat16) for _ in range(5))
        self.beta = z((B, T, H), torch.bfloat16)
        self.A_log = z((H,), torch.float32)
        self.dt_bias = z((H, D), torch.float32)
        self.cu = z((self.N + 1,), torch.int64) if N is not None else None
        self.state_dtype = state_dtype
        self.init = z((self.N, H, D, D), state_dtype) if (state_dtype is not None and has_initial) else None
        self.fin = z((self.N, H, D, D), state_dtype) if (state_dtype is not None and want_final) else None
        self.stream = torch.cuda.Stream(self.device)

    def h2d_bytes(self, has_cu: bool) -> int:
        ts = [self.q, self.k, self.v, self.g, self.beta, self.A_log, self.dt_bias]
        ts += [t for t in (self.init, self.cu if has_cu else None) if t is not None]
        return sum(t.numel() * t.element_size() for t in ts)

    def d2h_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.out, self.fin) if t is not None)

    def run(self, q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state=None,
            cu_seqlens=None, out_host=None, final_host=None):
        """Host tensors in, host tensors out (written into out_host / final_host when given)."""
        with torch.cuda.stream(self.stream):
            for dst, src in ((self.q, q), (self.k, k), (self.v, v), (self.g, g), (self.beta, beta),
                             (self.A_log, A_log), (self.dt_bias, dt_bias)):
                dst.copy_(src, non_blocking=True)
            if initial_state is not None:
                self.init.copy_(initial_state, non_blocking=True)
            if cu_seqlens is not None:
                self.cu.copy_(cu_seqlens, non_blocking=True)
            kda_fwd(self.q, self.k, self.v, self.g, self.beta, scale, self.out, self.A_log, self.dt_bias,
                    lower_bound, initial_state=self.init if initial_state is not None else None,
                    final_state=self.fin, cu_seqlens=self.cu if cu_seqlens is not None else None,
                    stream=self.stream)
            if out_host is None:
                out_host = torch.empty(self.shape, dtype=torch.bfloat16, pin_memory=True)
            out_host.copy_(self.out, non_blocking=True)
            if self.fin is not None:
                if final_host is None:
                    final_host = torch.empty(self.fin.shape, dtype=self.fin.dtype, pin_memory=True)
                final_host.copy_(self.fin, non_blocking=True)
        return out_host, final_host
