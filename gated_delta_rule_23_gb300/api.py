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
            recurrent: bool = False, variant: int = 0) -> None:
    """KDA chunked forward on CUDA tensors; writes ``out`` and ``final_state`` in place.

    q, k, v, g: bf16 [B, T, H, 128]; beta: bf16 [B, T, H]; out: bf16 [B, T, H, 128];
    A_log: fp32 [H]; dt_bias: fp32 [H, 128]; states: bf16 or fp32 [N, H, 128, 128] (same dtype
    when both are given); cu_seqlens: int64 [N + 1] with B = 1.  Runs asynchronously on
    ``stream`` (default: the current stream).  ``workspace``: optional uint8 CUDA tensor of at
    least ``workspace_size(...)`` bytes (kda_fwd_ws); without it the library's pool provides one.
    ``stage_events``: optional three recorded-once torch.cuda.Event objects (or None) marking the
    start of the prep kernel, the prep/recurrence boundary and the end (kda_fwd_ws_profiled, which
    always runs the single-launch schedule, never pieces; needs ``workspace``).  ``noalloc``: use the library's static workspace (kda_fwd_noalloc).
    ``recurrent``: evaluate token by token (kda_fwd_recurrent; decode and short sequences, no
    workspace).  ``variant``: KDA_VARIANT_* bits of the measurement variants (kda_fwd_ws_variant; needs
    ``workspace``).
    """
    lib = _native.load()
    if q.dim() != 4 or q.shape[-1] != D:
        raise ValueError("q must be [B, T, H, 128]")
    B, T, H, _ = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_fwd needs CUDA tensors (kda_fwd_host takes host tensors)")
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
    if variant and (workspace is None or stage_events is not None or noalloc or recurrent):
        raise ValueError("variant needs a workspace and excludes stage_events, noalloc and recurrent")
    with torch.cuda.device(dev):
        if recurrent:
            rc = lib.kda_fwd_recurrent(*args, s.cuda_stream)
        elif noalloc:
            rc = lib.kda_fwd_noalloc(*args, s.cuda_stream)
        elif workspace is None:
            rc = lib.kda_fwd(*args, s.cuda_stream)
        elif variant:
            rc = lib.kda_fwd_ws_variant(*args, _ptr(workspace), wsz, int(variant), s.cuda_stream)
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
    """Synchronise `stream` and raise KDAError with what the kernels reported since the last call
    (kda_device_status: a bounded wait that gave up, a malformed device cu_seqlens, a non-finite state)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _native.load().kda_device_status(s.cuda_stream)
    if rc != KDA_OK:
        raise KDAError(rc)


def kda_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                 scale: float, out: torch.Tensor, A_log: torch.Tensor, dt_bias: torch.Tensor, lower_bound: float,
                 initial_state: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
                 cu_seqlens: Optional[torch.Tensor] = None, device: Optional[int] = None) -> None:
    """kda_fwd on host (CPU) tensors (the C entry point kda_fwd_host): the library copies the inputs
    to the CUDA device, runs the forward pass and copies ``out`` and ``final_state`` back, with the
    copies pipelined against the kernels.  Returns when the results are in host memory.  Same shapes
    and dtypes as kda_fwd; pinned tensors let the copies overlap the kernels."""
    lib = _native.load()
    if q.dim() != 4 or q.shape[-1] != D:
        raise ValueError("q must be [B, T, H, 128]")
    B, T, H, _ = q.shape
    cpu = torch.device("cpu")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("out", out)):
        _check(t, name, torch.bfloat16, (B, T, H, D), cpu)
    _check(beta, "beta", torch.bfloat16, (B, T, H), cpu)
    _check(A_log, "A_log", torch.float32, (H,), cpu)
    _check(dt_bias, "dt_bias", torch.float32, (H, D), cpu)
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
            raise ValueError("cu_seqlens must be int64 [N + 1]")
        N = cu_seqlens.numel() - 1
        _check(cu_seqlens, "cu_seqlens", torch.int64, (N + 1,), cpu)
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
        _check(t, name, sd, (N, H, D, D), cpu)
    state_dtype = KDA_DTYPE_NONE if sd is None else (KDA_DTYPE_BF16 if sd == torch.bfloat16 else KDA_DTYPE_FP32)
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    with torch.cuda.device(dev):
        rc = lib.kda_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out), _ptr(A_log),
                              _ptr(dt_bias), float(lower_bound), _ptr(initial_state), _ptr(final_state), state_dtype,
                              _ptr(cu_seqlens), int(N), int(T), int(H))
    if rc != KDA_OK:
        raise KDAError(rc)
