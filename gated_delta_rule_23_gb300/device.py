"""Device copies of a seeded problem (torch marshalling only).

Turns the numpy arrays of an ``inputs.KDAProblem`` into contiguous CUDA tensors in the
dtypes the C ABI expects (bf16 bit patterns reinterpreted as torch.bfloat16, fp32
parameters, int64 cu_seqlens).  Used by the benchmark and the GPU tests; no arithmetic.
"""
from __future__ import annotations

import numpy as np
import torch

from .inputs import STATE_BF16, STATE_FP32


def bf16_tensor(bits, device="cuda"):
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on `device` (same bits)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_device(p, device="cuda"):
    """Dict of device tensors for problem p: q, k, v, g, beta, A_log, dt_bias, cu (or None),
    init (or None) and sdt, the torch dtype of the states (or None)."""
    d = dict(q=bf16_tensor(p.q, device), k=bf16_tensor(p.k, device), v=bf16_tensor(p.v, device),
             g=bf16_tensor(p.g, device), beta=bf16_tensor(p.beta, device),
             A_log=torch.from_numpy(p.A_log).to(device), dt_bias=torch.from_numpy(p.dt_bias).to(device))
    d["cu"] = None if p.cu_seqlens is None else torch.from_numpy(p.cu_seqlens).to(device)
    sdt = {STATE_BF16: torch.bfloat16, STATE_FP32: torch.float32}.get(p.state_dtype)
    d["sdt"] = sdt
    if p.initial_state is not None:
        d["init"] = (bf16_tensor(p.initial_state, device) if p.state_dtype == STATE_BF16
                     else torch.from_numpy(p.initial_state).to(device))
    else:
        d["init"] = None
    return d
