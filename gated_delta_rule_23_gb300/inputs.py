"""Seeded synthetic inputs for the KDA forward pass.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from
it without sharing any computation.

Shapes follow the kernel API table of the FlashKDA README mirror (ai-feeds.com,
"FlashKDA", section "内核 API"): q, k, v, g are bf16 [B, T, H, 128], beta is bf16
[B, T, H], A_log fp32 [H], dt_bias fp32 [H, 128], states [N, H, V=128, K=128].
With cu_seqlens, B = 1 and T is the total length of all N sequences.

The value distributions are the ones the five workloads use: q, k, v, g and the
beta logits ~ N(0, 1) rounded to bf16; A_log ~ U(0, ln 16); dt_bias ~ N(0, 0.1);
initial states ~ N(0, 0.1) (0.1 is read as the standard deviation);
lower_bound = -5; scale = 1/sqrt(128).  Arrays are numpy; bf16 tensors are held
as their uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

D = 128  # K = V = 128 is the only head dimension the API accepts

STATE_NONE, STATE_BF16, STATE_FP32 = "none", "bf16", "fp32"


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = np.empty(u.shape, np.uint32)          # in-place uint32 ops: no temporaries, no int64 promotion
    np.right_shift(u, 16, out=r)
    np.bitwise_and(r, np.uint32(1), out=r)
    np.add(r, np.uint32(0x7FFF), out=r)
    np.add(r, u, out=r)
    np.right_shift(r, 16, out=r)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class KDAProblem:
    """One forward-pass problem: inputs, parameters and the state/varlen options."""

    name: str
    q: np.ndarray            # uint16 bf16 bits [B, T, H, 128]
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray         # uint16 bf16 bits [B, T, H]
    A_log: np.ndarray        # float32 [H]
    dt_bias: np.ndarray      # float32 [H, 128]
    lower_bound: float
    scale: float
    state_dtype: str         # "none" | "bf16" | "fp32"
    initial_state: Optional[np.ndarray]  # [N, H, 128, 128]: float32, or uint16 bf16 bits; None = zeros
    want_final: bool
    cu_seqlens: Optional[np.ndarray]     # int64 [N + 1] or None

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def T(self) -> int:
        return self.q.shape[1]

    @property
    def H(self) -> int:
        return self.q.shape[2]

    @property
    def N(self) -> int:
        return self.B if self.cu_seqlens is None else len(self.cu_seqlens) - 1

    def seq_lengths(self) -> np.ndarray:
        if self.cu_seqlens is None:
            return np.full(self.B, self.T, dtype=np.int64)
        return np.diff(self.cu_seqlens)

    def initial_state_f64(self) -> Optional[np.ndarray]:
        if self.initial_state is None:
            return None
        if self.state_dtype == STATE_BF16:
            return bf16_to_f32(self.initial_state).astype(np.float64)
        return self.initial_state.astype(np.float64)

    def token_heads(self) -> int:
        return int(self.seq_lengths().sum()) * self.H


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x)


def irregular_lengths(rng: np.random.Generator, n: int, total: int, lo: int = 16, hi: int = 2048) -> np.ndarray:
    """n lengths drawn log-uniform on [lo, hi], rescaled to sum to `total`, each >= 1.

    The rounding residual goes to the longest sequence.  If every length comes out a
    multiple of 16, one token moves from the longest to the shortest, so that at least
    one sequence ends in a partial 16-token block.
    """
    raw = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    lens = np.maximum(1, np.rint(raw * (total / raw.sum())).astype(np.int64))
    lens[np.argmax(lens)] += total - int(lens.sum())
    if np.all(lens % 16 == 0):
        lens[np.argmax(lens)] -= 1
        lens[np.argmin(lens)] += 1
    assert int(lens.sum()) == total and lens.min() >= 1
    return lens


def make_problem(*, B: int, T: int, H: int, seed: int, state_dtype: str = STATE_FP32,
                 with_initial: bool = True, want_final: bool = True,
                 cu_seqlens: Optional[np.ndarray] = None, lower_bound: float = -5.0,
                 scale: Optional[float] = None, name: str = "custom") -> KDAProblem:
    """Draw one problem with the standard value distributions (see module docstring)."""
    rng = np.random.default_rng(seed)
    shape = (B, T, H, D)
    q = _normal_bf16(rng, shape)
    k = _normal_bf16(rng, shape)
    v = _normal_bf16(rng, shape)
    g = _normal_bf16(rng, shape)
    beta = _normal_bf16(rng, (B, T, H))
    A_log = rng.uniform(0.0, math.log(16.0), size=H).astype(np.float32)
    dt_bias = (rng.standard_normal(size=(H, D), dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    if cu_seqlens is not None:
        assert B == 1 and int(cu_seqlens[-1]) == T
        cu_seqlens = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = B if cu_seqlens is None else len(cu_seqlens) - 1
    init = None
    if state_dtype != STATE_NONE and with_initial:
        s = rng.standard_normal(size=(N, H, D, D), dtype=np.float32) * np.float32(0.1)
        init = bf16_bits(s) if state_dtype == STATE_BF16 else s.astype(np.float32)
    if state_dtype == STATE_NONE:
        want_final = False
    return KDAProblem(name=name, q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
                      lower_bound=float(lower_bound),
                      scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
                      state_dtype=state_dtype, initial_state=init, want_final=want_final,
                      cu_seqlens=cu_seqlens)


# The five standard workloads.  Index 0 is the small case the oracle finishes in
# well under a second; 1-4 are the T = 8192 prefill shapes of the benchmark tables.
WORKLOADS = {
    0: "tiny: B=1 T=64 H=2, fp32 initial and final state",
    1: "fixed-length prefill: B=1 T=8192 H=64, no initial state, fp32 final state",
    2: "fixed-length prefill: B=1 T=8192 H=96, bf16 initial and final state",
    3: "uniform varlen: 8 x 1024 tokens, H=96, fp32 states",
    4: "irregular varlen: 12 log-uniform lengths summing to 8192, H=96, fp32 states",
}


def make_workload(idx: int) -> KDAProblem:
    """Build standard workload `idx` (0-4); the seed is the workload index."""
    seed = idx
    if idx == 0:
        return make_problem(B=1, T=64, H=2, seed=seed, state_dtype=STATE_FP32, name=WORKLOADS[0])
    if idx == 1:
        return make_problem(B=1, T=8192, H=64, seed=seed, state_dtype=STATE_FP32, with_initial=False,
                            name=WORKLOADS[1])
    if idx == 2:
        return make_problem(B=1, T=8192, H=96, seed=seed, state_dtype=STATE_BF16, name=WORKLOADS[2])
    if idx == 3:
        cu = np.arange(0, 8193, 1024, dtype=np.int64)
        return make_problem(B=1, T=8192, H=96, seed=seed, state_dtype=STATE_FP32, cu_seqlens=cu,
                            name=WORKLOADS[3])
    if idx == 4:
        lens = irregular_lengths(np.random.default_rng(1000 + seed), 12, 8192)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        return make_problem(B=1, T=8192, H=96, seed=seed, state_dtype=STATE_FP32, cu_seqlens=cu,
                            name=WORKLOADS[4])
    raise ValueError(f"unknown workload {idx}")


def subset_heads(p: KDAProblem, heads) -> KDAProblem:
    """The same problem restricted to a subset of heads (heads are independent)."""
    heads = np.asarray(heads, dtype=np.int64)
    init = None if p.initial_state is None else np.ascontiguousarray(p.initial_state[:, heads])
    return dataclasses.replace(
        p, q=np.ascontiguousarray(p.q[:, :, heads]), k=np.ascontiguousarray(p.k[:, :, heads]),
        v=np.ascontiguousarray(p.v[:, :, heads]), g=np.ascontiguousarray(p.g[:, :, heads]),
        beta=np.ascontiguousarray(p.beta[:, :, heads]), A_log=np.ascontiguousarray(p.A_log[heads]),
        dt_bias=np.ascontiguousarray(p.dt_bias[heads]), initial_state=init)
