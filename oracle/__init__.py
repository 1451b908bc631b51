"""CPU oracle for the KDA forward pass -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The CUDA library and its Python binding never touch
it.  ``kda_oracle.c`` holds the arithmetic (fp64, token by token); this module
compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None
_override: Optional[str] = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libkda_oracle.so (gcc, portable flags)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                        "-lm", "-lpthread"], check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def use_library(path: Optional[str]) -> None:
    """Point the binding at another build of kda_oracle.c (None: the default build).

    Used by the tests that plant mistakes in a copy of the oracle's source to show that
    the pins catch them; nothing else calls it.
    """
    global _lib, _override
    _override = path
    _lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_override or build())
        P = ctypes.c_void_p
        lib.kda_oracle_fwd.argtypes = [P, P, P, P, P, ctypes.c_double, P, P, P, ctypes.c_double,
                                       P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                       ctypes.c_int]
        lib.kda_oracle_fwd.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)


def kda_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, g: np.ndarray, beta: np.ndarray,
            scale: float, A_log: np.ndarray, dt_bias: np.ndarray, lower_bound: float,
            initial_state: Optional[np.ndarray] = None, want_final: bool = True,
            cu_seqlens: Optional[np.ndarray] = None,
            nthreads: Optional[int] = None) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """fp64 reference forward.

    q, k, v, g: uint16 bf16 bit patterns [B, T, H, 128]; beta: uint16 [B, T, H];
    A_log float32 [H]; dt_bias float32 [H, 128]; initial_state float64 [N, H, 128, 128] or None.
    Returns (out float64 [B, T, H, 128], final_state float64 [N, H, 128, 128] or None).
    """
    lib = _load()
    B, T, H, Dk = q.shape
    assert Dk == 128 and k.shape == q.shape and v.shape == q.shape and g.shape == q.shape
    assert beta.shape == (B, T, H)
    arr16 = lambda a: np.ascontiguousarray(a, dtype=np.uint16)
    q, k, v, g, beta = (arr16(a) for a in (q, k, v, g, beta))
    A_log = np.ascontiguousarray(A_log, dtype=np.float32)
    dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32)
    if cu_seqlens is not None:
        assert B == 1
        cu_seqlens = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
        N, Tp = len(cu_seqlens) - 1, T
    else:
        N, Tp = B, T
    init = None if initial_state is None else np.ascontiguousarray(initial_state, dtype=np.float64)
    if init is not None:
        assert init.shape == (N, H, 128, 128)
    out = np.zeros((B, T, H, 128), dtype=np.float64)
    final = np.zeros((N, H, 128, 128), dtype=np.float64) if want_final else None
    rc = lib.kda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out),
                            _ptr(A_log), _ptr(dt_bias), float(lower_bound), _ptr(init), _ptr(final),
                            _ptr(cu_seqlens), int(N), int(Tp), int(H),
                            int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"kda_oracle_fwd rejected its arguments (rc={rc})")
    return out, final


def kda_fwd_problem(p, nthreads: Optional[int] = None):
    """Run the oracle on a `gated_delta_rule_23_gb300.inputs.KDAProblem`."""
    return kda_fwd(p.q, p.k, p.v, p.g, p.beta, p.scale, p.A_log, p.dt_bias, p.lower_bound,
                   initial_state=p.initial_state_f64(), want_final=p.want_final,
                   cu_seqlens=p.cu_seqlens, nthreads=nthreads)
