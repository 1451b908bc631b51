"""Build and load the CUDA library (libkda.so) and expose its C ABI through ctypes.

The library is compiled in-tree with nvcc for sm_103a only.  Loading fails loudly
when the library is missing or cannot be built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(_PKG)
CSRC = os.path.join(_PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(_PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libkda.so")
UNITS = ["kda_api", "kda_prep", "kda_recur", "kda_recurrent", "kda_decode", "kda_host", "kda_noalloc", "kda_scan"]
SOURCES = [os.path.join(CSRC, u + ".cu") for u in UNITS]
HEADERS = [os.path.join(INCLUDE, "kda.h"), os.path.join(CSRC, "kda_device.cuh"), os.path.join(CSRC, "kda_internal.h"),
           os.path.join(CSRC, "kda_plan.h")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > t for s in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu (sm_103a, -O3, -lineinfo), one process per unit, and link _build/libkda.so."""
    with _lock:
        if not force and not _stale():
            return LIB_PATH
        os.makedirs(BUILD_DIR, exist_ok=True)
        tag = f".tmp{os.getpid()}"
        common = [nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE]
        if verbose:
            common.append("-Xptxas=-v")
        objs, procs = [], []
        for u, src in zip(UNITS, SOURCES):
            obj = os.path.join(BUILD_DIR, u + tag + ".o")
            objs.append(obj)
            procs.append(subprocess.Popen(common + ["-c", "-o", obj, src]))
        codes = [pr.wait() for pr in procs]
        try:
            for src, rc in zip(SOURCES, codes):
                if rc != 0:
                    raise subprocess.CalledProcessError(rc, f"nvcc {src}")
            tmp = LIB_PATH + tag
            subprocess.run([nvcc(), *ARCH_FLAGS, "-shared", "-o", tmp, *objs], check=True)
            os.replace(tmp, LIB_PATH)
        finally:
            for o in objs:
                if os.path.exists(o):
                    os.remove(o)
        return LIB_PATH


def load() -> ctypes.CDLL:
    """Load libkda.so (building it first if it is missing or older than its sources)."""
    global _lib
    if _lib is None:
        path = build()
        lib = ctypes.CDLL(path)
        P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.kda_fwd.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, I, P, I, I64, I, P]
        lib.kda_fwd.restype = I
        lib.kda_fwd_noalloc.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, I, P, I, I64, I, P]
        lib.kda_fwd_noalloc.restype = I
        lib.kda_fwd_recurrent.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, I, P, I, I64, I, P]
        lib.kda_fwd_recurrent.restype = I
        lib.kda_fwd_host.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, I, P, I, I64, I]
        lib.kda_fwd_host.restype = I
        lib.kda_fwd_host_plan.argtypes = [I, I64, P, P, P, P, P, I]
        lib.kda_fwd_host_plan.restype = I
        lib.kda_fwd_ws.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, I, P, I, I64, I, P, ctypes.c_size_t, P]
        lib.kda_fwd_ws.restype = I
        lib.kda_fwd_ws_profiled.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, I, P, I, I64, I, P, ctypes.c_size_t,
                                             P, P]
        lib.kda_fwd_ws_profiled.restype = I
        lib.kda_fwd_ws_variant.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, I, P, I, I64, I, P, ctypes.c_size_t,
                                           ctypes.c_uint, P]
        lib.kda_fwd_ws_variant.restype = I
        lib.kda_fwd_workspace_size.argtypes = [I, I64, I, I]
        lib.kda_fwd_workspace_size.restype = ctypes.c_size_t
        lib.kda_fwd_pieces.argtypes = [I, I64, I, I]
        lib.kda_fwd_pieces.restype = I
        lib.kda_fwd_scan_groups.argtypes = [I, I64, I, I]
        lib.kda_fwd_scan_groups.restype = I
        lib.kda_workspace_trim.argtypes = []
        lib.kda_workspace_trim.restype = I
        lib.kda_check_cu_seqlens.argtypes = [P, I, I64]
        lib.kda_check_cu_seqlens.restype = I
        lib.kda_status_string.argtypes = [I]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_device_status.argtypes = [P]
        lib.kda_device_status.restype = I
        lib.kda_set_wait_limit.argtypes = [ctypes.c_uint32]
        lib.kda_set_wait_limit.restype = None
        lib.kda_fwd_smem_bytes.argtypes = []
        lib.kda_fwd_smem_bytes.restype = ctypes.c_size_t
        _lib = lib
    return _lib


def declared_functions() -> List[str]:
    """Names of the functions include/kda.h declares (for export checks)."""
    import re
    text = open(HEADERS[0]).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kda_[a-z_0-9]+)\s*\(", text, re.M)))


KDA_DEFAULT_WAIT_POLLS = 16777216
KDA_VARIANT_BF16_STATE, KDA_VARIANT_NEUMANN_INVERSE = 1, 2
# status codes, as in include/kda.h
KDA_OK, KDA_ERR_INVALID_ARGUMENT, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_NONFINITE = range(6)
KDA_DTYPE_NONE, KDA_DTYPE_BF16, KDA_DTYPE_FP32 = range(3)


class KDAError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(f"kda: {load().kda_status_string(status).decode()} (status {status})")
