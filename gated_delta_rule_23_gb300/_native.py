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
SOURCES = [os.path.join(CSRC, "kda_fwd.cu")]
HEADERS = [os.path.join(INCLUDE, "kda.h")]
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
    """Compile csrc/*.cu into _build/libkda.so (sm_103a, -O3, -lineinfo)."""
    with _lock:
        if not force and not _stale():
            return LIB_PATH
        os.makedirs(BUILD_DIR, exist_ok=True)
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
               "-I" + INCLUDE, "-o", tmp, *SOURCES]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
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
        lib.kda_check_cu_seqlens.argtypes = [P, I, I64]
        lib.kda_check_cu_seqlens.restype = I
        lib.kda_status_string.argtypes = [I]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_device_status.argtypes = [P]
        lib.kda_device_status.restype = I
        lib.kda_fwd_smem_bytes.argtypes = []
        lib.kda_fwd_smem_bytes.restype = ctypes.c_size_t
        _lib = lib
    return _lib


def declared_functions() -> List[str]:
    """Names of the functions include/kda.h declares (for export checks)."""
    import re
    text = open(HEADERS[0]).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kda_[a-z_0-9]+)\s*\(", text, re.M)))


# status codes, as in include/kda.h
KDA_OK, KDA_ERR_INVALID_ARGUMENT, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(5)
KDA_DTYPE_NONE, KDA_DTYPE_BF16, KDA_DTYPE_FP32 = range(3)


class KDAError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(f"kda: {load().kda_status_string(status).decode()} (status {status})")
