"""GB300-native (sm_103a) Kimi Delta Attention forward pass.

The computation lives in libkda.so (CUDA sources in csrc/, C ABI in include/kda.h);
this package builds and loads it and marshals arguments.  There is no CPU path.
"""
from ._native import KDAError, build, load  # noqa: F401
from .api import device_status, kda_fwd, kda_fwd_host, kda_fwd_recurrent, workspace_size  # noqa: F401

__all__ = ["kda_fwd", "kda_fwd_recurrent", "workspace_size", "device_status", "kda_fwd_host", "KDAError", "build", "load"]
