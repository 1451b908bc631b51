"""CPU checks of the C ABI: the library builds and loads, exports what include/kda.h
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes

import numpy as np
import pytest

from gated_delta_rule_23_gb300 import _native
from gated_delta_rule_23_gb300._native import (KDA_DTYPE_BF16, KDA_DTYPE_FP32, KDA_DTYPE_NONE, KDA_ERR_INVALID_ARGUMENT,
                                               KDA_ERR_UNSUPPORTED, KDA_OK)


@pytest.fixture(scope="module")
def lib():
    return _native.load()


def test_exports_every_declared_function(lib):
    names = _native.declared_functions()
    assert {"kda_fwd", "kda_fwd_ws", "kda_fwd_workspace_size", "kda_workspace_trim", "kda_check_cu_seqlens",
            "kda_status_string", "kda_fwd_smem_bytes", "kda_device_status", "kda_fwd_recurrent",
            "kda_fwd_host"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_smem_fits_one_cta_per_sm(lib):
    assert 0 < lib.kda_fwd_smem_bytes() <= 232448


def test_status_strings(lib):
    for s in range(6):
        assert lib.kda_status_string(s) and lib.kda_status_string(s) != b"unknown status"
    assert lib.kda_status_string(99) == b"unknown status"


# fake, 256-byte aligned "device" addresses: kda_fwd must reject the call before touching them
A = 1 << 20


def call(lib, entry="kda_fwd", **kw):
    args = dict(q=A, k=A + 0x1000, v=A + 0x2000, g=A + 0x3000, beta=A + 0x4000, scale=0.1, out=A + 0x5000,
                A_log=A + 0x6000, dt_bias=A + 0x7000, lower_bound=-5.0, init=None, fin=None,
                state_dtype=KDA_DTYPE_NONE, cu=None, N=1, T=64, H=2, stream=None)
    args.update(kw)
    return getattr(lib, entry)(args["q"], args["k"], args["v"], args["g"], args["beta"], args["scale"], args["out"],
                       args["A_log"], args["dt_bias"], args["lower_bound"], args["init"], args["fin"],
                       args["state_dtype"], args["cu"], args["N"], args["T"], args["H"], args["stream"])


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(k=None), dict(v=None), dict(g=None), dict(beta=None), dict(out=None),
    dict(A_log=None), dict(dt_bias=None),
    dict(N=0), dict(H=0), dict(T=-1), dict(N=1 << 20, H=1 << 12),
    dict(q=A + 8), dict(out=A + 0x5002), dict(beta=A + 0x4001), dict(cu=A + 0x9004),
    dict(init=A + 0x8000, state_dtype=KDA_DTYPE_NONE), dict(fin=A + 0x8000, state_dtype=7),
    dict(init=A + 0x8008, state_dtype=KDA_DTYPE_FP32), dict(dt_bias=A + 0x7004),
])
@pytest.mark.parametrize("entry", ["kda_fwd", "kda_fwd_recurrent"])
def test_invalid_arguments_rejected(lib, kw, entry):
    assert call(lib, entry, **kw) == KDA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("lb", [-5.01, 0.5, float("nan"), float("-inf")])
@pytest.mark.parametrize("entry", ["kda_fwd", "kda_fwd_recurrent"])
def test_lower_bound_outside_range_unsupported(lib, lb, entry):
    assert call(lib, entry, lower_bound=lb) == KDA_ERR_UNSUPPORTED


@pytest.mark.parametrize("entry", ["kda_fwd", "kda_fwd_recurrent"])
def test_nonfinite_scale_unsupported(lib, entry):
    assert call(lib, entry, scale=float("inf")) == KDA_ERR_UNSUPPORTED


def test_recurrent_entry_limits_tokens(lib):
    """The token-recurrent entry point takes fewer than 2^31 tokens and 2^30 (sequence, head) pairs."""
    assert call(lib, "kda_fwd_recurrent", T=1 << 31) == KDA_ERR_UNSUPPORTED
    assert call(lib, "kda_fwd_recurrent", N=1 << 15, H=1 << 15) == KDA_ERR_UNSUPPORTED


def test_check_cu_seqlens(lib):
    def chk(cu, N, T):
        a = np.ascontiguousarray(cu, dtype=np.int64)
        return lib.kda_check_cu_seqlens(a.ctypes.data_as(ctypes.c_void_p), N, T)
    assert chk([0, 3, 3, 10], 3, 10) == KDA_OK
    assert chk([0, 0], 1, 0) == KDA_OK
    assert chk([1, 3, 10], 2, 10) == KDA_ERR_INVALID_ARGUMENT
    assert chk([0, 5, 3, 10], 3, 10) == KDA_ERR_INVALID_ARGUMENT
    assert chk([0, 3, 9], 2, 10) == KDA_ERR_INVALID_ARGUMENT
    assert lib.kda_check_cu_seqlens(None, 1, 0) == KDA_ERR_INVALID_ARGUMENT


def test_binding_rejects_cpu_tensors():
    import torch
    from gated_delta_rule_23_gb300 import kda_fwd
    x = torch.zeros(1, 4, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kda_fwd(x, x, x, x, torch.zeros(1, 4, 1, dtype=torch.bfloat16), 1.0, x.clone(),
                torch.zeros(1), torch.zeros(1, 128), -5.0)


def test_workspace_size(lib):
    slot = 74240   # fp16 operands of one (64-token chunk, head)
    state = 128 * 128 * 4   # fp32 state of one (sequence, head)
    # fixed length with N x H <= 64 and at least 32 chunks: may run in pieces, the fp32 state between
    # pieces ahead of the slots
    assert lib.kda_fwd_workspace_size(1, 8192, 96, 0) == 128 * 96 * slot
    assert lib.kda_fwd_workspace_size(1, 8192, 64, 0) == 64 * state + 128 * 64 * slot
    assert lib.kda_fwd_workspace_size(2, 4096, 32, 0) == 64 * state + 2 * 64 * 32 * slot
    assert lib.kda_fwd_workspace_size(1, 2049, 40, 0) == 40 * state + 33 * 40 * slot
    assert lib.kda_fwd_workspace_size(1, 1985, 40, 0) == 40 * state + 32 * 40 * slot
    assert lib.kda_fwd_workspace_size(1, 1984, 40, 0) == 31 * 40 * slot
    assert lib.kda_fwd_workspace_size(1, 8192, 65, 0) == 128 * 65 * slot
    assert lib.kda_fwd_workspace_size(2, 65, 3, 0) == 2 * 2 * 3 * slot
    assert lib.kda_fwd_workspace_size(1, 0, 4, 0) == 0
    # varlen: a header (chunk offsets, order, 16 bytes per chunk of chunk info), then at most
    # (T + 63 N) / 64 chunks
    mc = (8192 + 63 * 8) // 64
    hdr = -(-(-(-(9 * 8 + 8 * 4) // 16) * 16 + mc * 16) // 256) * 256
    assert lib.kda_fwd_workspace_size(8, 8192, 96, 1) == hdr + mc * 96 * slot
    assert lib.kda_fwd_workspace_size(0, 10, 1, 0) == 0
    # fixed-length problems of 1-16 tokens per sequence take the token-recurrent kernels: no workspace
    assert lib.kda_fwd_workspace_size(256, 1, 96, 0) == 0
    assert lib.kda_fwd_workspace_size(256, 4, 96, 0) == 0
    assert lib.kda_fwd_workspace_size(256, 16, 96, 0) == 0
    assert lib.kda_fwd_workspace_size(256, 17, 96, 0) == 256 * 96 * slot
    assert lib.kda_fwd_workspace_size(1, 5, 96, 1) > 0   # varlen: always the chunked form


def test_scan_groups_and_workspace(lib):
    slot, state = 74240, 128 * 128 * 4
    # the scan along T: at most 16 (sequence, head) pairs, at least 32 chunks, when the cost model prefers it;
    # the count depends on N, T, H only
    assert lib.kda_fwd_scan_groups(2, 8200, 8, 0) == 9      # 129 chunks: 9 groups of 15 (the last 9)
    assert lib.kda_fwd_scan_groups(1, 2049, 3, 0) == 7      # 33 chunks: 7 groups of 5 (the last 3)
    assert lib.kda_fwd_scan_groups(1, 32768, 8, 0) == 19    # 512 chunks: 19 groups of 27 (the last 26)
    assert lib.kda_fwd_scan_groups(1, 32768, 1, 0) == 27    # 512 chunks: 27 groups of 19 (the last 18)
    assert lib.kda_fwd_scan_groups(1, 8192, 17, 0) == 1     # more than 16 pairs
    assert lib.kda_fwd_scan_groups(1, 1984, 1, 0) == 1      # fewer than 32 chunks
    assert lib.kda_fwd_scan_groups(8, 8192, 1, 1) == 1      # varlen
    assert lib.kda_fwd_scan_groups(0, 100, 1, 0) == 0
    # scan problems run without pieces; their header: initial state, then M, B and start states of G - 1 groups
    assert lib.kda_fwd_pieces(2, 8200, 8, 0) == 1
    assert lib.kda_fwd_workspace_size(2, 8200, 8, 0) == (1 + 3 * 8) * 16 * state + 2 * 129 * 8 * slot
    assert lib.kda_fwd_workspace_size(1, 2049, 3, 0) == (1 + 3 * 6) * 3 * state + 33 * 3 * slot


def test_pieces_query_without_pieces(lib):
    # problems outside the piece rule report 1 without touching the device; invalid sizes 0
    assert lib.kda_fwd_pieces(1, 8192, 96, 0) == 1      # more than 64 (sequence, head) pairs
    assert lib.kda_fwd_pieces(1, 1984, 8, 0) == 1       # fewer than 32 chunks
    assert lib.kda_fwd_pieces(8, 8192, 8, 1) == 1       # varlen
    assert lib.kda_fwd_pieces(256, 1, 96, 0) == 1       # decode step
    assert lib.kda_fwd_pieces(0, 100, 8, 0) == 0
    assert lib.kda_fwd_pieces(1, -1, 8, 0) == 0
    assert lib.kda_fwd_pieces(1, 100, 0, 0) == 0


def test_ws_entry_rejects_missing_workspace(lib):
    args = [A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 0.1, A + 0x5000, A + 0x6000, A + 0x7000, -5.0,
            None, None, KDA_DTYPE_NONE, None, 1, 64, 2]
    need = lib.kda_fwd_workspace_size(1, 64, 2, 0)
    assert lib.kda_fwd_ws(*args, None, need, None) == KDA_ERR_INVALID_ARGUMENT
    assert lib.kda_fwd_ws(*args, A + 0x100000, need - 16, None) == KDA_ERR_INVALID_ARGUMENT
    assert lib.kda_fwd_ws(*args, A + 0x100010, need, None) == KDA_ERR_INVALID_ARGUMENT   # not 256-byte aligned


def test_host_entry_rejects_bad_arguments_before_any_cuda_call(lib):
    """kda_fwd_host checks its (host) arguments like kda_fwd, and cu_seqlens on the host."""
    args = [A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 0.1, A + 0x5000, A + 0x6000, A + 0x7000, -5.0,
            None, None, KDA_DTYPE_NONE, None, 1, 64, 2]
    bad = list(args)
    bad[0] = None
    assert lib.kda_fwd_host(*bad) == KDA_ERR_INVALID_ARGUMENT
    bad = list(args)
    bad[9] = 1.0
    assert lib.kda_fwd_host(*bad) == KDA_ERR_UNSUPPORTED
    cu = (ctypes.c_int64 * 3)(0, 40, 70)          # ends at 70, not T = 64
    bad = list(args)
    bad[13], bad[14] = ctypes.cast(cu, ctypes.c_void_p).value, 2
    assert lib.kda_fwd_host(*bad) == KDA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("N,T,H", [(1 << 20, 1 << 40, 1 << 10),   # workspace bytes do not fit in 64 bits
                                   (1, 1 << 40, 1)])              # more than 2^31 - 1 (chunk, head) items
def test_oversize_problems_unsupported_before_any_cuda_call(lib, N, T, H):
    """Sizes that pass the argument checks but whose workspace size or item count the chunked path cannot
    represent are refused with KDA_ERR_UNSUPPORTED on the host (the pointers are fake)."""
    assert lib.kda_fwd_workspace_size(N, T, H, 0) == 0
    assert call(lib, "kda_fwd", N=N, T=T, H=H) == KDA_ERR_UNSUPPORTED
    assert call(lib, "kda_fwd_noalloc", N=N, T=T, H=H) == KDA_ERR_UNSUPPORTED
    args = [A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 0.1, A + 0x5000, A + 0x6000, A + 0x7000, -5.0,
            None, None, KDA_DTYPE_NONE, None, N, T, H]
    assert lib.kda_fwd_ws(*args, A + 0x100000, 1 << 30, None) == KDA_ERR_UNSUPPORTED
    assert lib.kda_fwd_host(*args) == KDA_ERR_UNSUPPORTED


def test_variant_entry_rejects_unknown_bits(lib):
    args = [A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 0.1, A + 0x5000, A + 0x6000, A + 0x7000, -5.0,
            None, None, KDA_DTYPE_NONE, None, 1, 64, 2]
    need = lib.kda_fwd_workspace_size(1, 64, 2, 0)
    assert lib.kda_fwd_ws_variant(*args, A + 0x100000, need, 4, None) == KDA_ERR_INVALID_ARGUMENT
    assert lib.kda_fwd_ws_variant(*args, None, need, 1, None) == KDA_ERR_INVALID_ARGUMENT
