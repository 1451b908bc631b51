"""kda_fwd_noalloc: the forward pass for callers that cannot allocate device memory during
the call (its workspace is a fixed array in the library's device code).

CPU: the entry point rejects a problem whose workspace exceeds the array before any CUDA
call.  GPU: two calls in a row give the same results as kda_fwd (which takes its workspace
from the library's pool) on a fixed-length, a varlen and a decode-sized problem, and on one
that runs in pieces and one that runs the scan along T; the comparison is bit for bit, which
is stricter than the parity tolerances of the other tests.
This file is collected last, so a run that stops at the first failure has run every other
test before it; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest

from gated_delta_rule_23_gb300 import _native
from gated_delta_rule_23_gb300._native import KDA_DTYPE_NONE, KDA_ERR_UNSUPPORTED

SCRATCH = 268435456   # KDA_NOALLOC_SCRATCH_BYTES


def test_oversize_rejected_before_any_cuda_call():
    lib = _native.load()
    A = 1 << 20   # fake, aligned device addresses: the call must fail on the size check
    args = [A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 0.1, A + 0x5000, A + 0x6000, A + 0x7000, -5.0,
            None, None, KDA_DTYPE_NONE, None]
    assert lib.kda_fwd_workspace_size(1, 8192, 96, 0) > SCRATCH
    assert lib.kda_fwd_noalloc(*args, 1, 8192, 96, None) == KDA_ERR_UNSUPPORTED
    assert lib.kda_fwd_workspace_size(1, 1024, 96, 0) <= SCRATCH


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,H,cu", [(2, 333, 3, None), (1, 333, 3, np.array([0, 90, 90, 300, 333])), (2, 2, 3, None),
                                      (1, 4097, 40, None), (2, 8200, 8, None)])
def test_noalloc_matches_kda_fwd(B, T, H, cu):
    """The last two problems run in pieces (4097 tokens, 40 heads) and with the scan along T (2 x 8200 tokens,
    8 heads); slow decay, so that the state carries across pieces and groups."""
    import torch
    from gated_delta_rule_23_gb300 import kda_fwd
    from gated_delta_rule_23_gb300.device import to_device
    from gated_delta_rule_23_gb300.inputs import make_problem
    lib = _native.load()
    assert lib.kda_fwd_workspace_size(B, T, H, int(cu is not None)) <= SCRATCH
    if (B, T, H) == (1, 4097, 40):
        assert lib.kda_fwd_pieces(B, T, H, 0) >= 2
    if (B, T, H) == (2, 8200, 8):
        assert lib.kda_fwd_scan_groups(B, T, H, 0) >= 2
    p = make_problem(B=B, T=T, H=H, seed=31, cu_seqlens=cu, lower_bound=-0.05)
    dev = to_device(p)
    res = {}
    for noalloc in (False, True, True):
        out = torch.full_like(dev["q"], float("nan"))
        fin = torch.full((p.N, p.H, 128, 128), float("nan"), dtype=dev["sdt"], device="cuda")
        kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
                p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"], noalloc=noalloc)
        torch.cuda.synchronize()
        res.setdefault(noalloc, []).append((out.float().cpu().numpy(), fin.float().cpu().numpy()))
    ref = res[False][0]
    for o, f in res[True]:
        assert np.array_equal(o, ref[0]) and np.array_equal(f, ref[1])
