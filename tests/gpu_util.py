"""Helpers shared by the GPU tests: move a seeded problem to the device, run the CUDA
path through the C ABI, and compare with the oracle under the parity tolerances."""
import numpy as np
import torch

from gated_delta_rule_23_gb300 import device_status, kda_fwd
from gated_delta_rule_23_gb300.device import bf16_tensor, to_device  # noqa: F401
from gated_delta_rule_23_gb300.inputs import bf16_to_f32

# Parity bar: outputs rel-L2 <= 5e-3 and max-abs <= 3e-2; final states rel-L2 <= 5e-3.
OUT_REL_L2 = 5e-3
OUT_MAX_ABS = 3e-2
STATE_REL_L2 = 5e-3


def run_gpu(p, dev=None, inplace=False, recurrent=False):
    """Run the CUDA path on problem p (the chunked entry point, or the token-recurrent one);
    returns (out float32 [B,T,H,128], final float32 or None)."""
    dev = dev or to_device(p)
    out = torch.empty_like(dev["q"])
    fin = None
    if p.want_final and dev["sdt"] is not None:
        if inplace and dev["init"] is not None:
            fin = dev["init"]
        else:
            fin = torch.empty((p.N, p.H, 128, 128), dtype=dev["sdt"], device=dev["q"].device)
    kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
            p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"], recurrent=recurrent)
    device_status()            # synchronises; raises if a bounded device wait expired
    return out.float().cpu().numpy(), (None if fin is None else fin.float().cpu().numpy())


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def parity_report(out, fin, o_ref, f_ref):
    r = dict(out_rel_l2=rel_l2(out, o_ref), out_max_abs=float(np.abs(out - o_ref).max()) if out.size else 0.0)
    if f_ref is not None:
        r["state_rel_l2"] = rel_l2(fin, f_ref)
    return r


def assert_parity(out, fin, o_ref, f_ref):
    assert np.all(np.isfinite(out)), "non-finite output"
    r = parity_report(out, fin, o_ref, f_ref)
    if out.size:
        assert r["out_rel_l2"] <= OUT_REL_L2, r
        assert r["out_max_abs"] <= OUT_MAX_ABS, r
    if f_ref is not None:
        assert fin is not None and np.all(np.isfinite(fin))
        assert r["state_rel_l2"] <= STATE_REL_L2, r
    return r


def state_as_f64(p, arr):
    return None if arr is None else np.asarray(arr, np.float64)


__all__ = ["to_device", "run_gpu", "assert_parity", "parity_report", "rel_l2", "bf16_to_f32"]
