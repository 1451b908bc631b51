"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded
inputs, element by element, at the five standard workloads and at edge cases.

Tolerances (outputs rel-L2 <= 5e-3 and max-abs <= 3e-2, final states rel-L2 <= 5e-3,
varlen indexing bit-exact) are in tests/gpu_util.py.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_23_gb300 import kda_fwd
from gated_delta_rule_23_gb300.inputs import (STATE_BF16, STATE_FP32, STATE_NONE, bf16_bits, make_problem,
                                              make_workload)
from tests.gpu_util import assert_parity, rel_l2, run_gpu, to_device

pytestmark = pytest.mark.gpu


def oracle_run(p):
    return oracle.kda_fwd_problem(p)


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_workload_parity(idx):
    """All five standard workloads, every head and token, at full size."""
    p = make_workload(idx)
    out, fin = run_gpu(p)
    o_ref, f_ref = oracle_run(p)
    r = assert_parity(out, fin, o_ref, f_ref)
    print(f"workload {idx}: {r}")


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 31, 63, 64, 65, 127, 128, 129, 200, 333])
@pytest.mark.parametrize("varlen", [False, True])
def test_lengths_across_chunk_and_subblock_edges(T, varlen):
    """Every length across the 16-token sub-blocks and the 64-token chunks; as one varlen sequence the chunked
    kernels take every length (fixed-length problems of up to 16 tokens take the token-recurrent kernels)."""
    p = make_problem(B=1, T=T, H=3, seed=100 + T, cu_seqlens=np.array([0, T]) if varlen else None)
    out, fin = run_gpu(p)
    assert_parity(out, fin, *oracle_run(p))


@pytest.mark.parametrize("state", [STATE_NONE, STATE_BF16, STATE_FP32])
@pytest.mark.parametrize("with_initial", [False, True])
def test_state_dtypes_and_presence(state, with_initial):
    p = make_problem(B=2, T=150, H=2, seed=7, state_dtype=state, with_initial=with_initial)
    out, fin = run_gpu(p)
    o_ref, f_ref = oracle_run(p)
    assert_parity(out, fin, o_ref, f_ref)
    if state == STATE_NONE:
        assert fin is None


def test_initial_state_without_final_state():
    p = make_problem(B=1, T=100, H=2, seed=8, state_dtype=STATE_FP32, want_final=False)
    out, fin = run_gpu(p)
    assert fin is None
    assert_parity(out, None, *oracle_run(p)[:1], None)


def test_fixed_length_batch():
    p = make_problem(B=3, T=130, H=2, seed=9)
    out, fin = run_gpu(p)
    assert_parity(out, fin, *oracle_run(p))


def test_varlen_bitexact_against_separate_calls():
    """One varlen call equals separate per-sequence calls bit for bit (cu_seqlens indexing).  The separate
    calls are one-sequence varlen calls, so that every call takes the chunked form (fixed-length calls of
    1-16 tokens take the token-recurrent kernels)."""
    lens = [5, 0, 64, 131, 1, 17]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    p = make_problem(B=1, T=int(cu[-1]), H=3, seed=10, cu_seqlens=cu)
    out, fin = run_gpu(p)
    assert_parity(out, fin, *oracle_run(p))
    for n in range(len(lens)):
        s = slice(int(cu[n]), int(cu[n + 1]))
        pn = dataclasses.replace(p, q=p.q[:, s].copy(), k=p.k[:, s].copy(), v=p.v[:, s].copy(), g=p.g[:, s].copy(),
                                 beta=p.beta[:, s].copy(), initial_state=p.initial_state[n:n + 1].copy(),
                                 cu_seqlens=np.array([0, lens[n]], dtype=np.int64))
        o_n, f_n = run_gpu(pn)
        assert np.array_equal(o_n, out[:, s]), n
        assert np.array_equal(f_n[0], fin[n]), n
    assert np.array_equal(fin[1], p.initial_state[1])    # zero-length: final = initial exactly


def test_more_sequences_than_the_plan_orders():
    """2100 varlen sequences of 0-3 tokens: the plan kernel scans more sequences than its block has threads and
    leaves the longest-first order off (beyond 2048 sequences); every output and final state (empty sequences:
    final = initial exactly) against the oracle."""
    rng = np.random.default_rng(77)
    lens = rng.integers(0, 4, size=2100)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    p = make_problem(B=1, T=int(cu[-1]), H=1, seed=78, cu_seqlens=cu)
    out, fin = run_gpu(p)
    assert_parity(out, fin, *oracle_run(p))
    empty = np.flatnonzero(lens == 0)
    assert np.array_equal(fin[empty], p.initial_state[empty])


def test_all_sequences_empty():
    cu = np.zeros(4, dtype=np.int64)
    p = make_problem(B=1, T=0, H=2, seed=11, cu_seqlens=cu)
    out, fin = run_gpu(p)
    assert out.size == 0 and np.array_equal(fin, p.initial_state)


def test_guard_bands_untouched():
    """Writes stay inside out and final_state: canaries around both are unchanged."""
    p = make_problem(B=1, T=77, H=2, seed=12, cu_seqlens=np.array([0, 30, 77]))
    dev = to_device(p)
    pad = 4096
    canary = -12288.0          # exactly representable in bf16 and fp32
    out_buf = torch.full((pad * 2 + p.q.size,), canary, dtype=torch.bfloat16, device="cuda")
    fin_buf = torch.full((pad * 2 + p.initial_state.size,), canary, dtype=torch.float32, device="cuda")
    out = out_buf[pad:pad + p.q.size].view(p.q.shape)
    fin = fin_buf[pad:pad + p.initial_state.size].view(p.initial_state.shape)
    kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
            p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"])
    torch.cuda.synchronize()
    ob, fb = out_buf.float().cpu().numpy(), fin_buf.cpu().numpy()
    assert np.all(ob[:pad] == canary) and np.all(ob[-pad:] == canary)
    assert np.all(fb[:pad] == canary) and np.all(fb[-pad:] == canary)
    assert_parity(out.float().cpu().numpy(), fin.cpu().numpy(), *oracle_run(p))


@pytest.mark.parametrize("state", [STATE_BF16, STATE_FP32])
def test_in_place_state_update(state):
    p = make_problem(B=2, T=90, H=2, seed=13, state_dtype=state)
    out_sep, fin_sep = run_gpu(p)
    out_inp, fin_inp = run_gpu(p, inplace=True)
    assert np.array_equal(out_sep, out_inp) and np.array_equal(fin_sep, fin_inp)


def test_no_write_no_decay_keeps_state_exactly():
    """beta logit = -inf and lower_bound = 0: the state passes through unchanged (bit-exact)."""
    p = make_problem(B=1, T=150, H=2, seed=14, lower_bound=0.0)
    p.beta[:] = 0xFF80
    out, fin = run_gpu(p)
    assert np.array_equal(fin, p.initial_state)
    assert_parity(out, fin, *oracle_run(p))


def test_write_invariant_reads_back_v():
    """beta = 1 and q = k: every output equals scale * v."""
    p = make_problem(B=1, T=200, H=2, seed=15)
    p.q[:] = p.k
    p.beta[:] = bf16_bits(np.full(p.beta.shape, 100.0, np.float32))
    out, fin = run_gpu(p)
    o_ref, f_ref = oracle_run(p)
    assert_parity(out, fin, o_ref, f_ref)


@pytest.mark.parametrize("lb", [0.0, -0.5, -5.0])
def test_gate_extremes(lb):
    """Saturated gates at the lower bound (strongest decay the range argument allows) and none."""
    p = make_problem(B=1, T=160, H=2, seed=16, lower_bound=lb)
    p.A_log[:] = 12.0
    out, fin = run_gpu(p)
    assert_parity(out, fin, *oracle_run(p))


def test_split_and_resume():
    """Splitting at a token that is not a chunk boundary and chaining final -> initial state."""
    p = make_problem(B=1, T=300, H=2, seed=17)
    out, fin = run_gpu(p)
    cut = 101
    p1 = dataclasses.replace(p, q=p.q[:, :cut].copy(), k=p.k[:, :cut].copy(), v=p.v[:, :cut].copy(),
                             g=p.g[:, :cut].copy(), beta=p.beta[:, :cut].copy())
    o1, f1 = run_gpu(p1)
    p2 = dataclasses.replace(p, q=p.q[:, cut:].copy(), k=p.k[:, cut:].copy(), v=p.v[:, cut:].copy(),
                             g=p.g[:, cut:].copy(), beta=p.beta[:, cut:].copy(), initial_state=f1.astype(np.float32))
    o2, f2 = run_gpu(p2)
    o_ref, f_ref = oracle_run(p)
    assert_parity(np.concatenate([o1, o2], axis=1), f2, o_ref, f_ref)
    assert rel_l2(f2, fin) < 5e-3


def test_repeat_calls_are_deterministic():
    p = make_problem(B=1, T=257, H=4, seed=18, cu_seqlens=np.array([0, 100, 257]))
    dev = to_device(p)
    a = run_gpu(p, dev)
    b = run_gpu(p, dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_side_stream():
    p = make_problem(B=1, T=70, H=2, seed=19)
    dev = to_device(p)
    s = torch.cuda.Stream()
    out = torch.empty_like(dev["q"])
    fin = torch.empty((1, 2, 128, 128), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
            p.lower_bound, initial_state=dev["init"], final_state=fin, stream=s)
    s.synchronize()
    assert_parity(out.float().cpu().numpy(), fin.cpu().numpy(), *oracle_run(p))


def _call(p, dev, out, fin, **kw):
    kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
            p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"], **kw)


def _fresh(shape, dtype):
    """An output buffer filled with NaN, so that a call that writes nothing cannot pass on stale memory."""
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


@pytest.mark.parametrize("varlen", [False, True])
def test_caller_workspace_matches_pool_workspace(varlen):
    """kda_fwd_ws (caller-owned workspace, reused twice) and kda_fwd_ws_profiled give the same bits as kda_fwd."""
    from gated_delta_rule_23_gb300 import workspace_size
    cu = np.array([0, 90, 90, 300, 333]) if varlen else None
    p = make_problem(B=1, T=333, H=3, seed=21, cu_seqlens=cu)
    dev = to_device(p)
    nbytes = workspace_size(p.N, p.T, p.H, varlen)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    results = []
    for kw in ({}, {"workspace": ws}, {"workspace": ws},
               {"workspace": ws, "stage_events": [torch.cuda.Event(enable_timing=True) for _ in range(3)]}):
        if "stage_events" in kw:
            for e in kw["stage_events"]:
                e.record()   # creates the event handles
        out = torch.empty_like(dev["q"])
        fin = torch.empty((p.N, p.H, 128, 128), dtype=dev["sdt"], device="cuda")
        _call(p, dev, out, fin, **kw)
        torch.cuda.synchronize()
        results.append((out.float().cpu().numpy(), fin.float().cpu().numpy()))
        if "stage_events" in kw:
            e0, e1, e2 = kw["stage_events"]
            assert e0.elapsed_time(e1) >= 0 and e1.elapsed_time(e2) >= 0
    for o, f in results[1:]:
        assert np.array_equal(o, results[0][0]) and np.array_equal(f, results[0][1])
    assert_parity(results[0][0], results[0][1], *oracle_run(p))


# (B, T, H) -> pieces on a 152-SM GB300
PIECE_SHAPES = {(1, 8200, 24): 3, (1, 4097, 40): 2, (1, 32768, 24): 6}


@pytest.mark.parametrize("B,T,H,state,with_initial", [
    (1, 8200, 24, STATE_NONE, False), (1, 8200, 24, STATE_BF16, True), (1, 8200, 24, STATE_BF16, False),
    (1, 8200, 24, STATE_FP32, True), (1, 8200, 24, STATE_FP32, False), (1, 4097, 40, STATE_BF16, True),
    (1, 32768, 24, STATE_FP32, True)])
@pytest.mark.parametrize("lb", [-5.0, -0.05])
def test_pieces_match_single_launch(B, T, H, state, with_initial, lb):
    """Long fixed-length problems on few (sequence, head) pairs run in pieces along T (the next piece's prep
    kernel launched beside the recurrence over the current one): the same bits as the single-launch schedule
    of kda_fwd_ws_profiled, for every state kind, with 2 to 6 pieces and ragged last chunks; and work that
    the caller enqueues on the same stream after the call sees the finished results."""
    from gated_delta_rule_23_gb300 import _native, workspace_size
    pieces = _native.load().kda_fwd_pieces(B, T, H, 0)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert pieces == PIECE_SHAPES[(B, T, H)]
    assert pieces >= 2
    p = make_problem(B=B, T=T, H=H, seed=23, state_dtype=state, with_initial=with_initial, lower_bound=lb)
    dev = to_device(p)
    ws = torch.empty(workspace_size(p.N, p.T, p.H, False), dtype=torch.uint8, device="cuda")
    nch = -(-T // 64)
    assert ws.numel() == p.N * p.H * 128 * 128 * 4 + p.N * nch * p.H * 74240   # the piece-state header is there
    s = torch.cuda.Stream()
    results = []
    for kw in ({"workspace": ws, "stage_events": [None, None, None]}, {"workspace": ws}, {}):
        out = _fresh(dev["q"].shape, torch.bfloat16)
        fin = _fresh((p.N, p.H, 128, 128), dev["sdt"]) if dev["sdt"] is not None else None
        torch.cuda.synchronize()
        _call(p, dev, out, fin, stream=s, **kw)
        with torch.cuda.stream(s):   # ordered after the call on s only
            out_c = out.clone()
            fin_c = fin.clone() if fin is not None else None
        s.synchronize()
        assert torch.equal(out_c, out) and (fin is None or torch.equal(fin_c, fin))
        results.append((out.float().cpu().numpy(), None if fin is None else fin.float().cpu().numpy()))
    for o, f in results[1:]:
        assert np.array_equal(o, results[0][0])
        assert (f is None and results[0][1] is None) or np.array_equal(f, results[0][1])
    o_ref, f_ref = oracle_run(p)
    assert_parity(results[1][0], results[1][1], o_ref, f_ref)


@pytest.mark.parametrize("state", [STATE_BF16, STATE_FP32])
def test_pieces_in_place_state(state):
    """In pieces, an initial state updated in place (final_state = initial_state) gives the oracle's result."""
    from gated_delta_rule_23_gb300 import _native
    assert _native.load().kda_fwd_pieces(1, 8200, 24, 0) >= 2
    p = make_problem(B=1, T=8200, H=24, seed=24, state_dtype=state, lower_bound=-0.05)
    out, fin = run_gpu(p, inplace=True)
    assert_parity(out, fin, *oracle_run(p))


@pytest.mark.parametrize("B,T,H,state,with_initial,lb", [
    (2, 8200, 8, STATE_NONE, False, -5.0), (2, 8200, 8, STATE_BF16, True, -5.0), (2, 8200, 8, STATE_FP32, True, -5.0),
    (2, 8200, 8, STATE_NONE, False, -0.05), (2, 8200, 8, STATE_BF16, True, -0.05), (2, 8200, 8, STATE_BF16, False, -0.05),
    (2, 8200, 8, STATE_FP32, True, -0.05), (2, 8200, 8, STATE_FP32, False, 0.0), (1, 2049, 3, STATE_FP32, True, -0.05),
    (1, 32768, 8, STATE_BF16, True, -0.05), (2, 30000, 1, STATE_FP32, True, 0.0)])
def test_scan_along_t_matches_oracle(B, T, H, state, with_initial, lb):
    """Few (sequence, head) pairs and long sequences take the chunk-transition scan along T (groups composed in
    parallel, their start states chained in fp32, the groups run in parallel): within the parity tolerances
    of the oracle and close to the serial chain of kda_fwd_ws_profiled, for every state kind, 7 to 28 groups
    with ragged last groups and chunks and both compose forms (two CTAs per group and pair, or one carrying
    both states); and work that the caller enqueues on the same stream after
    the call sees the finished results.  With lower_bound = -5 the state forgets a chunk's start within the
    chunk (its decay underflows), so each group's transition is exactly zero and the scan gives the serial
    chain's bits; with -0.05 and 0 (no decay) the state carries across many chunks and groups."""
    from gated_delta_rule_23_gb300 import _native, workspace_size
    lib = _native.load()
    groups = lib.kda_fwd_scan_groups(B, T, H, 0)
    assert groups >= 7 and lib.kda_fwd_pieces(B, T, H, 0) == 1
    p = make_problem(B=B, T=T, H=H, seed=25, state_dtype=state, with_initial=with_initial, lower_bound=lb)
    dev = to_device(p)
    ws = torch.empty(workspace_size(p.N, p.T, p.H, False), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    results = []
    for kw in ({"workspace": ws}, {}, {"workspace": ws, "stage_events": [None, None, None]}):
        out = _fresh(dev["q"].shape, torch.bfloat16)
        fin = _fresh((p.N, p.H, 128, 128), dev["sdt"]) if dev["sdt"] is not None else None
        torch.cuda.synchronize()
        _call(p, dev, out, fin, stream=s, **kw)
        with torch.cuda.stream(s):
            out_c = out.clone()
            fin_c = fin.clone() if fin is not None else None
        s.synchronize()
        assert torch.equal(out_c, out) and (fin is None or torch.equal(fin_c, fin))
        results.append((out.float().cpu().numpy(), None if fin is None else fin.float().cpu().numpy()))
    # the caller's and the pool's workspace: the same schedule, the same bits
    assert np.array_equal(results[0][0], results[1][0])
    assert results[0][1] is None or np.array_equal(results[0][1], results[1][1])
    o_ref, f_ref = oracle_run(p)
    r_scan = assert_parity(results[0][0], results[0][1], o_ref, f_ref)
    r_serial = assert_parity(results[2][0], results[2][1], o_ref, f_ref)
    # the scan's own rounding stays small against the tolerance
    assert r_scan["out_rel_l2"] <= 1.5 * r_serial["out_rel_l2"] + 5e-4, (r_scan, r_serial)
    if lb == -5.0:
        assert np.array_equal(results[0][0], results[2][0])
    print(f"groups {groups} lb {lb}: scan {r_scan} serial {r_serial} "
          f"scan-serial out rel-L2 {rel_l2(results[0][0], results[2][0]):.3e}")


@pytest.mark.parametrize("state", [STATE_BF16, STATE_FP32])
def test_scan_in_place_state(state):
    """With the scan, an initial state updated in place (final_state = initial_state) gives the oracle's result:
    the last group's final state may not overwrite the initial state before the other groups have read it."""
    from gated_delta_rule_23_gb300 import _native
    assert _native.load().kda_fwd_scan_groups(2, 8200, 8, 0) >= 2
    p = make_problem(B=2, T=8200, H=8, seed=26, state_dtype=state, lower_bound=-0.05)
    out, fin = run_gpu(p, inplace=True)
    assert_parity(out, fin, *oracle_run(p))


def test_workspace_too_small_rejected():
    from gated_delta_rule_23_gb300 import KDAError, workspace_size
    p = make_problem(B=1, T=130, H=2, seed=22)
    dev = to_device(p)
    ws = torch.empty(workspace_size(p.N, p.T, p.H, False) - 256, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev["q"])
    with pytest.raises(KDAError):
        _call(p, dev, out, None, workspace=ws)


@pytest.mark.parametrize("T", [1, 3, 4, 5, 12, 16])
@pytest.mark.parametrize("state", [STATE_NONE, STATE_BF16, STATE_FP32])
def test_short_fixed_length_takes_the_token_recurrent_kernels(T, state):
    """kda_fwd on fixed-length problems of 1-16 tokens gives the bits of kda_fwd_recurrent (the same
    kernels) and meets the oracle."""
    p = make_problem(B=6, T=T, H=3, seed=60 + T, state_dtype=state)
    a = run_gpu(p)
    b = run_gpu(p, recurrent=True)
    assert np.array_equal(a[0], b[0])
    assert (a[1] is None and b[1] is None) or np.array_equal(a[1], b[1])
    assert_parity(*a, *oracle_run(p))


def _scaled(p, v_scale, state_std, seed):
    """Problem p with v multiplied by a power of two (exact in bf16) and fp32 initial states ~N(0, state_std)."""
    from gated_delta_rule_23_gb300.inputs import bf16_to_f32
    rng = np.random.default_rng(seed)
    v = bf16_bits(bf16_to_f32(p.v) * np.float32(v_scale))
    init = (rng.standard_normal(size=(p.N, p.H, 128, 128), dtype=np.float32) * np.float32(state_std))
    return dataclasses.replace(p, v=v, initial_state=init.astype(np.float32), state_dtype=STATE_FP32,
                               want_final=True)


@pytest.mark.parametrize("lb", [-5.0, -0.05])
def test_large_values_within_fp16_operand_range(lb):
    """Magnitudes that bf16 inputs allow and that approach the fp16 range of the tensor-core operands:
    v scaled by 256 (|v| up to ~1.3e3) and fp32 initial states ~N(0, 300), at strong and at slow decay."""
    from tests.gpu_util import OUT_REL_L2, STATE_REL_L2, parity_report
    p = _scaled(make_problem(B=1, T=333, H=4, seed=61, lower_bound=lb), 256.0, 300.0, 62)
    out, fin = run_gpu(p)   # raises if kda_device_status reports anything
    o_ref, f_ref = oracle_run(p)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(fin))
    # the relative bars (the absolute max-abs bar is for unit-scale inputs; these outputs are ~1e3 larger)
    r = parity_report(out, fin, o_ref, f_ref)
    assert r["out_rel_l2"] <= OUT_REL_L2 and r["state_rel_l2"] <= STATE_REL_L2, r


def test_values_beyond_fp16_operand_range_are_reported():
    """v scaled by 2^17 (|v| up to ~6e5) overflows the fp16 operands: the state turns non-finite and
    kda_device_status reports KDA_ERR_NONFINITE once (the report is cleared by reading it)."""
    from gated_delta_rule_23_gb300 import KDAError, device_status
    from gated_delta_rule_23_gb300._native import KDA_ERR_NONFINITE
    p = _scaled(make_problem(B=1, T=200, H=2, seed=63), 2.0 ** 17, 0.1, 64)
    dev = to_device(p)
    out = torch.empty_like(dev["q"])
    kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
            p.lower_bound, initial_state=dev["init"], final_state=None)
    with pytest.raises(KDAError) as e:
        device_status()
    assert e.value.status == KDA_ERR_NONFINITE
    device_status()   # cleared


@pytest.mark.parametrize("B,T,H,cu", [(1, 200, 2, None), (1, 200, 2, np.array([0, 70, 200])),
                                      (1, 4097, 40, None), (2, 8200, 8, None), (1, 2049, 3, None)])
def test_wait_that_gives_up_is_reported_and_the_next_call_is_correct(B, T, H, cu):
    """With a zero wait budget every wait of the chunked kernels gives up at once: the kernels drain their
    own work in flight, free their tensor memory and return, kda_device_status reports KDA_ERR_TIMEOUT once,
    and a following call with the default budget is correct against the oracle.  Nothing waits without a
    limit at any point.  The last three problems run in pieces (the next piece's prep kernel waiting, in the
    hardware, for a recurrence that gives up) and with the scan along T (both compose forms)."""
    from gated_delta_rule_23_gb300 import KDAError, _native, device_status
    from gated_delta_rule_23_gb300._native import KDA_DEFAULT_WAIT_POLLS, KDA_ERR_TIMEOUT
    lib = _native.load()
    if (B, T, H) == (1, 4097, 40):
        assert lib.kda_fwd_pieces(B, T, H, 0) >= 2
    if T > 2000 and H <= 8:
        assert lib.kda_fwd_scan_groups(B, T, H, 0) >= 2
    p = make_problem(B=B, T=T, H=H, seed=71, cu_seqlens=cu, lower_bound=-0.05)
    dev = to_device(p)
    out = torch.empty_like(dev["q"])
    fin = torch.empty((p.N, p.H, 128, 128), dtype=dev["sdt"], device="cuda")
    try:
        lib.kda_set_wait_limit(0)
        kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"],
                dev["dt_bias"], p.lower_bound, initial_state=dev["init"], final_state=fin,
                cu_seqlens=dev["cu"])
        with pytest.raises(KDAError) as e:
            device_status()
        assert e.value.status == KDA_ERR_TIMEOUT
    finally:
        lib.kda_set_wait_limit(KDA_DEFAULT_WAIT_POLLS)
    device_status()   # the report was cleared
    out, fin = run_gpu(p, dev)
    assert_parity(out, fin, *oracle_run(p))


@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("lb", [-5.0, -0.05])
def test_measurement_variants_within_parity(variant, lb):
    """The pages' own precision choices, as measurement variants of the chunked path (kda_fwd_ws_variant): the
    state rounded to bf16 between chunks (1), the fp16 Neumann-series inverse (2), both (3).  They stay within
    the parity bar against the oracle at strong and at slow decay, fixed length and varlen."""
    from gated_delta_rule_23_gb300 import device_status, workspace_size
    from tests.gpu_util import parity_report
    for cu in (None, np.array([0, 90, 333])):
        p = make_problem(B=1, T=333, H=3, seed=81, lower_bound=lb, cu_seqlens=cu)
        dev = to_device(p)
        out = torch.empty_like(dev["q"])
        fin = torch.empty((p.N, p.H, 128, 128), dtype=dev["sdt"], device="cuda")
        ws = torch.empty(workspace_size(p.N, p.T, p.H, cu is not None), dtype=torch.uint8, device="cuda")
        kda_fwd(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"], dev["dt_bias"],
                p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"], workspace=ws,
                variant=variant)
        device_status()
        o, f = out.float().cpu().numpy(), fin.float().cpu().numpy()
        o_ref, f_ref = oracle_run(p)
        r = assert_parity(o, f, o_ref, f_ref)
        print(f"variant {variant} lb {lb} varlen {cu is not None}: {parity_report(o, f, o_ref, f_ref)}")


def _random_cases(n=16, seed=2024):
    """Seeded random shapes across the schedules: fixed length with and without pieces or the scan along T,
    varlen with empty and ragged sequences; random state dtype, initial state and lower bound."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        varlen = i % 4 == 3
        H = int(rng.choice([1, 2, 3, 5, 8, 12, 24, 40]))
        if varlen:
            N = int(rng.integers(2, 9))
            cu = np.concatenate([[0], np.cumsum(rng.integers(0, 1500, size=N))]).astype(np.int64)
            B, T = 1, int(cu[-1])
        else:
            cu = None
            B, T = int(rng.integers(1, 3)), int(rng.choice([65, 700, 2049, 3000, 4100, 6000, 8200]))
        state = [STATE_NONE, STATE_BF16, STATE_FP32][int(rng.integers(0, 3))]
        cases.append(dict(B=B, T=T, H=H, cu=cu, state=state, with_initial=bool(rng.integers(0, 2)),
                          lb=float(rng.choice([-5.0, -1.0, -0.05])), seed=1000 + i))
    return cases


@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: f"B{c['B']}T{c['T']}H{c['H']}{'v' if c['cu'] is not None else ''}")
def test_random_shapes(case):
    """Random shapes against the oracle, whichever schedule each takes (single launch, pieces, scan, varlen)."""
    p = make_problem(B=case["B"], T=case["T"], H=case["H"], seed=case["seed"], cu_seqlens=case["cu"],
                     state_dtype=case["state"], with_initial=case["with_initial"], lower_bound=case["lb"])
    out, fin = run_gpu(p)
    assert_parity(out, fin, *oracle_run(p))
