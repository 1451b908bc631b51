"""GPU parity of the token-recurrent entry point (kda_fwd_recurrent: decode steps and short
sequences) against the fp64 oracle, plus the properties that hold for it exactly: a chain of
one-token calls equals one call over the same tokens (fp32 state), varlen equals separate
calls, a zero-length sequence passes its state through.  Tolerances are those of
tests/gpu_util.py."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_23_gb300 import kda_fwd_recurrent
from gated_delta_rule_23_gb300.inputs import STATE_BF16, STATE_FP32, STATE_NONE, bf16_bits, make_problem
from tests.gpu_util import assert_parity, rel_l2, run_gpu, to_device

pytestmark = pytest.mark.gpu


def oracle_run(p):
    return oracle.kda_fwd_problem(p)


def run_rec(p, dev=None, inplace=False):
    return run_gpu(p, dev, inplace=inplace, recurrent=True)


def token_slice(p, s, **kw):
    return dataclasses.replace(p, q=p.q[:, s].copy(), k=p.k[:, s].copy(), v=p.v[:, s].copy(), g=p.g[:, s].copy(),
                               beta=p.beta[:, s].copy(), **kw)


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 31, 32, 33, 64, 100, 257])
def test_lengths_across_tile_edges(T):
    p = make_problem(B=2, T=T, H=3, seed=300 + T)
    assert_parity(*run_rec(p), *oracle_run(p))


@pytest.mark.parametrize("state", [STATE_NONE, STATE_BF16, STATE_FP32])
@pytest.mark.parametrize("with_initial", [False, True])
def test_state_dtypes_and_presence(state, with_initial):
    p = make_problem(B=3, T=40, H=2, seed=301, state_dtype=state, with_initial=with_initial)
    out, fin = run_rec(p)
    assert_parity(out, fin, *oracle_run(p))
    if state == STATE_NONE:
        assert fin is None


def test_decode_batch():
    """One token for each of 256 sequences at 16 heads: the decode-step shape."""
    p = make_problem(B=256, T=1, H=16, seed=302)
    assert_parity(*run_rec(p), *oracle_run(p))


@pytest.mark.parametrize("state", [STATE_BF16, STATE_FP32])
def test_in_place_decode_matches_separate_buffers(state):
    p = make_problem(B=8, T=3, H=4, seed=303, state_dtype=state)
    a = run_rec(p)
    b = run_rec(p, inplace=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def chain(p, seg):
    """Run p as consecutive calls of `seg` tokens, each starting from the last call's fp32 state."""
    state = p.initial_state
    outs = []
    for t0 in range(0, p.q.shape[1], seg):
        o, state = run_rec(token_slice(p, slice(t0, t0 + seg), initial_state=state.astype(np.float32)))
        outs.append(o)
    return np.concatenate(outs, axis=1), state


def test_chain_of_stage_aligned_calls_equals_one_call():
    """The kernel works in stages of 8 tokens from each sequence's start: calls of 8 tokens chaining an
    fp32 state give the bits of one call over all the tokens."""
    p = make_problem(B=2, T=24, H=3, seed=304)
    out_all, fin_all = run_rec(p)
    out_c, fin_c = chain(p, 8)
    assert np.array_equal(out_c, out_all)
    assert np.array_equal(fin_c, fin_all)


def test_decode_chain_matches_one_call():
    """One-token decode calls chaining an fp32 state agree with one call to fp32 rounding (the decay is
    applied per token instead of per stage) and both meet the oracle."""
    p = make_problem(B=2, T=21, H=3, seed=314)
    out_all, fin_all = run_rec(p)
    out_c, fin_c = chain(p, 1)
    assert rel_l2(out_c, out_all) < 1e-5 and rel_l2(fin_c, fin_all) < 1e-5
    o_ref, f_ref = oracle_run(p)
    assert_parity(out_c, fin_c, o_ref, f_ref)


def test_varlen_bitexact_against_separate_calls():
    lens = [5, 0, 16, 33, 1, 64]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    p = make_problem(B=1, T=int(cu[-1]), H=3, seed=305, cu_seqlens=cu)
    out, fin = run_rec(p)
    assert_parity(out, fin, *oracle_run(p))
    for n in range(len(lens)):
        s = slice(int(cu[n]), int(cu[n + 1]))
        o_n, f_n = run_rec(token_slice(p, s, initial_state=p.initial_state[n:n + 1].copy(), cu_seqlens=None))
        assert np.array_equal(o_n, out[:, s]), n
        assert np.array_equal(f_n[0], fin[n]), n
    assert np.array_equal(fin[1], p.initial_state[1])


def test_all_sequences_empty():
    cu = np.zeros(5, dtype=np.int64)
    p = make_problem(B=1, T=0, H=2, seed=306, cu_seqlens=cu, state_dtype=STATE_BF16)
    out, fin = run_rec(p)
    assert out.size == 0
    assert np.array_equal(bf16_bits(fin), p.initial_state)


def test_no_write_no_decay_keeps_state_exactly():
    p = make_problem(B=2, T=37, H=2, seed=307, lower_bound=0.0)
    p.beta[:] = 0xFF80
    out, fin = run_rec(p)
    assert np.array_equal(fin, p.initial_state)
    assert_parity(out, fin, *oracle_run(p))


def test_write_invariant_reads_back_v():
    """beta = 1 and q = k: every output equals scale * v (the oracle's pin, on this path)."""
    p = make_problem(B=1, T=50, H=2, seed=308)
    p.q[:] = p.k
    p.beta[:] = bf16_bits(np.full(p.beta.shape, 100.0, np.float32))
    assert_parity(*run_rec(p), *oracle_run(p))


@pytest.mark.parametrize("lb", [0.0, -0.5, -5.0])
def test_gate_extremes(lb):
    p = make_problem(B=1, T=48, H=2, seed=309, lower_bound=lb)
    p.A_log[:] = 12.0
    assert_parity(*run_rec(p), *oracle_run(p))


def test_agrees_with_chunked_path():
    """Both entry points evaluate the same recurrence: they agree within the parity bar."""
    cu = np.array([0, 7, 7, 70, 200], dtype=np.int64)
    p = make_problem(B=1, T=200, H=4, seed=310, cu_seqlens=cu)
    o_r, f_r = run_rec(p)
    o_c, f_c = run_gpu(p)
    assert rel_l2(o_r, o_c) < 5e-3 and rel_l2(f_r, f_c) < 5e-3


def test_guard_bands_untouched():
    p = make_problem(B=1, T=45, H=2, seed=311, cu_seqlens=np.array([0, 13, 45]))
    dev = to_device(p)
    pad = 4096
    canary = -12288.0
    out_buf = torch.full((pad * 2 + p.q.size,), canary, dtype=torch.bfloat16, device="cuda")
    fin_buf = torch.full((pad * 2 + p.initial_state.size,), canary, dtype=torch.float32, device="cuda")
    out = out_buf[pad:pad + p.q.size].view(p.q.shape)
    fin = fin_buf[pad:pad + p.initial_state.size].view(p.initial_state.shape)
    kda_fwd_recurrent(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], p.scale, out, dev["A_log"],
                      dev["dt_bias"], p.lower_bound, initial_state=dev["init"], final_state=fin, cu_seqlens=dev["cu"])
    torch.cuda.synchronize()
    ob, fb = out_buf.float().cpu().numpy(), fin_buf.cpu().numpy()
    assert np.all(ob[:pad] == canary) and np.all(ob[-pad:] == canary)
    assert np.all(fb[:pad] == canary) and np.all(fb[-pad:] == canary)
    assert_parity(out.float().cpu().numpy(), fin.cpu().numpy(), *oracle_run(p))


def test_repeat_calls_are_deterministic():
    p = make_problem(B=4, T=30, H=3, seed=312)
    dev = to_device(p)
    a = run_rec(p, dev)
    b = run_rec(p, dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("T", [1, 2, 4, 5, 7, 8])
@pytest.mark.parametrize("state", [STATE_BF16, STATE_FP32])
def test_decode_kernel_matches_staged_kernel(T, state):
    """Fixed-length problems of up to 7 tokens (5 with an fp32 state) take the barrier-free decode kernel; the
    same tokens as varlen sequences take the staged kernel.  Both evaluate the tokens as one stage with the
    same rounding: the bits agree."""
    p = make_problem(B=5, T=T, H=3, seed=320 + T, state_dtype=state)
    o_dec, f_dec = run_rec(p)
    cu = np.arange(0, 5 * T + 1, T, dtype=np.int64)
    flat = lambda a: a.reshape((1, 5 * T) + a.shape[2:]).copy()
    pv = dataclasses.replace(p, q=flat(p.q), k=flat(p.k), v=flat(p.v), g=flat(p.g), beta=flat(p.beta), cu_seqlens=cu)
    o_stg, f_stg = run_rec(pv)
    assert np.array_equal(o_dec.reshape(o_stg.shape), o_stg)
    assert np.array_equal(f_dec, f_stg)
