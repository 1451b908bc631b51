"""The host-buffer entry point kda_fwd_host against kda_fwd on the device: the pipelined pieces
(whole 64-token chunks with the state chained in fp32; for varlen problems, whole sequences) give the
same bits as one device call, for every state dtype and presence, ragged last pieces, batches, varlen
problems (in place too), pageable memory and T = 0; where the device call runs the scan along T (at most
16 (sequence, head) pairs, long sequences) and the decay is slow, the two agree within the parity bar."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_23_gb300 import _native, kda_fwd_host
from gated_delta_rule_23_gb300.inputs import STATE_BF16, STATE_FP32, STATE_NONE, make_problem
from tests.gpu_util import assert_parity, bf16_tensor, rel_l2, run_gpu

pytestmark = pytest.mark.gpu


def host_tensors(p, pinned=True):
    fix = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    h = dict(q=fix(bf16_tensor(p.q, "cpu")), k=fix(bf16_tensor(p.k, "cpu")), v=fix(bf16_tensor(p.v, "cpu")),
             g=fix(bf16_tensor(p.g, "cpu")), beta=fix(bf16_tensor(p.beta, "cpu")),
             A_log=fix(torch.from_numpy(p.A_log)), dt_bias=fix(torch.from_numpy(p.dt_bias)))
    h["cu"] = None if p.cu_seqlens is None else fix(torch.from_numpy(p.cu_seqlens))
    sdt = {STATE_BF16: torch.bfloat16, STATE_FP32: torch.float32}.get(p.state_dtype)
    h["init"] = None
    if p.initial_state is not None:
        h["init"] = fix(bf16_tensor(p.initial_state, "cpu") if p.state_dtype == STATE_BF16
                        else torch.from_numpy(p.initial_state))
    h["out"] = fix(torch.empty(p.q.shape, dtype=torch.bfloat16))
    h["fin"] = fix(torch.empty((p.N, p.H, 128, 128), dtype=sdt)) if (sdt is not None and p.want_final) else None
    return h


def run_host(p, pinned=True):
    h = host_tensors(p, pinned)
    kda_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], p.scale, h["out"], h["A_log"], h["dt_bias"],
                 p.lower_bound, initial_state=h["init"], final_state=h["fin"], cu_seqlens=h["cu"])
    return h["out"].float().numpy(), (None if h["fin"] is None else h["fin"].float().numpy())


def assert_same(p, pinned=True):
    out_h, fin_h = run_host(p, pinned)
    out_d, fin_d = run_gpu(p)
    assert np.array_equal(out_h, out_d)
    if fin_d is None:
        assert fin_h is None
    else:
        assert np.array_equal(fin_h, fin_d)


@pytest.mark.parametrize("T", [1, 64, 512, 513, 2500, 4096])
def test_pieces_equal_one_device_call(T):
    assert_same(make_problem(B=1, T=T, H=3, seed=400 + T))


@pytest.mark.parametrize("T", [2500, 8200])
def test_pieces_equal_one_device_call_slow_decay(T):
    """Slow decay (the state carries across every piece) with 17 heads: more than 16 pairs, so the device call
    runs one chain per pair (in pieces beside the prep kernel); the host pieces, ending in a tail of 16, 8, 4
    and 2 chunks at T = 8200 (the last chunk 8 tokens), give its bits."""
    assert _native.load().kda_fwd_scan_groups(1, T, 17, 0) == 1
    assert_same(make_problem(B=1, T=T, H=17, seed=420 + T, state_dtype=STATE_FP32, lower_bound=-0.05))


def test_scan_problem_within_parity_of_device_call():
    """Three heads, T = 4096, slow decay: the device call runs the scan along T, the host pieces (8 chunks and
    fewer) one chain per pair; both match the oracle within the parity bar and each other closely."""
    p = make_problem(B=1, T=4096, H=3, seed=421, state_dtype=STATE_FP32, lower_bound=-0.05)
    assert _native.load().kda_fwd_scan_groups(1, 4096, 3, 0) > 1
    out_h, fin_h = run_host(p)
    out_d, fin_d = run_gpu(p)
    o_ref, f_ref = oracle.kda_fwd_problem(p)
    assert_parity(out_h, fin_h, o_ref, f_ref)
    assert_parity(out_d, fin_d, o_ref, f_ref)
    assert rel_l2(out_h, out_d) < 2e-3 and rel_l2(fin_h, fin_d) < 2e-3


@pytest.mark.parametrize("state", [STATE_NONE, STATE_BF16, STATE_FP32])
@pytest.mark.parametrize("with_initial", [False, True])
def test_state_dtypes_and_presence(state, with_initial):
    assert_same(make_problem(B=2, T=1300, H=2, seed=410, state_dtype=state, with_initial=with_initial))


def test_initial_state_without_final_state():
    assert_same(make_problem(B=1, T=1500, H=2, seed=411, state_dtype=STATE_FP32, want_final=False))


def test_batch_rows_are_strided_copies():
    assert_same(make_problem(B=3, T=1100, H=4, seed=412))


@pytest.mark.parametrize("cu", [
    [0, 5, 5, 700, 1800, 1801],                       # empty sequences, a one-token last piece
    [0, 2000, 2010, 2020],                            # one sequence dominates
    list(np.cumsum([0] + [97 * (i % 5) + 31 for i in range(20)])),   # more sequences than pieces
    [0, 300, 600]])                                   # too short to cut
@pytest.mark.parametrize("state", [STATE_BF16, STATE_FP32])
def test_varlen_pieces_of_whole_sequences(cu, state):
    """Varlen problems run in pieces of whole sequences (each its own varlen call, no state between them); a last
    longest sequence of 4 chunks or more is cut into a halving tail of chunk pieces, its state chained in fp32."""
    cu = np.array(cu, dtype=np.int64)
    assert_same(make_problem(B=1, T=int(cu[-1]), H=3, seed=413, cu_seqlens=cu, state_dtype=state,
                             lower_bound=-0.05))


@pytest.mark.parametrize("cu,state,with_initial", [
    ([1024 * i for i in range(9)], STATE_FP32, True),            # 8 equal sequences: the last one in 8, 4, 2, 2 chunks
    ([1024 * i for i in range(9)], STATE_BF16, True),
    ([0, 100, 150, 3000], STATE_BF16, False),                   # a long last sequence, no initial state
    ([0, 2000, 2000, 2000, 2193], STATE_FP32, True),            # the first sequence longest, then empty ones
    ([0, 43, 124, 208, 481, 1355, 3852, 3931, 4584, 4747, 7102, 8070, 8192], STATE_FP32, True),  # irregular
    ([0, 700, 1400, 1657], STATE_NONE, False)])                 # no states; last chunk ragged
def test_varlen_longest_sequence_in_a_tail(cu, state, with_initial):
    """The longest sequence (the last of equals) comes last, in tail pieces of whole chunks that chain its state
    in fp32: the bits of one call, at slow decay, wherever it sits among the others."""
    cu = np.array(cu, dtype=np.int64)
    assert_same(make_problem(B=1, T=int(cu[-1]), H=3, seed=417, cu_seqlens=cu, state_dtype=state,
                             with_initial=with_initial, lower_bound=-0.05))


def _random_host_cases(n=10):
    """Seeded varlen mixes: 2 to 14 sequences of log-uniform lengths (with empty ones), 1 to 5 heads, every
    state kind, slow or strong decay."""
    rng = np.random.default_rng(4242)
    cases = []
    for i in range(n):
        nseq = int(rng.integers(2, 15))
        lens = np.exp(rng.uniform(np.log(1), np.log(1500), nseq)).astype(np.int64)
        lens[rng.random(nseq) < 0.15] = 0
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        if cu[-1] <= 512:   # below that the host call is one piece
            cu[-1] += 600
        cases.append(dict(cu=cu, H=int(rng.integers(1, 6)), seed=500 + i,
                          state=[STATE_NONE, STATE_BF16, STATE_FP32][i % 3], with_initial=bool(i % 2),
                          lb=[-0.05, -5.0][i % 2]))
    return cases


@pytest.mark.parametrize("case", _random_host_cases(), ids=lambda c: f"N{len(c['cu']) - 1}T{c['cu'][-1]}H{c['H']}")
def test_random_varlen_mixes(case):
    """Seeded random varlen mixes through the host pipeline: the bits of one device call."""
    assert_same(make_problem(B=1, T=int(case["cu"][-1]), H=case["H"], seed=case["seed"], cu_seqlens=case["cu"],
                             state_dtype=case["state"], with_initial=case["with_initial"], lower_bound=case["lb"]))


def test_varlen_pieces_in_place_state():
    """In place (final_state = initial_state, host memory): each piece reads its sequences' initial states
    before its final states overwrite them, and no two pieces share a sequence."""
    cu = np.array(np.cumsum([0] + [300, 700, 64, 900, 1, 600]), dtype=np.int64)
    p = make_problem(B=1, T=int(cu[-1]), H=2, seed=416, cu_seqlens=cu, lower_bound=-0.05)
    h = host_tensors(p)
    kda_fwd_host(h["q"], h["k"], h["v"], h["g"], h["beta"], p.scale, h["out"], h["A_log"], h["dt_bias"],
                 p.lower_bound, initial_state=h["init"], final_state=h["init"], cu_seqlens=h["cu"])
    out_d, fin_d = run_gpu(p)
    assert np.array_equal(h["out"].float().numpy(), out_d)
    assert np.array_equal(h["init"].float().numpy(), fin_d)


def test_pageable_memory():
    assert_same(make_problem(B=1, T=1200, H=2, seed=414), pinned=False)


def test_no_tokens():
    p = make_problem(B=1, T=0, H=2, seed=415, cu_seqlens=np.zeros(3, dtype=np.int64))
    out, fin = run_host(p)
    assert out.size == 0
    assert np.array_equal(fin, p.initial_state)
