"""The piece plan of kda_fwd_host, read through kda_fwd_host_plan (a host-side query; no GPU): the pieces cover
every token once.  Fixed-length problems over 512 tokens go in whole 64-token chunks: up to 8 big pieces, then a
tail that halves down to 2 chunks.  Varlen problems go in pieces of whole sequences, except the longest sequence
(the last of equals, from 4 chunks on), which comes last in chunk-aligned parts that halve."""
import ctypes

import numpy as np
import pytest

from gated_delta_rule_23_gb300 import _native

CH = 64


def plan(N, T, cu=None, max_pieces=64):
    lib = _native.load()
    ft = (ctypes.c_int64 * max_pieces)()
    tk = (ctypes.c_int64 * max_pieces)()
    fs = (ctypes.c_int * max_pieces)()
    ns = (ctypes.c_int * max_pieces)()
    cu_np = None if cu is None else np.ascontiguousarray(cu, dtype=np.int64)
    n = lib.kda_fwd_host_plan(N, T, None if cu_np is None else cu_np.ctypes.data, ft, tk, fs, ns, max_pieces)
    assert 0 <= n <= max_pieces
    assert lib.kda_fwd_host_plan(N, T, None if cu_np is None else cu_np.ctypes.data, None, None, None, None, 0) == n
    return [(ft[i], tk[i], fs[i], ns[i]) for i in range(n)]


def chunks(tokens):
    return -(-tokens // CH)


def assert_tiles(pieces, T):
    """Pieces in token order, each starting where the previous ended, covering [0, T)."""
    t = 0
    for t0, pt, _, _ in pieces:
        assert t0 == t and pt >= 0
        t += pt
    assert t == T


@pytest.mark.parametrize("T,expect", [
    (0, [0]), (1, [1]), (512, [512]),
    (513, [5, 4]),                                          # too short for a tail
    (4096, [8, 8, 7, 7, 7, 7, 7, 7, 4, 2]),
    (8192, [15, 15, 14, 14, 14, 14, 14, 14, 8, 4, 2]),      # workload 2
    (8200, [17, 17, 17, 16, 16, 16, 16, 8, 4, 2]),          # last chunk 8 tokens
])
def test_fixed_length_plan(T, expect):
    pieces = plan(2, T)
    assert_tiles(pieces, T)
    assert all(s0 == 0 and ns == 2 for _, _, s0, ns in pieces)
    if T <= 512:
        assert [pt for _, pt, _, _ in pieces] == expect
        return
    assert [chunks(pt) for _, pt, _, _ in pieces] == expect
    assert all(pt % CH == 0 for _, pt, _, _ in pieces[:-1])


@pytest.mark.parametrize("T", [600, 1000, 2500, 10_000, 32_768, 100_000, 1_000_000])
def test_fixed_length_plan_shape(T):
    """Big pieces within one chunk of each other, at most 8 of them, then a tail that halves to 2 chunks."""
    c = [chunks(pt) for _, pt, _, _ in plan(1, T)]
    assert_tiles(plan(1, T), T)
    assert all(a >= b for a, b in zip(c, c[1:]))            # never grows
    tail = []
    while len(c) > 1 and (not tail or c[-1] == 2 * tail[0]) and c[-1] < c[0]:
        tail.insert(0, c.pop())
    big = c
    assert len(big) <= 8 and max(big) - min(big) <= 1
    if tail:
        assert tail[-1] == 2 and all(a == 2 * b for a, b in zip(tail, tail[1:]))


def lens_of(cu):
    return np.diff(np.asarray(cu, dtype=np.int64))


def assert_varlen_plan(cu):
    cu = np.asarray(cu, dtype=np.int64)
    N, T = len(cu) - 1, int(cu[-1])
    pieces = plan(N, T, cu)
    covered = np.zeros(T, dtype=np.int32)
    for t0, pt, _, _ in pieces:
        covered[t0:t0 + pt] += 1
    assert (covered == 1).all()
    lens = lens_of(cu)
    star = max(range(N), key=lambda s: (lens[s], s))         # the longest, the last of equals
    split = chunks(int(lens[star])) >= 4
    whole = [p for p in pieces if not (split and p[2] == star)]
    tail = [p for p in pieces if split and p[2] == star]
    assert pieces[:len(whole)] == whole                     # the tail comes last
    seen = []
    for t0, pt, s0, ns in whole:                             # pieces of whole sequences, the star in none
        assert ns >= 1 and t0 == cu[s0] and pt == cu[s0 + ns] - cu[s0]
        assert not (split and s0 <= star < s0 + ns)
        seen += list(range(s0, s0 + ns))
    assert sorted(seen + ([star] if split else [])) == list(range(N))
    if split:
        assert len(tail) >= 2 and tail[0][0] == cu[star]
        for t0, pt, s0, ns in tail:
            assert ns == 1 and (t0 - cu[star]) % CH == 0
        c = [chunks(pt) for _, pt, _, _ in tail]
        assert all(a >= b for a, b in zip(c, c[1:])) and c[-1] <= 3
    return pieces


def test_varlen_equal_sequences():
    """8 sequences of 1024 tokens (workload 3): seven whole ones, then the last in 512, 256, 128 and 128 tokens."""
    pieces = assert_varlen_plan([1024 * i for i in range(9)])
    assert [(s0, ns, pt) for _, pt, s0, ns in pieces] == [(i, 1, 1024) for i in range(7)] + \
        [(7, 1, 512), (7, 1, 256), (7, 1, 128), (7, 1, 128)]


def test_varlen_irregular_sequences():
    """Workload 4's lengths: the 2497-token sequence last, in 1280, 640, 320, 192 and 65 tokens."""
    cu = [0, 43, 124, 208, 481, 1355, 3852, 3931, 4584, 4747, 7102, 8070, 8192]
    pieces = assert_varlen_plan(cu)
    assert [pt for _, pt, s0, _ in pieces if s0 == 5] == [1280, 640, 320, 192, 65]


def test_varlen_random_mixes():
    rng = np.random.default_rng(77)
    for _ in range(300):
        n = int(rng.integers(2, 40))
        lens = np.exp(rng.uniform(0, np.log(5000), n)).astype(np.int64)
        lens[rng.random(n) < 0.2] = 0
        cu = np.concatenate([[0], np.cumsum(lens)])
        if cu[-1] > 512:
            assert_varlen_plan(cu)


def test_single_piece_cases():
    assert plan(1, 5000, [0, 5000]) == [(0, 5000, 0, 1)]           # one varlen sequence: one piece
    assert plan(3, 500, [0, 100, 200, 500]) == [(0, 500, 0, 3)]     # 512 tokens or fewer
    assert plan(3, 0, [0, 0, 0, 0]) == [(0, 0, 0, 3)]


def test_rejected_inputs():
    lib = _native.load()
    assert lib.kda_fwd_host_plan(0, 100, None, None, None, None, None, 0) == -1
    assert lib.kda_fwd_host_plan(1, -1, None, None, None, None, None, 0) == -1
    bad = np.array([0, 300, 200, 600], dtype=np.int64)               # decreasing
    assert lib.kda_fwd_host_plan(3, 600, bad.ctypes.data, None, None, None, None, 0) == -1
    short = np.array([0, 300, 500], dtype=np.int64)                  # cu[N] != T
    assert lib.kda_fwd_host_plan(2, 600, short.ctypes.data, None, None, None, None, 0) == -1
