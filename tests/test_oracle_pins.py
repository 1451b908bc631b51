"""Pins for the CPU oracle: checks against closed forms, invariants, brute force and
independent (chunked) formulations -- never against the oracle itself.

Each test names the property of the method it relies on.  The method: the gated
delta rule of Kimi Delta Attention as the FlashKDA pages state it (guancyxx.cn
FlashKDA article, section 一 and section 2.2; FlashKDA README mirror, sections
"内核 API" and "将 FlashKDA 用作 FLA 后端").
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from gated_delta_rule_23_gb300 import inputs
from gated_delta_rule_23_gb300.inputs import bf16_bits, bf16_to_f32, make_problem
from tests import chunked_ref

HERE = os.path.dirname(os.path.abspath(__file__))


def run(p, **kw):
    return oracle.kda_fwd_problem(p, **kw)


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def small(seed=0, T=37, H=2, B=1, **kw):
    return make_problem(B=B, T=T, H=H, seed=seed, **kw)


# ---------------------------------------------------------------- closed forms

def test_single_token_closed_form():
    """T = 1: o = scale [S'^T q^ + b (k^ . q^)(v - S'^T k^)], S_1 = S' + b k^ (v - S'^T k^)^T."""
    p = small(seed=3, T=1, H=3)
    out, fin = run(p)
    qh, kh, v, b, a = chunked_ref.prepare(p)
    init = p.initial_state_f64()
    for h in range(p.H):
        S0 = init[0, h].T                       # math state S[k][v]
        Sp = np.exp(a[0, 0, h])[:, None] * S0
        r = v[0, 0, h] - Sp.T @ kh[0, 0, h]
        o = p.scale * (Sp.T @ qh[0, 0, h] + b[0, 0, h] * (kh[0, 0, h] @ qh[0, 0, h]) * r)
        S1 = Sp + b[0, 0, h] * np.outer(kh[0, 0, h], r)
        np.testing.assert_allclose(out[0, 0, h], o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(fin[0, h], S1.T, rtol=1e-12, atol=1e-13)


def test_no_write_no_decay_is_identity():
    """beta logit = -inf gives b = 0 and lower_bound = 0 gives a = 0: the state is untouched
    (bit-exact) and o_t = scale S0^T q^_t, a plain mat-vec that pins the [V, K] state layout."""
    p = small(seed=4, T=20, H=2, lower_bound=0.0)
    p.beta[:] = 0xFF80                           # bf16 -inf
    out, fin = run(p)
    init = p.initial_state_f64()
    assert np.array_equal(fin, init)
    qh = chunked_ref.prepare(p)[0]
    for h in range(p.H):
        np.testing.assert_allclose(out[0, :, h], p.scale * qh[0, :, h] @ init[0, h].T, rtol=1e-12, atol=1e-14)


def test_write_invariant_beta_one_reads_back_v():
    """With b = 1 the write makes S_t^T k^_t = v_t (up to |k^|^2 = s/(s + 1e-6)); with q = k the
    read-out therefore returns scale * v_t for every token, whatever the gates and the state."""
    p = small(seed=5, T=50, H=2)
    p.q[:] = p.k
    p.beta[:] = bf16_bits(np.full(p.beta.shape, 100.0, np.float32))   # sigmoid(100) == 1.0 in fp64
    out, _ = run(p)
    v = bf16_to_f32(p.v).astype(np.float64)
    np.testing.assert_allclose(out, p.scale * v, rtol=0, atol=1e-6)


def test_gate_saturation_decays_key_channels_exactly():
    """exp(A_log) = e^20 saturates the sigmoid: g + dt_bias > 0 gives a = lower_bound exactly, < 0
    gives a = 0.  With b = 0 the state's key channels (contiguous axis of [V, K]) decay by exactly
    exp(lower_bound * T) on the first set and not at all on the second."""
    T, lb = 7, -0.75
    p = small(seed=6, T=T, H=2, lower_bound=lb)
    p.beta[:] = 0xFF80
    p.A_log[:] = 20.0
    p.dt_bias[:] = 0.0
    sign = np.where(np.arange(128) % 3 == 0, 1.0, -1.0).astype(np.float32)
    p.g[:] = bf16_bits(np.broadcast_to(sign, p.g.shape).copy())
    _, fin = run(p)
    init = p.initial_state_f64()
    expect = init * np.where(sign > 0, math.exp(lb * T), 1.0)[None, None, None, :]
    np.testing.assert_allclose(fin, expect, rtol=1e-13, atol=0)
    # dt_bias enters the same sum as g: g = 0 and dt_bias = sign give the same decay
    p.g[:] = 0
    p.dt_bias[:] = sign[None, :]
    _, fin2 = run(p)
    np.testing.assert_allclose(fin2, expect, rtol=1e-13, atol=0)


def test_gate_unsaturated_value():
    """A_log = 0 (exp = 1), g = 1, dt_bias = 0.5 on every channel, b = 0: each step multiplies the
    state by exp(lower_bound * sigmoid(1.5)), sigmoid(1.5) = 1 / (1 + e^-1.5)."""
    T, lb = 5, -3.0
    p = small(seed=7, T=T, H=1, lower_bound=lb)
    p.beta[:] = 0xFF80
    p.A_log[:] = 0.0
    p.dt_bias[:] = 0.5
    p.g[:] = bf16_bits(np.ones(p.g.shape, np.float32))
    _, fin = run(p)
    step = math.exp(lb / (1.0 + math.exp(-1.5)))
    np.testing.assert_allclose(fin, p.initial_state_f64() * step ** T, rtol=1e-13)


# ---------------------------------------------------------------- invariants

def test_l2_norm_makes_q_and_k_scale_free():
    """q^ and k^ are unit vectors: scaling q and k by a power of two (exact in bf16) leaves the
    result unchanged up to the 1e-6 in the norm."""
    p = small(seed=8, T=40, H=2)
    o1, f1 = run(p)
    for arr, fac in ((p.q, 8.0), (p.k, 0.25)):
        arr[:] = bf16_bits(bf16_to_f32(arr) * np.float32(fac))
    o2, f2 = run(p)
    assert rel_l2(o2, o1) < 1e-7 and rel_l2(f2, f1) < 1e-7


def test_linear_in_v_and_state_and_scale():
    """For fixed q, k, g, beta the map (v, S0) -> (out, S_T) is linear, and out is proportional to scale."""
    rng = np.random.default_rng(9)
    p1 = small(seed=9, T=45, H=2)
    p2 = small(seed=9, T=45, H=2)
    v1 = rng.integers(-8, 9, size=p1.v.shape).astype(np.float32)
    v2 = rng.integers(-8, 9, size=p1.v.shape).astype(np.float32)
    s1 = rng.integers(-4, 5, size=p1.initial_state.shape).astype(np.float32)
    s2 = rng.integers(-4, 5, size=p1.initial_state.shape).astype(np.float32)
    p1.v[:], p2.v[:] = bf16_bits(v1), bf16_bits(v2)
    p1.initial_state[:], p2.initial_state[:] = s1, s2
    o1, f1 = run(p1)
    o2, f2 = run(p2)
    p1.v[:] = bf16_bits(v1 + v2)
    p1.initial_state[:] = s1 + s2
    o12, f12 = run(p1)
    assert rel_l2(o12, o1 + o2) < 1e-12 and rel_l2(f12, f1 + f2) < 1e-12
    p2.scale = 3.0 * p2.scale
    o2s, f2s = run(p2)
    assert rel_l2(o2s, 3.0 * o2) < 1e-14 and np.array_equal(f2s, f2)


def test_zero_query_gives_zero_output():
    p = small(seed=10, T=9, H=2)
    p.q[:] = 0
    out, _ = run(p)
    assert np.all(out == 0.0)


# ---------------------------------------------------------------- brute force

def test_brute_force_dense_transitions():
    """T <= 8: S_t = prod_{s<=t} M_s S0 + sum_{s<=t} (prod_{s<r<=t} M_r) b_s k^_s v_s^T with the dense
    K x K transition M_s = (I - b_s k^_s k^_s^T) Diag(alpha_s), evaluated by explicit matrix products."""
    p = small(seed=11, T=8, H=2)
    out, fin = run(p)
    qh, kh, v, b, a = chunked_ref.prepare(p)
    init = p.initial_state_f64()
    I = np.eye(128)
    for h in range(p.H):
        M = [(I - b[0, s, h] * np.outer(kh[0, s, h], kh[0, s, h])) @ np.diag(np.exp(a[0, s, h]))
             for s in range(p.T)]
        for t in range(p.T):
            prod_all = I
            for s in range(t + 1):
                prod_all = M[s] @ prod_all
            St = prod_all @ init[0, h].T
            for s in range(t + 1):
                tail = I
                for r in range(s + 1, t + 1):
                    tail = M[r] @ tail
                St = St + tail @ (b[0, s, h] * np.outer(kh[0, s, h], v[0, s, h]))
            np.testing.assert_allclose(out[0, t, h], p.scale * St.T @ qh[0, t, h], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(fin[0, h], St.T, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- chunked forms

@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("inverse", [chunked_ref.inv_forward_substitution, chunked_ref.inv_neumann,
                                     chunked_ref.inv_blocked])
def test_chunked_form_equals_recurrence(C, inverse):
    p = small(seed=12, T=150, H=2)
    out, fin = run(p)
    oc, fc = chunked_ref.chunked_direct(p, C=C, inverse=inverse)
    assert rel_l2(oc, out) < 1e-10 and rel_l2(fc, fin) < 1e-10


@pytest.mark.parametrize("groups", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("lb", [-0.05, 0.0])
def test_scan_along_t_equals_recurrence(groups, lb):
    """The chunk-transition scan along T (group maps S -> M S + B composed from S = I with U0 = 0 and from
    S = 0, start states chained, groups re-run) equals the token recurrence, with ragged last groups and chunks;
    with slow or no decay the group transitions stay far above the tolerance (a mistake in the chaining would
    show at their size), so the chaining is exercised."""
    p = inputs.make_problem(B=2, T=1000, H=1, seed=31, lower_bound=lb)
    out, fin = run(p)
    oc, fc, Ms = chunked_ref.scan_form(p, groups)
    assert rel_l2(oc, out) < 1e-10 and rel_l2(fc, fin) < 1e-10
    if groups > 1:
        assert min(np.linalg.norm(M) for M in Ms) > (1.0 if lb == 0.0 else 1e-6)


@pytest.mark.parametrize("lb", [-0.05, 0.0, -5.0])
def test_lookahead_form_equals_recurrence(lb):
    """The two-chunk lookahead of the chunk recurrence (the next chunk's W S formed as W Diag(Gamma_C) S_c +
    (W K~^T) U_c from this chunk's start state) equals the token recurrence, varlen with ragged and one-chunk
    sequences; with slow or no decay the lookahead term carries a large part of the product, so a mistake in it
    (a transposed or missing factor) would show."""
    p = inputs.make_problem(B=1, T=600, H=1, seed=33, lower_bound=lb, cu_seqlens=np.array([0, 40, 300, 600]))
    out, fin = run(p)
    oc, fc, shares = chunked_ref.lookahead_form(p)
    assert rel_l2(oc, out) < 1e-10 and rel_l2(fc, fin) < 1e-10
    if lb > -1.0:
        assert len(shares) >= 5 and min(shares) > 0.05


def test_subblock_factorised_chunked_form_equals_recurrence():
    """The 16-row sub-block factorisation of the decay (no overflow at lower_bound = -5, C = 64)."""
    p = inputs.make_problem(B=1, T=200, H=2, seed=13, cu_seqlens=np.array([0, 1, 64, 65, 200]))
    out, fin = run(p)
    oc, fc = chunked_ref.chunked_subblock(p, C=64)
    assert np.all(np.isfinite(oc)) and np.all(np.isfinite(fc))
    assert rel_l2(oc, out) < 1e-10 and rel_l2(fc, fin) < 1e-10


def test_strong_decay_lower_bound_minus5_subblock():
    """All gates at the bound (sigmoid saturated at 1): the decay per token is e^-5 on every
    channel, the worst case for the factorised form's range."""
    p = small(seed=14, T=130, H=1)
    p.A_log[:] = 20.0
    p.dt_bias[:] = 0.0
    p.g[:] = bf16_bits(np.ones(p.g.shape, np.float32))
    out, fin = run(p)
    oc, fc = chunked_ref.chunked_subblock(p, C=64)
    assert np.all(np.isfinite(oc)) and rel_l2(oc, out) < 1e-10 and rel_l2(fc, fin) < 1e-10


# ---------------------------------------------------------------- varlen and resume

def test_varlen_equals_separate_calls_bitexact():
    lens = [5, 0, 64, 17, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    p = make_problem(B=1, T=int(cu[-1]), H=2, seed=15, cu_seqlens=cu)
    out, fin = run(p)
    for n in range(len(lens)):
        s = slice(int(cu[n]), int(cu[n + 1]))
        init_n = p.initial_state_f64()[n:n + 1]
        o_n, f_n = oracle.kda_fwd(p.q[:, s], p.k[:, s], p.v[:, s], p.g[:, s], p.beta[:, s], p.scale,
                                  p.A_log, p.dt_bias, p.lower_bound, initial_state=init_n)
        assert np.array_equal(o_n, out[:, s])
        assert np.array_equal(f_n[0], fin[n])
    assert np.array_equal(fin[1], p.initial_state_f64()[1])     # zero-length: final = initial


def test_fixed_batch_equals_varlen_layout():
    p = make_problem(B=3, T=21, H=2, seed=16)
    out, fin = run(p)
    cu = np.arange(0, 64, 21, dtype=np.int64)
    flat = lambda a: a.reshape((1, -1) + a.shape[2:])
    o2, f2 = oracle.kda_fwd(flat(p.q), flat(p.k), flat(p.v), flat(p.g), flat(p.beta), p.scale, p.A_log,
                            p.dt_bias, p.lower_bound, initial_state=p.initial_state_f64(), cu_seqlens=cu)
    assert np.array_equal(o2.reshape(out.shape), out) and np.array_equal(f2, fin)


@pytest.mark.parametrize("split", [1, 23, 64])
def test_split_and_resume_equals_single_call(split):
    p = small(seed=17, T=100, H=2)
    out, fin = run(p)
    s1, s2 = slice(0, split), slice(split, p.T)
    args = lambda s: (p.q[:, s], p.k[:, s], p.v[:, s], p.g[:, s], p.beta[:, s], p.scale, p.A_log, p.dt_bias,
                      p.lower_bound)
    o1, f1 = oracle.kda_fwd(*args(s1), initial_state=p.initial_state_f64())
    o2, f2 = oracle.kda_fwd(*args(s2), initial_state=f1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(f2, fin, rtol=1e-12, atol=1e-14)


def test_threads_do_not_change_results():
    p = make_problem(B=2, T=30, H=3, seed=18)
    o1, f1 = run(p, nthreads=1)
    o4, f4 = run(p, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(f1, f4)


def test_rejects_bad_cu_seqlens():
    p = make_problem(B=1, T=10, H=1, seed=19)
    with pytest.raises(ValueError):
        oracle.kda_fwd(p.q, p.k, p.v, p.g, p.beta, p.scale, p.A_log, p.dt_bias, p.lower_bound,
                       cu_seqlens=np.array([0, 6, 4, 10]))


# ---------------------------------------------------------------- hand-worked example

def _golden_eval(expr, consts):
    return eval(expr, {"__builtins__": {}}, dict(consts))


def test_golden_hand_worked_example():
    """tests/golden/onehot_three_tokens.json: a three-token example on one-hot vectors, worked by
    hand from the definition (derivation in the fixture)."""
    with open(os.path.join(HERE, "golden", "onehot_three_tokens.json")) as f:
        gold = json.load(f)
    T, H = 3, 1
    p = make_problem(B=1, T=T, H=H, seed=0, lower_bound=gold["lower_bound"], scale=gold["scale"])
    for arr in (p.q, p.k, p.v, p.g):
        arr[:] = 0
    p.A_log[:] = gold["A_log"]
    p.dt_bias[:] = 0.0
    p.initial_state[:] = 0.0
    for (vv, kk), val in gold["initial_state_vk"]:
        p.initial_state[0, 0, vv, kk] = val
    for t, tok in enumerate(gold["tokens"]):
        for name in ("q", "k", "v"):
            vec = np.zeros(128, np.float32)
            for idx, val in tok[name]:
                vec[idx] = val
            getattr(p, name)[0, t, 0] = bf16_bits(vec)
        gvec = np.full(128, tok["g_default"], np.float32)
        for idx, val in tok.get("g", []):
            gvec[idx] = val
        p.g[0, t, 0] = bf16_bits(gvec)
        p.beta[0, t, 0] = bf16_bits(np.array([tok["beta_logit"]], np.float32))[0]
    out, fin = run(p)
    consts = {"sqrt": math.sqrt, "exp": math.exp}
    for name, expr in gold["constants"].items():      # in file order; later ones may use earlier ones
        consts[name] = _golden_eval(expr, consts)
    expect_out = np.zeros((T, 128))
    for t, vv, expr in gold["expected_out"]:
        expect_out[t, vv] = _golden_eval(expr, consts)
    expect_fin = np.zeros((128, 128))
    for vv, kk, expr in gold["expected_final_state_vk"]:
        expect_fin[vv, kk] = _golden_eval(expr, consts)
    np.testing.assert_allclose(out[0, :, 0], expect_out, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(fin[0, 0], expect_fin, rtol=1e-13, atol=1e-15)
