"""Plants plausible mistakes in copies of the oracle's C source and checks that the pins
in test_oracle_pins.py catch every one of them (CPU only; the oracle itself is untouched).
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, exact text in kda_oracle.c, replacement); the first one is handled by _mutate
MUTANTS = [
    ("read-out before the write", None, None),
    ("no delta term (plain linear-attention write)",
     "u[vv] = b * (bf16_to_f64(job->v[row + vv]) - p);", "u[vv] = b * bf16_to_f64(job->v[row + vv]);"),
    ("delta sign flipped",
     "u[vv] = b * (bf16_to_f64(job->v[row + vv]) - p);", "u[vv] = b * (bf16_to_f64(job->v[row + vv]) + p);"),
    ("beta not applied to the write",
     "u[vv] = b * (bf16_to_f64(job->v[row + vv]) - p);", "u[vv] = (bf16_to_f64(job->v[row + vv]) - p);"),
    ("beta logit used without sigmoid",
     "const double b = sigmoid(bf16_to_f64(job->beta[t * H + h]));",
     "const double b = bf16_to_f64(job->beta[t * H + h]);"),
    ("decay along the value axis",
     "S[kk * KDA_D + vv] *= alpha[kk];", "S[kk * KDA_D + vv] *= alpha[vv];"),
    ("decay skipped",
     "S[kk * KDA_D + vv] *= alpha[kk];", "S[kk * KDA_D + vv] *= 1.0;"),
    ("A_log used without exp",
     "const double ea = exp((double)job->A_log[h]);", "const double ea = (double)job->A_log[h];"),
    ("dt_bias outside the scaled sum",
     "const double z = ea * (bf16_to_f64(job->g[row + c]) + (double)dtb[c]);",
     "const double z = ea * bf16_to_f64(job->g[row + c]) + (double)dtb[c];"),
    ("gate sigmoid sign flipped",
     "alpha[c] = exp(job->lower_bound * sigmoid(z));", "alpha[c] = exp(job->lower_bound * sigmoid(-z));"),
    ("gate without sigmoid",
     "alpha[c] = exp(job->lower_bound * sigmoid(z));", "alpha[c] = exp(job->lower_bound * z);"),
    ("q not normalised", "qh[c] *= rq;", "qh[c] *= 1.0;"),
    ("k not normalised", "kh[c] *= rk;", "kh[c] *= 1.0;"),
    ("no epsilon in the norm",
     "const double rq = 1.0 / sqrt(sq + 1e-6), rk = 1.0 / sqrt(sk + 1e-6);",
     "const double rq = 1.0 / sqrt(sq), rk = 1.0 / sqrt(sk);"),
    ("scale not applied",
     "job->out[row + vv] = job->scale * o;", "job->out[row + vv] = o;"),
    ("initial state read transposed",
     "? job->initial_state[(((int64_t)n * H + h) * KDA_D + vv) * KDA_D + kk]",
     "? job->initial_state[(((int64_t)n * H + h) * KDA_D + kk) * KDA_D + vv]"),
    ("final state written transposed",
     "job->final_state[(((int64_t)n * H + h) * KDA_D + vv) * KDA_D + kk] = S[kk * KDA_D + vv];",
     "job->final_state[(((int64_t)n * H + h) * KDA_D + kk) * KDA_D + vv] = S[kk * KDA_D + vv];"),
    ("read-out with k instead of q",
     "o += S[kk * KDA_D + vv] * qh[kk];", "o += S[kk * KDA_D + vv] * kh[kk];"),
    ("varlen sequence start off by one",
     "const int64_t bos = job->cu_seqlens ? job->cu_seqlens[n] : (int64_t)n * job->T;",
     "const int64_t bos = job->cu_seqlens ? job->cu_seqlens[n] + (n > 0) : (int64_t)n * job->T;"),
]

# The read-out-before-write mutant moves the output loop above the decay/write steps.
_READOUT = """        /* o = scale S^T q^ */
        for (int vv = 0; vv < KDA_D; ++vv) {
            double o = 0.0;
            for (int kk = 0; kk < KDA_D; ++kk)
                o += S[kk * KDA_D + vv] * qh[kk];
            job->out[row + vv] = job->scale * o;
        }
"""
_DECAY = "        /* S' = Diag(alpha) S */\n"


def _mutate(src, name, old, new):
    if old is None:
        assert _READOUT in src and _DECAY in src
        return src.replace(_READOUT, "").replace(_DECAY, _READOUT + _DECAY)
    assert src.count(old) == 1, name
    return src.replace(old, new)


PIN_TESTS = [
    pins.test_single_token_closed_form,
    pins.test_no_write_no_decay_is_identity,
    pins.test_write_invariant_beta_one_reads_back_v,
    pins.test_gate_saturation_decays_key_channels_exactly,
    pins.test_gate_unsaturated_value,
    pins.test_brute_force_dense_transitions,
    pins.test_golden_hand_worked_example,
    pins.test_varlen_equals_separate_calls_bitexact,
    pins.test_l2_norm_makes_q_and_k_scale_free,
]


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="kda_oracle_mut_")
    yield d
    oracle.use_library(None)
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(workdir, name, old, new):
    with open(SRC) as f:
        src = f.read()
    tag = "".join(ch if ch.isalnum() else "_" for ch in name)
    c_path = os.path.join(workdir, tag + ".c")
    so_path = os.path.join(workdir, tag + ".so")
    with open(c_path, "w") as f:
        f.write(_mutate(src, name, old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", so_path, c_path, "-lm", "-lpthread"],
                   check=True)
    caught = []
    oracle.use_library(so_path)
    try:
        for t in PIN_TESTS:
            try:
                t()
            except (AssertionError, ValueError):
                caught.append(t.__name__)
    finally:
        oracle.use_library(None)
    assert caught, f"no pin caught the planted mistake: {name}"
