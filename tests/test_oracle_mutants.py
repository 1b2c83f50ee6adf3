"""Planted mistakes in the oracle: each must fail at least one of its pins.

The pins of tests/test_oracle_pins.py are meant to catch any plausible mistake in the oracle (a
dropped term, a wrong sign, a wrong index, a transposed operand, a missing chain-rule factor).
This test checks that claim directly: it plants one mistake at a time into a copy of
oracle/kda_oracle.c (a textual edit of one line), compiles the copy with the oracle's own gcc
command into a temporary directory, runs every pin against that build and requires at least one
pin to fail.  The real oracle source is never modified.
"""
import os
import shutil
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, the line as written, the line with the planted mistake)
MUTANTS = [
    # forward: the token step and the read-out
    ("decay on the value dim", "for (int j = 0; j < d; ++j) S[i * d + j] *= e;",
     "for (int j = 0; j < d; ++j) S[i * d + j] *= exp(x->g[j]) + 0.0 * e;"),
    ("one gate for every channel", "double e = exp(x->g[i]);", "double e = exp(x->g[0]);"),
    ("prediction sign", "u[j] = x->v[j] - acc;", "u[j] = x->v[j] + acc;"),
    ("prediction reads S transposed", "for (int i = 0; i < d; ++i) acc += S[i * d + j] * x->k[i];",
     "for (int i = 0; i < d; ++i) acc += S[j * d + i] * x->k[i];"),
    ("write without beta", "double bk = x->beta * x->k[i];", "double bk = x->k[i];"),
    ("read-out transposed", "for (int i = 0; i < d; ++i) acc += S[i * d + j] * x.q[i];",
     "for (int i = 0; i < d; ++i) acc += S[j * d + i] * x.q[i];"),
    ("read-out with k", "for (int i = 0; i < d; ++i) acc += S[i * d + j] * x.q[i];",
     "for (int i = 0; i < d; ++i) acc += S[i * d + j] * x.k[i];"),
    ("read-out without scale", "o[j] = J->scale * acc;", "o[j] = acc;"),
    ("raw gate without exp(A_log)", "x->g[c] = -exp(J->A_log[h]) * softplus(a);",
     "x->g[c] = -J->A_log[h] * softplus(a);"),
    ("softplus branch", "return (x > 0 ? x : 0.0) + log1p(exp(-fabs(x)));",
     "return (x > 0 ? x : 0.0) + log1p(exp(-x));"),
    ("L2 norm without eps", "x->qn = sqrt(sq + J->eps);", "x->qn = sqrt(sq);"),
    ("L2 norm of q only", "x->k[c] /= x->kn;", "x->k[c] /= 1.0;"),
    # backward: the adjoint of the step, the gate chain, the L2-norm chain
    ("dq without scale", "s->dq[i] = J->scale * acc;", "s->dq[i] = acc;"),
    ("dbeta sign", "db += x.k[i] * acc;", "db -= x.k[i] * acc;"),
    ("du without beta", "s->du[j] = x.beta * acc;", "s->du[j] = acc;"),
    ("dk misses the prediction term", "s->dk[i] -= acc;", "s->dk[i] += 0.0 * acc;"),
    ("dg from the undecayed state", "acc += s->Sp[i * d + j] * v;", "acc += S[i * d + j] * v;"),
    ("dS not decayed", "dS[i * d + j] = e * v;", "dS[i * d + j] = v;"),
    ("dS keeps the write term", "double v = dS[i * d + j] - x.k[i] * s->du[j];",
     "double v = dS[i * d + j];"),
    ("da sigmoid sign", "double da = dg * (-eA) * sigmoid(J->gin[base + c] + J->dt_bias[(int64_t)h * d + c]);",
     "double da = dg * (-eA) * sigmoid(-J->gin[base + c] - J->dt_bias[(int64_t)h * d + c]);"),
    ("dA_log without g", "dA += dg * x.g[c]; /* dg/dA_log = g */", "dA += dg;"),
    ("L2 backward without projection", "J->dq[base + c] = (s->dq[c] - x.q[c] * pq) / x.qn;",
     "J->dq[base + c] = s->dq[c] / x.qn;"),
    ("checkpoint off by one", "memcpy(S, s->seg + (t - t0) * dd, sizeof(double) * dd); /* S_{t-1} */",
     "memcpy(S, s->seg + (t > t0 ? t - t0 - 1 : 0) * dd, sizeof(double) * dd);"),
    # fragment algebra and the transfer walk
    ("walk uses M transposed", "double m = reverse ? Mf[(size_t)l * d + i] : Mf[(size_t)i * d + l];",
     "double m = reverse ? Mf[(size_t)i * d + l] : Mf[(size_t)l * d + i];"),
    ("walk drops B", "double acc = Bf[(size_t)i * d + j];", "double acc = 0.0 * Bf[(size_t)i * d + j];"),
    ("summary M from a zero start", "eye[f * dd + (size_t)i * d + i] = 1.0;",
     "eye[f * dd + (size_t)i * d + i] = 0.0;"),
]


def _pins():
    """Every pin as (name, callable), cheapest first."""
    out = [
        ("worked_examples_d2", pins.test_worked_examples_d2),
        ("zero_state_single_token_d128", pins.test_zero_state_single_token_d128),
        ("pure_decay", lambda: pins.test_pure_decay_closed_form(False)),
        ("plain_read_out", lambda: pins.test_pure_decay_closed_form(True)),
        ("one_hot_keys", pins.test_one_hot_keys_gated_linear_attention),
        ("exact_read_back", pins.test_exact_read_back),
        ("pack_equals_documents", pins.test_pack_equals_documents),
        ("l2norm_equals_prenormalised", pins.test_l2norm_equals_prenormalised),
        ("raw_gate_equals_g_form", pins.test_raw_gate_equals_g_form),
        ("fragment_M_product_g", lambda: pins.test_fragment_M_is_transition_product(False)),
        ("fragment_M_product_raw", lambda: pins.test_fragment_M_is_transition_product(True)),
        ("fragment_affine_map_and_walk", pins.test_fragment_affine_map_and_walk),
        ("fragment_backward_walk", pins.test_fragment_backward_walk),
    ]
    for case in pins.FD_CASES:
        out.append((f"finite_differences_{case}",
                    lambda case=case: pins.test_gradients_finite_differences(case)))
    return out


def _first_failing_pin(lib_path):
    with oracle.using_build(lib_path):
        for name, fn in _pins():
            try:
                fn()
            except (AssertionError, RuntimeError, FloatingPointError, ValueError):
                return name
    return None


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_unmodified_build_passes_every_pin(workdir):
    lib = oracle.compile_source(SRC, os.path.join(workdir, "clean.so"))
    assert _first_failing_pin(lib) is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(workdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"the line of mutant '{name}' is not unique in the oracle"
    path = os.path.join(workdir, "".join(ch if ch.isalnum() else "_" for ch in name) + ".c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, path[:-2] + ".so")
    assert _first_failing_pin(lib) is not None, f"no pin catches the planted mistake '{name}'"
