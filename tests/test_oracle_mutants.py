"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle (the C recurrence is
edited as text and compiled to a temporary library; the numpy chunked form is
patched in memory), then checks that at least one pin fails.  Nothing here
touches a GPU.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_CHECKS, recurrence_fn

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

# (name, text in the C source, replacement) -- one planted mistake each
C_MUTANTS = [
    ("no_decay", "row[n] = decay * row[n] + u * (double)bt[n];", "row[n] = row[n] + u * (double)bt[n];"),
    ("decay_sign", "exp(dt_t * a_h)", "exp(-dt_t * a_h)"),
    ("decay_without_dt", "exp(dt_t * a_h)", "exp(a_h)"),
    ("input_without_dt", "const double u = dt_t * (double)xt[p];", "const double u = (double)xt[p];"),
    ("exclusive_state", "row[n] = decay * row[n] + u * (double)bt[n];\n                    acc += row[n] * (double)ct[n];",
     "acc += row[n] * (double)ct[n];\n                    row[n] = decay * row[n] + u * (double)bt[n];"),
    ("b_c_swapped", "row[n] = decay * row[n] + u * (double)bt[n];\n                    acc += row[n] * (double)ct[n];",
     "row[n] = decay * row[n] + u * (double)ct[n];\n                    acc += row[n] * (double)bt[n];"),
    ("no_skip", "yt[p] = acc + d_h * (double)xt[p];", "yt[p] = acc;"),
    ("skip_with_dt", "yt[p] = acc + d_h * (double)xt[p];", "yt[p] = acc + d_h * u;"),
    ("group_modulo", "const int64_t g = h / heads_per_group;", "const int64_t g = h % G;"),
    ("init_ignored", "state[i] = init_state ? (double)init_state[((b * H + h) * P) * N + i] : 0.0;", "state[i] = 0.0;"),
    ("x_index_transposed", "const float* xt = x + ((b * L + t) * H + h) * P;", "const float* xt = x + ((b * L + t) * H + (H - 1 - h)) * P;"),
    ("final_decayed_once_more", "memcpy(final_state + ((b * H + h) * P) * N, state, (size_t)(P * N) * sizeof(double));",
     "for (int64_t i = 0; i < P * N; ++i) final_state[((b * H + h) * P) * N + i] = state[i] * exp(a_h * 0.01);"),
]


def _compile_mutant(tmp, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path_c = os.path.join(tmp, f"{name}.c")
    path_so = os.path.join(tmp, f"lib{name}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", path_c, "-o", path_so, "-lm"], check=True)
    return oracle.load_library(path_so)


@pytest.fixture(scope="module")
def tmpdir_mod():
    d = tempfile.mkdtemp(prefix="ssd_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_c_mutant_is_caught(tmpdir_mod, name, old, new):
    lib = _compile_mutant(tmpdir_mod, name, old, new)
    rec = recurrence_fn(lib)
    failed = [k for k, chk in ALL_CHECKS.items() if not chk(rec)]
    assert failed, f"planted mistake {name} passed every pin"


def _exclusive_cumsum(orig):
    def f(dt, A, Q):
        G = orig(dt, A, Q)
        a = G - np.concatenate([np.zeros_like(G[..., :1]), G[..., :-1]], axis=-1)
        return G - a
    return f


PY_MUTANTS = {
    # cumsum that excludes the current token
    "exclusive_cumsum": ("chunk_cumsum", _exclusive_cumsum),
    # state passing that forgets the chunk decay
    "passing_without_decay": ("state_passing", lambda orig: (
        lambda S, G, init: orig(S, np.zeros_like(G), init))),
    # carried-state term dropped from compute_out
    "no_carried_term": ("compute_out", lambda orig: (
        lambda x, dt, Bm, Cm, D, G, hprev, Q: orig(x, dt, Bm, Cm, D, G, np.zeros_like(hprev), Q))),
    # chunk state without dt
    "state_without_dt": ("chunk_state", lambda orig: (
        lambda x, dt, Bm, G, Q: orig(x, np.ones_like(dt), Bm, G, Q))),
    # causal mask that also drops the diagonal (strictly lower triangle)
    "strict_mask": ("compute_out", lambda orig: (
        lambda x, dt, Bm, Cm, D, G, hprev, Q: orig(x, dt, Bm, Cm, D, G, hprev, Q)
        - _diag_term(x, dt, Bm, Cm, G, Q))),
}


def _diag_term(x, dt, Bm, Cm, G, Q):
    H = x.shape[2]
    r = H // Bm.shape[2]
    bh = np.repeat(Bm, r, axis=2).astype(np.float64)
    ch = np.repeat(Cm, r, axis=2).astype(np.float64)
    return dt.astype(np.float64)[..., None] * np.sum(bh * ch, axis=-1)[..., None] * x


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_chunked_mutant_is_caught(monkeypatch, name):
    attr, make = PY_MUTANTS[name]
    monkeypatch.setattr(oracle, attr, make(getattr(oracle, attr)))

    def rec(inp):
        return oracle.chunked(inp, 4)
    failed = [k for k in ("geometric_series", "single_token", "golden_decay_half", "golden_dt_scaling",
                          "golden_jump_no_decay", "jump_formula_integers") if not ALL_CHECKS[k](rec)]
    inp = _sample()
    y, f, _ = oracle.recurrence(inp)
    yc, fc = rec(inp)
    disagrees = not (np.allclose(y, yc, rtol=1e-10, atol=1e-12) and np.allclose(f, fc, rtol=1e-10, atol=1e-12))
    assert failed or disagrees, f"planted mistake {name} passed every pin"


def _sample():
    from oracle_pins import tiny_inputs
    return tiny_inputs(seed=21, dt_scale=8.0)
