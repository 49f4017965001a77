"""The oracle against facts it does not compute itself (no GPU needed).

Each pin cites what fixes it: a worked example derived from a statement on the
pages (tests/golden), a closed form, an invariant of the recurrence, or agreement
between independently written formulations on tiny inputs.
"""
import numpy as np
import pytest

import oracle
import ssd_synth
from oracle_pins import ALL_CHECKS, recurrence_fn, rel_err, tiny_inputs

pytestmark = pytest.mark.timeout(120) if hasattr(pytest.mark, "timeout") else []


@pytest.mark.parametrize("name", sorted(ALL_CHECKS))
def test_pin_recurrence(name):
    assert ALL_CHECKS[name](recurrence_fn())


@pytest.mark.parametrize("name", ["golden_jump_no_decay", "golden_decay_half", "golden_dt_scaling",
                                  "jump_formula_integers", "geometric_series", "single_token",
                                  "causality", "group_map", "extreme_decay", "bidiagonal_solve"])
@pytest.mark.parametrize("Q", [1, 2, 5, 64])
def test_pin_chunked_form(name, Q):
    """The chunked form (the per-kernel reference) passes the same pins."""
    def rec(inp):
        return oracle.chunked(inp, Q)
    assert ALL_CHECKS[name](rec)


def test_chunk_size_invariance_large():
    """y and the final state do not depend on the chunk size (mathematically
    exact; differences are fp64 rounding only)."""
    w = ssd_synth.WORKLOADS["tiny"].with_(seqlen=200, init_state=True)
    inp = ssd_synth.make_inputs(w)
    y64, f64 = oracle.chunked(inp, 64)
    for Q in (16, 128, 256):
        y, f = oracle.chunked(inp, Q)
        assert rel_err(y, y64) < 1e-12 and rel_err(f, f64) < 1e-12


def test_recurrence_vs_chunked_tiny_workload():
    w = ssd_synth.WORKLOADS["tiny"]
    inp = ssd_synth.make_inputs(w)
    y, f, _ = oracle.recurrence(inp)
    yc, fc = oracle.chunked(inp, w.chunk_size)
    assert rel_err(y, yc) < 1e-12 and rel_err(f, fc) < 1e-12


def test_pair_sampling_matches_full():
    inp = tiny_inputs(B=2, L=20, H=4, P=3, N=5, G=2, seed=12)
    y, f, _ = oracle.recurrence(inp)
    pairs = np.array([[1, 2], [0, 3]])
    ys, fs, _ = oracle.recurrence(inp, pairs=pairs)
    for b, h in pairs:
        assert np.array_equal(ys[b, :, h], y[b, :, h]) and np.array_equal(fs[b, h], f[b, h])
    assert np.isnan(ys[0, :, 0]).all()


def test_step_functions_shapes_and_ragged_tail():
    """Ragged last chunk: padded tokens carry no decay and no input."""
    inp = tiny_inputs(B=1, L=11, H=2, P=2, N=3, G=1, seed=13)
    Q = 4
    G = oracle.chunk_cumsum(inp["dt"], inp["A"], Q)
    assert G.shape == (1, 2, 3, 4)
    # tokens 11 (pad) keep the cumsum flat
    assert G[0, 0, 2, 3] == G[0, 0, 2, 2]
    S = oracle.chunk_state(inp["x"], inp["dt"], inp["Bm"], G, Q)
    hprev, fin = oracle.state_passing(S, G, inp["init"])
    assert np.array_equal(hprev[:, 0], inp["init"].astype(np.float64))
    y, f, _ = oracle.recurrence(inp)
    assert rel_err(fin, f) < 1e-12
