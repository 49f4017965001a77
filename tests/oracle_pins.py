"""Pins for the fp64 oracle: facts from the pages and from mathematics that a
plausible mistake in the oracle would violate.  Each check takes the recurrence
as a callable so that ``test_oracle_mutants.py`` can run the same checks on
copies of the oracle with planted mistakes.

A recurrence callable maps an input dict to (y fp64, final fp64).
"""
from __future__ import annotations

import math
import os
from typing import Callable, Dict, Tuple

import numpy as np

import oracle
import ssd_synth

Rec = Callable[[Dict[str, np.ndarray]], Tuple[np.ndarray, np.ndarray]]
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rel_err(a: np.ndarray, b: np.ndarray) -> float:
    scale = max(float(np.max(np.abs(b))), 1e-300)
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) / scale


def tiny_inputs(B=2, L=13, H=4, P=3, N=5, G=2, init=True, seed=11, dt_scale=1.0) -> Dict[str, np.ndarray]:
    """Small random inputs with the workload value distributions."""
    w = ssd_synth.custom("pin", batch=B, seqlen=L, nheads=H, headdim=P, dstate=N, ngroups=G,
                         chunk_size=4, dtype="f32", init_state=init, seed=seed)
    inp = ssd_synth.make_inputs(w)
    if dt_scale != 1.0:
        inp["dt"] = (inp["dt"] * dt_scale).astype(np.float32)
    return inp


def load_golden(name: str):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = [float(t) for t in v.split()]
    B, L, H, P, N, G = (int(t) for t in vals["shape"])
    inp = {
        "x": np.array(vals["x"], np.float32).reshape(B, L, H, P),
        "dt": np.array(vals["dt"], np.float32).reshape(B, L, H),
        "A": np.array(vals["A"], np.float32).reshape(H),
        "Bm": np.array(vals["Bm"], np.float32).reshape(B, L, G, N),
        "Cm": np.array(vals["Cm"], np.float32).reshape(B, L, G, N),
        "D": np.array(vals["D"], np.float32).reshape(H),
        "init": np.array(vals["init"], np.float32).reshape(B, H, P, N),
    }
    y = np.array(vals["y"]).reshape(B, L, H, P)
    fin = np.array(vals["final"]).reshape(B, H, P, N)
    return inp, y, fin, vals["tol"][0]


# ---------------------------------------------------------------- the checks

def check_golden(rec: Rec, name: str) -> bool:
    inp, y_ref, f_ref, tol = load_golden(name)
    y, f = rec(inp)
    ok_y = np.allclose(y, y_ref, rtol=tol, atol=tol * np.max(np.abs(y_ref)))
    ok_f = np.allclose(f, f_ref, rtol=tol, atol=tol * np.max(np.abs(f_ref)))
    return bool(ok_y and ok_f)


def check_formulations_agree(rec: Rec, seed=11, tol=1e-12) -> bool:
    """Recurrence = quadratic form = chunked form for several chunk sizes."""
    inp = tiny_inputs(seed=seed, dt_scale=8.0)  # larger dt: decay matters within a few tokens
    y, f = rec(inp)
    yq, fq = oracle.quadratic(inp)
    ok = rel_err(y, yq) < tol and rel_err(f, fq) < tol
    for Q in (1, 3, 4, 16, inp["x"].shape[1]):
        yc, fc = oracle.chunked(inp, Q)
        ok = ok and rel_err(y, yc) < tol and rel_err(f, fc) < tol
    return bool(ok)


def check_jump_formula_integers(rec: Rec) -> bool:
    """A = 0, dt = 1, small integers: h_T = h_0 + sum_t x_t b_t^T and
    y_t = (h_0 + sum_{s<=t} x_s b_s^T) c_t + D x_t, exactly (jump formula)."""
    rng = np.random.default_rng(5)
    B, L, H, P, N, G = 2, 9, 4, 3, 5, 2
    inp = {
        "x": rng.integers(-3, 4, (B, L, H, P)).astype(np.float32),
        "dt": np.ones((B, L, H), np.float32),
        "A": np.zeros(H, np.float32),
        "Bm": rng.integers(-3, 4, (B, L, G, N)).astype(np.float32),
        "Cm": rng.integers(-3, 4, (B, L, G, N)).astype(np.float32),
        "D": rng.integers(-2, 3, H).astype(np.float32),
        "init": rng.integers(-3, 4, (B, H, P, N)).astype(np.float32),
    }
    y, f = rec(inp)
    r = H // G
    ok = True
    for b in range(B):
        for h in range(H):
            g = h // r
            st = inp["init"][b, h].astype(np.int64)
            for t in range(L):
                st = st + np.outer(inp["x"][b, t, h], inp["Bm"][b, t, g]).astype(np.int64)
                yt = st @ inp["Cm"][b, t, g].astype(np.int64) + inp["D"][h] * inp["x"][b, t, h]
                ok = ok and np.array_equal(y[b, t, h], yt)
            ok = ok and np.array_equal(f[b, h], st)
    return bool(ok)


def check_geometric_series(rec: Rec) -> bool:
    """P = N = 1 with constant a = dt*A, x, b, c: the state is a geometric sum,
    h_t = dt x b (1 - e^{a(t+1)}) / (1 - e^a) + e^{a(t+1)} h_0."""
    L = 40
    dt, A, x, b, c, D, h0 = 0.05, -3.0, 1.5, 0.75, -2.0, 0.25, 0.5
    inp = {
        "x": np.full((1, L, 1, 1), x, np.float32), "dt": np.full((1, L, 1), dt, np.float32),
        "A": np.array([A], np.float32), "Bm": np.full((1, L, 1, 1), b, np.float32),
        "Cm": np.full((1, L, 1, 1), c, np.float32), "D": np.array([D], np.float32),
        "init": np.full((1, 1, 1, 1), h0, np.float32),
    }
    dt = float(np.float32(dt))  # the value the recurrence actually receives
    a = dt * float(np.float32(A))
    t = np.arange(L)
    h = dt * x * b * (1 - np.exp(a * (t + 1))) / (1 - math.exp(a)) + np.exp(a * (t + 1)) * h0
    y_ref = h * c + D * x
    y, f = rec(inp)
    return bool(rel_err(y[0, :, 0, 0], y_ref) < 1e-12 and abs(f[0, 0, 0, 0] - h[-1]) < 1e-12)


def check_single_token(rec: Rec) -> bool:
    """L = 1: y = dt x (b.c) + e^{dt A} h_0 c + D x;  final = e^{dt A} h_0 + dt x b^T."""
    inp = tiny_inputs(B=2, L=1, H=4, P=3, N=5, G=2, seed=3)
    y, f = rec(inp)
    ok = True
    for b in range(2):
        for h in range(4):
            g = h // 2
            dt = float(inp["dt"][b, 0, h]); e = math.exp(dt * float(inp["A"][h]))
            x = inp["x"][b, 0, h].astype(np.float64)
            bb = inp["Bm"][b, 0, g].astype(np.float64); cc = inp["Cm"][b, 0, g].astype(np.float64)
            h0 = inp["init"][b, h].astype(np.float64)
            y_ref = dt * x * (bb @ cc) + e * (h0 @ cc) + float(inp["D"][h]) * x
            f_ref = e * h0 + dt * np.outer(x, bb)
            ok = ok and rel_err(y[b, 0, h], y_ref) < 1e-13 and rel_err(f[b, h], f_ref) < 1e-13
    return bool(ok)


def check_special_cases(rec: Rec) -> bool:
    """Cm = 0 gives y = D x; total decay (dt*A = -1000, exp underflows to 0)
    gives y_t = dt_t (b_t . c_t) x_t + D x_t and final = dt x b^T of the last token."""
    inp = tiny_inputs(seed=4)
    z = dict(inp); z["Cm"] = np.zeros_like(inp["Cm"])
    y, _ = rec(z)
    ok = np.allclose(y, inp["D"][None, None, :, None].astype(np.float64) * inp["x"], rtol=0, atol=0)
    s = dict(inp); s["A"] = np.full_like(inp["A"], -1e4); s["dt"] = np.full_like(inp["dt"], 0.1)
    y, f = rec(s)
    H = inp["x"].shape[2]; G = inp["Bm"].shape[2]
    bh = np.repeat(inp["Bm"], H // G, axis=2).astype(np.float64)
    ch = np.repeat(inp["Cm"], H // G, axis=2).astype(np.float64)
    dt = float(np.float32(0.1))
    x64 = inp["x"].astype(np.float64)
    y_ref = dt * np.sum(bh * ch, axis=-1)[..., None] * x64 + inp["D"].astype(np.float64)[None, None, :, None] * x64
    f_ref = dt * np.einsum("bhp,bhn->bhpn", inp["x"][:, -1].astype(np.float64), bh[:, -1])
    ok = ok and rel_err(y, y_ref) < 1e-13 and rel_err(f, f_ref) < 1e-13
    return bool(ok)


def check_linearity(rec: Rec) -> bool:
    """With a zero initial state, y and the final state are linear in x
    (integer-valued x, so the combined input is exact in fp32)."""
    inp = tiny_inputs(init=False, seed=6)
    rng = np.random.default_rng(1)
    x1 = rng.integers(-4, 5, inp["x"].shape).astype(np.float32)
    x2 = rng.integers(-4, 5, inp["x"].shape).astype(np.float32)
    a, b = 0.5, -2.0
    i1 = dict(inp); i1["x"] = x1
    i2 = dict(inp); i2["x"] = x2
    i3 = dict(inp); i3["x"] = (a * x1 + b * x2).astype(np.float32)
    y1, f1 = rec(i1); y2, f2 = rec(i2); y3, f3 = rec(i3)
    return bool(rel_err(y3, a * y1 + b * y2) < 1e-12 and rel_err(f3, a * f1 + b * f2) < 1e-12)


def check_causality(rec: Rec) -> bool:
    """Changing tokens after t leaves y[:t+1] unchanged bit for bit."""
    inp = tiny_inputs(seed=7)
    y, _ = rec(inp)
    t = 6
    p = {k: v.copy() for k, v in inp.items()}
    rng = np.random.default_rng(2)
    for k in ("x", "Bm", "Cm"):
        p[k][:, t + 1:] = rng.standard_normal(p[k][:, t + 1:].shape).astype(np.float32)
    p["dt"][:, t + 1:] = 0.05
    y2, _ = rec(p)
    return bool(np.array_equal(y[:, :t + 1], y2[:, :t + 1]) and not np.allclose(y[:, t + 1:], y2[:, t + 1:]))


def check_resume(rec: Rec) -> bool:
    """Running the first L1 tokens and then the rest from the carried final
    state equals one run over the whole sequence."""
    inp = tiny_inputs(L=17, seed=8)
    y, f = rec(inp)
    L1 = 7
    a = {k: (v[:, :L1] if k in ("x", "dt", "Bm", "Cm") else v) for k, v in inp.items()}
    ya, fa = rec(a)
    b = {k: (v[:, L1:] if k in ("x", "dt", "Bm", "Cm") else v) for k, v in inp.items()}
    b["init"] = fa.astype(np.float32)
    # the carried state is rounded to fp32 for the second call; compare loosely
    yb, fb = rec(b)
    return bool(rel_err(np.concatenate([ya, yb], axis=1), y) < 1e-6 and rel_err(fb, f) < 1e-6)


def check_group_map(rec: Rec) -> bool:
    """Head h reads group h // (H / G): zeroing group 1's Cm turns exactly the
    second half of the heads into pure skip connections."""
    inp = tiny_inputs(H=4, G=2, init=False, seed=9)
    z = dict(inp); z["Cm"] = inp["Cm"].copy(); z["Cm"][:, :, 1] = 0
    y, _ = rec(z)
    skip = inp["D"][None, None, :, None].astype(np.float64) * inp["x"]
    return bool(np.array_equal(y[:, :, 2:], skip[:, :, 2:]) and not np.allclose(y[:, :, :2], skip[:, :, :2]))


def check_extreme_decay(rec: Rec) -> bool:
    """A = -16, dt = 0.1 (the most negative decay the workloads draw): all
    outputs finite and equal to the chunked form (whose masked exponents would
    be exp(+400) = inf if they were multiplied instead of selected)."""
    inp = tiny_inputs(L=33, seed=10)
    inp["A"] = np.full_like(inp["A"], -16.0)
    inp["dt"] = np.full_like(inp["dt"], 0.1)
    y, f = rec(inp)
    yc, fc = oracle.chunked(inp, 32)
    return bool(np.all(np.isfinite(y)) and np.all(np.isfinite(f)) and rel_err(y, yc) < 1e-12)


def check_bidiagonal_solve(rec: Rec) -> bool:
    """Time-varying decay: every state entry (b, h, p, n) obeys the first-order
    linear recurrence h_t - alpha_t h_{t-1} = dt_t x_t[p] b_t[n] with
    alpha_t = exp(dt_t A_h), i.e. a lower-bidiagonal linear system in
    (h_0 .. h_{L-1}).  scipy's banded solver gives the states without any loop
    of the oracle's; y_t = h_t c_t + D x_t and the final state follow."""
    from scipy.linalg import solve_banded
    B, L, H, P, N, G = 2, 17, 4, 3, 5, 2
    inp = tiny_inputs(B=B, L=L, H=H, P=P, N=N, G=G, seed=29, dt_scale=4.0)
    x, dt, A = (inp[k].astype(np.float64) for k in ("x", "dt", "A"))
    Bm, Cm, D, h0 = (inp[k].astype(np.float64) for k in ("Bm", "Cm", "D", "init"))
    r = H // G
    y_ref = np.empty((B, L, H, P))
    f_ref = np.empty((B, H, P, N))
    for b in range(B):
        for h in range(H):
            g = h // r
            alpha = np.exp(dt[b, :, h] * A[h])                      # [L]
            ab = np.zeros((2, L))
            ab[0] = 1.0
            ab[1, :L - 1] = -alpha[1:]                               # row t, column t - 1
            rhs = dt[b, :, h, None, None] * x[b, :, h, :, None] * Bm[b, :, g, None, :]   # [L, P, N]
            rhs[0] += alpha[0] * h0[b, h]
            states = solve_banded((1, 0), ab, rhs.reshape(L, P * N)).reshape(L, P, N)
            y_ref[b, :, h] = np.einsum("tpn,tn->tp", states, Cm[b, :, g]) + D[h] * x[b, :, h]
            f_ref[b, h] = states[-1]
    y, f = rec(inp)
    return bool(rel_err(y, y_ref) < 1e-12 and rel_err(f, f_ref) < 1e-12)


ALL_CHECKS = {
    "golden_jump_no_decay": lambda r: check_golden(r, "jump_no_decay.txt"),
    "golden_decay_half": lambda r: check_golden(r, "decay_half.txt"),
    "golden_dt_scaling": lambda r: check_golden(r, "dt_scaling.txt"),
    "formulations_agree": check_formulations_agree,
    "jump_formula_integers": check_jump_formula_integers,
    "geometric_series": check_geometric_series,
    "single_token": check_single_token,
    "special_cases": check_special_cases,
    "linearity": check_linearity,
    "causality": check_causality,
    "resume": check_resume,
    "group_map": check_group_map,
    "extreme_decay": check_extreme_decay,
    "bidiagonal_solve": check_bidiagonal_solve,
}


def recurrence_fn(lib=None) -> Rec:
    def rec(inp):
        y, f, _ = oracle.recurrence(inp, lib=lib)
        return y, f
    return rec
