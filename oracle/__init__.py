"""fp64 CPU oracle for the Mamba-2 chunked SSD forward pass.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers.  Nothing
here is imported by, or imports, the CUDA package; the two share no code.

Three formulations, all in fp64, all from the SSD-forward write-up ("Jane
Street ML Engineers Map Mamba-2 Recurrent State Computation to Tensor Cores
with cuTile" and its two companion summaries):

* ``recurrence`` (O-a, in C with OpenMP): the definition -- the token-by-token
  state-space recurrence h_t = exp(dt_t A) h_{t-1} + dt_t x_t b_t^T,
  y_t = h_t c_t + D x_t (page 1, paragraphs on the RNN-like fixed-size state
  and on the jump formula).  This is the parity reference.
* ``chunked`` (O-b, numpy): the chunked closed form the write-up derives,
  one function per step of its kernel decomposition (page 1, "three-kernel
  decomposition" paragraph; page 3, per-kernel roles): ``chunk_cumsum``,
  ``chunk_state``, ``state_passing``, ``compute_out``.  Used to validate the
  oracle and as the per-kernel reference.
* ``quadratic`` (O-c, numpy, tiny inputs only): the whole sequence as one
  causally masked, decayed interaction matrix (page 1, compute_out paragraph,
  with the chunk as long as the sequence).

Readings where the pages are silent are listed in the module docstrings of the
step functions.  Pins that tie these functions to facts outside themselves
live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB = os.path.join(_HERE, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C recurrence into oracle/libssd_oracle.so (gcc, OpenMP, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def load_library(path: str):
    """Open a compiled recurrence library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64, f32p, f64p = ctypes.c_int64, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    lib.ssd_oracle_recurrence.restype = ctypes.c_int
    lib.ssd_oracle_recurrence.argtypes = [i64] * 6 + [f32p] * 7 + [f64p, f64p,
                                         ctypes.POINTER(ctypes.c_int64), i64, ctypes.c_int]
    lib.ssd_oracle_threads.restype = ctypes.c_int
    lib.ssd_oracle_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct)) if a is not None else None


def recurrence(inp: Dict[str, np.ndarray], pairs: Optional[np.ndarray] = None,
               threads: int = 0, lib=None) -> Tuple[np.ndarray, np.ndarray, int]:
    """O-a: the token-by-token recurrence in fp64 (C, OpenMP over (b, h)).

    ``inp`` holds x[B,L,H,P], dt[B,L,H], A[H], Bm/Cm[B,L,G,N], D[H] and
    optionally init[B,H,P,N] (fp32 values).  ``pairs`` is an optional int64
    array of shape [k, 2] of (b, h) pairs to compute; the other entries of y
    and final_state stay NaN.  Returns (y fp64 [B,L,H,P], final fp64
    [B,H,P,N], threads used).  ``lib`` selects another compiled copy of the
    recurrence (the tests use this to plant mistakes); default: this one.
    """
    lib = lib if lib is not None else _load()
    x, dt, A, Bm, Cm, D = (_f32(inp[k]) for k in ("x", "dt", "A", "Bm", "Cm", "D"))
    init = inp.get("init")
    init = _f32(init) if init is not None else None
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    y = np.full((B, L, H, P), np.nan)
    fin = np.full((B, H, P, N), np.nan)
    pr = None
    npairs = 0
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
        npairs = pr.shape[0]
    used = lib.ssd_oracle_recurrence(B, L, H, P, G, N,
                                     _ptr(x, ctypes.c_float), _ptr(dt, ctypes.c_float),
                                     _ptr(A, ctypes.c_float), _ptr(Bm, ctypes.c_float),
                                     _ptr(Cm, ctypes.c_float), _ptr(D, ctypes.c_float),
                                     _ptr(init, ctypes.c_float),
                                     _ptr(y, ctypes.c_double), _ptr(fin, ctypes.c_double),
                                     _ptr(pr, ctypes.c_int64), npairs, int(threads))
    if used < 0:
        raise ValueError("oracle recurrence rejected its arguments")
    return y, fin, used


def threads_available(requested: int = 0) -> int:
    return _load().ssd_oracle_threads(int(requested))


# --------------------------------------------------------------------------
# O-b: the chunked closed form, one function per kernel of the decomposition
# --------------------------------------------------------------------------

def _pad_tokens(a: np.ndarray, Lp: int, axis: int = 1) -> np.ndarray:
    L = a.shape[axis]
    if Lp == L:
        return a
    pad = [(0, 0)] * a.ndim
    pad[axis] = (0, Lp - L)
    return np.pad(a, pad)


def chunk_cumsum(dt: np.ndarray, A: np.ndarray, Q: int) -> np.ndarray:
    """Log-space decay cumsum within each chunk (page 1, three-kernel paragraph:
    per-token, per-head cumulative sums of the decay term, restarted per chunk).

    a_t = dt_t * A_h; G[b,h,c,i] = sum_{k <= i} a_{cQ+k} (inclusive).  Tokens
    past the sequence end (ragged last chunk) get a = 0, so G stays flat there.
    Returns G as fp64 [B, H, nc, Q] in the transposed head-major layout the
    write-up asks for (page 1, Blackwell paragraph: [batch, head, token]).
    """
    B, L, H = dt.shape
    nc = -(-L // Q)
    a = dt.astype(np.float64) * A.astype(np.float64)[None, None, :]
    a = _pad_tokens(a, nc * Q).transpose(0, 2, 1).reshape(B, H, nc, Q)
    return np.cumsum(a, axis=-1)


def _heads_view(Bm: np.ndarray, H: int) -> np.ndarray:
    """[B, L, G, N] -> [B, L, H, N]: head h reads group h // (H // G)."""
    G = Bm.shape[2]
    return np.repeat(Bm, H // G, axis=2)


def chunk_state(x: np.ndarray, dt: np.ndarray, Bm: np.ndarray, Gcs: np.ndarray, Q: int) -> np.ndarray:
    """Each chunk's state contribution from a zero start: the jump formula with
    decay (page 1, jump-formula paragraph: h(t+T) = h(t) + B X^T without decay;
    with decay the b rows are pre-multiplied by exponentials of log-space sums).

    S[b,c,h,p,n] = sum_j exp(Ghat_c - G_j) * dt_j * x_j[p] * b_j[n],
    Ghat_c = G at the chunk's last position.  fp64 [B, nc, H, P, N].
    """
    B, L, H, P = x.shape
    nc = Gcs.shape[2]
    Lp = nc * Q
    xs = _pad_tokens(x.astype(np.float64), Lp).reshape(B, nc, Q, H, P)
    dts = _pad_tokens(dt.astype(np.float64), Lp).reshape(B, nc, Q, H)
    bs = _pad_tokens(_heads_view(Bm, H).astype(np.float64), Lp).reshape(B, nc, Q, H, -1)
    w = np.exp(Gcs[..., -1:] - Gcs)                      # [B,H,nc,Q], exponents <= 0
    w = w * dts.transpose(0, 3, 1, 2)                     # times dt_j
    return np.einsum("bhcj,bcjhp,bcjhn->bchpn", w, xs, bs, optimize=True)


def state_passing(S: np.ndarray, Gcs: np.ndarray, init: Optional[np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
    """Sequential pass over chunks with the decayed jump formula
    h_c = exp(Ghat_c) h_{c-1} + S_c (page 1, fwd_pass_state: a sequential loop
    over chunks that advances the hidden state).

    Returns (hprev [B, nc, H, P, N]: the state entering each chunk,
    final [B, H, P, N]: the state after the last chunk).
    """
    B, nc, H, P, N = S.shape
    h = np.zeros((B, H, P, N)) if init is None else init.astype(np.float64).copy()
    hprev = np.empty_like(S)
    for c in range(nc):
        hprev[:, c] = h
        h = np.exp(Gcs[:, :, c, -1])[:, :, None, None] * h + S[:, c]
    return hprev, h


def compute_out(x: np.ndarray, dt: np.ndarray, Bm: np.ndarray, Cm: np.ndarray, D: np.ndarray,
                Gcs: np.ndarray, hprev: np.ndarray, Q: int) -> np.ndarray:
    """Output of every chunk as the sum of three terms (page 1, compute_out
    paragraph): the carried-state term exp(G_i) C_i hprev^T, the decayed and
    causally masked interaction matrix (C B^T) o exp(G - G^T) times dt-scaled
    X, and the skip connection D x.  Masked positions (j > i) are selected to
    zero, never multiplied (the write-up zeroes the positive exponents).

    Returns y fp64 [B, L, H, P].
    """
    B, L, H, P = x.shape
    nc = Gcs.shape[2]
    Lp = nc * Q
    xs = _pad_tokens(x.astype(np.float64), Lp).reshape(B, nc, Q, H, P)
    dts = _pad_tokens(dt.astype(np.float64), Lp).reshape(B, nc, Q, H)
    bs = _pad_tokens(_heads_view(Bm, H).astype(np.float64), Lp).reshape(B, nc, Q, H, -1)
    cs = _pad_tokens(_heads_view(Cm, H).astype(np.float64), Lp).reshape(B, nc, Q, H, -1)
    G = Gcs.transpose(0, 2, 3, 1)                         # [B, nc, Q, H]
    y = np.empty((B, nc, Q, H, P))
    causal = np.tril(np.ones((Q, Q), dtype=bool))
    for c in range(nc):
        # carried-state term
        carried = np.einsum("bih,bihn,bhpn->bihp", np.exp(G[:, c]), cs[:, c], hprev[:, c], optimize=True)
        # interaction matrix C B^T per head, decay exp(G_i - G_j) on the causal part only
        cb = np.einsum("bihn,bjhn->bhij", cs[:, c], bs[:, c], optimize=True)
        Gh = G[:, c].transpose(0, 2, 1)                   # [B, H, Q]
        seg = Gh[:, :, :, None] - Gh[:, :, None, :]       # G_i - G_j
        decay = np.where(causal, np.exp(np.where(causal, seg, 0.0)), 0.0)
        m = cb * decay * dts[:, c].transpose(0, 2, 1)[:, :, None, :]
        intra = np.einsum("bhij,bjhp->bihp", m, xs[:, c], optimize=True)
        y[:, c] = carried + intra + D.astype(np.float64)[None, None, :, None] * xs[:, c]
    return y.reshape(B, Lp, H, P)[:, :L]


def chunked(inp: Dict[str, np.ndarray], Q: int) -> Tuple[np.ndarray, np.ndarray]:
    """O-b end to end: chunk_cumsum -> chunk_state -> state_passing -> compute_out."""
    Gcs = chunk_cumsum(inp["dt"], inp["A"], Q)
    S = chunk_state(inp["x"], inp["dt"], inp["Bm"], Gcs, Q)
    hprev, fin = state_passing(S, Gcs, inp.get("init"))
    y = compute_out(inp["x"], inp["dt"], inp["Bm"], inp["Cm"], inp["D"], Gcs, hprev, Q)
    return y, fin


# --------------------------------------------------------------------------
# O-c: the quadratic (fully materialised) form, tiny inputs only
# --------------------------------------------------------------------------

def quadratic(inp: Dict[str, np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
    """The whole sequence as one masked interaction matrix, with explicit
    segment sums (no cumsum differences):

    y_t = sum_{s <= t} (c_t . b_s) exp(sum_{k=s+1}^{t} a_k) dt_s x_s
          + exp(sum_{k=0}^{t} a_k) h_0 c_t + D x_t
    final = exp(sum_k a_k) h_0 + sum_s exp(sum_{k=s+1}^{L-1} a_k) dt_s x_s b_s^T
    """
    x = inp["x"].astype(np.float64)
    dt = inp["dt"].astype(np.float64)
    A = inp["A"].astype(np.float64)
    B, L, H, P = x.shape
    bs = _heads_view(inp["Bm"], H).astype(np.float64)
    cs = _heads_view(inp["Cm"], H).astype(np.float64)
    N = bs.shape[-1]
    h0 = inp.get("init")
    h0 = np.zeros((B, H, P, N)) if h0 is None else h0.astype(np.float64)
    a = dt * A[None, None, :]                              # [B, L, H]
    y = np.zeros((B, L, H, P))
    fin = np.zeros((B, H, P, N))
    for b in range(B):
        for h in range(H):
            for t in range(L):
                acc = np.zeros(P)
                for s in range(t + 1):
                    seg = sum(a[b, k, h] for k in range(s + 1, t + 1))
                    acc += (cs[b, t, h] @ bs[b, s, h]) * np.exp(seg) * dt[b, s, h] * x[b, s, h]
                seg0 = sum(a[b, k, h] for k in range(0, t + 1))
                acc += np.exp(seg0) * (h0[b, h] @ cs[b, t, h])
                y[b, t, h] = acc + float(inp["D"][h]) * x[b, t, h]
            tot = sum(a[b, k, h] for k in range(L))
            st = np.exp(tot) * h0[b, h]
            for s in range(L):
                seg = sum(a[b, k, h] for k in range(s + 1, L))
                st = st + np.exp(seg) * dt[b, s, h] * np.outer(x[b, s, h], bs[b, s, h])
            fin[b, h] = st
    return y, fin
