"""Seeded synthetic inputs for the Mamba-2 chunked SSD forward pass.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the method's arithmetic (no decay, no cumsum, no state), so
both the fp64 oracle and the CUDA path can take their inputs from it without
sharing any computation.

Random numbers come from a counter-based generator written out here from its
published definition: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), finalizer constants as
published.  Value ``i`` of stream ``k`` is ``mix(key_k + (i + 1) * GAMMA)``,
so any element can be regenerated on its own.  Uniforms take the top 53 bits;
normals use the Box-Muller transform on consecutive uniform pairs.

Value recipe (Mamba-2 layer shapes: the ~370M and ~2.7B layers, a long
sequence with a large state, and a 65,536-token shape sweep; see WORKLOADS):

* x ~ N(0, 1)
* Bm, Cm ~ N(0, 1) / sqrt(N)
* dt = clip(softplus(z - 4.6), 1e-3, 0.1), z ~ N(0, 1)   (post-activation dt)
* A_h = -exp(U(log 1, log 16))
* D ~ N(0, 1)
* init_state ~ N(0, 0.1^2) where the workload asks for one, else absent

Tensors are drawn in the order x, dt, A, Bm, Cm, D, init, each from its own
stream.  Everything is generated in fp32; for bf16 workloads x, Bm and Cm are
then rounded to bf16 (round-to-nearest-even) and kept as the fp32 values of
those bf16 numbers, so that the oracle and the GPU see identical inputs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_SALT = np.uint64(0xD1B54A32D192ED03)

STREAM_IDS = {"x": 1, "dt": 2, "A": 3, "Bm": 4, "Cm": 5, "D": 6, "init": 7}


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finalizer on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed & 0xFFFFFFFFFFFFFFFF)], dtype=np.uint64)
        s = s ^ (np.uint64(stream) * _STREAM_SALT)
    return _mix64(s)[0]


def uniform01(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` uniforms in (0, 1) as float64: values offset..offset+count-1 of a stream."""
    key = _stream_key(seed, stream)
    with np.errstate(over="ignore"):
        ctr = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
        z = _mix64(key + ctr * _GAMMA)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def _box_muller(u: np.ndarray) -> np.ndarray:
    """Normals from consecutive uniform pairs (u1, u2): sqrt(-2 ln u1) times cos / sin of 2 pi u2."""
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(u.shape[0], dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * math.pi * u2)
    out[1::2] = r * np.sin(2.0 * math.pi * u2)
    return out


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` standard normals (float64) by Box-Muller on uniform pairs."""
    npairs = (count + 1) // 2
    return _box_muller(uniform01(seed, stream, 2 * npairs))[:count]


_CHUNK_PAIRS = 1 << 20


def normal_f32(seed: int, stream: int, count: int, scale: float = 1.0, bf16: bool = False) -> np.ndarray:
    """``(normal(seed, stream, count) * scale)`` as float32 (rounded on to bf16
    values when ``bf16``), computed in independent slices of the stream on a
    few threads.  Element i depends only on i (the generator is counter-based
    and each Box-Muller pair is whole inside a slice), so this is the same
    function of the index as ``normal``; the slices only keep large tensors
    fast to draw."""
    import concurrent.futures as cf
    out = np.empty(count, dtype=np.float32)
    npairs = (count + 1) // 2

    def fill(p0: int) -> None:
        p1 = min(npairs, p0 + _CHUNK_PAIRS)
        v = _box_muller(uniform01(seed, stream, 2 * (p1 - p0), offset=2 * p0))
        if scale != 1.0:
            v *= scale
        lo, hi = 2 * p0, min(count, 2 * p1)
        f = v[: hi - lo].astype(np.float32)
        out[lo:hi] = round_to_bf16(f) if bf16 else f

    starts = range(0, npairs, _CHUNK_PAIRS)
    if npairs <= _CHUNK_PAIRS:
        for p0 in starts:
            fill(p0)
    else:
        import os
        with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, starts))
    return out


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); return them as fp32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    bias = ((bits >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    rounded = ((bits + bias) >> np.uint64(16)) << np.uint64(16)
    return rounded.astype(np.uint32).view(np.float32).reshape(a.shape)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One SSD-forward problem: shape, storage dtype and value recipe."""

    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int
    dtype: str  # "f32" (TF32 tensor-core math) or "bf16"
    init_state: bool = False
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _sweep() -> Dict[str, Workload]:
    out = {}
    for L in (512, 2048, 8192, 32768):
        for N in (64, 128, 256):
            for Q in (128, 256):
                name = f"sweep-L{L}-N{N}-Q{Q}"
                out[name] = Workload(name, 65536 // L, L, 64, 64, N, 8, Q, "bf16")
    return out


WORKLOADS: Dict[str, Workload] = {
    # tiny fp32 case the oracle finishes in well under a second
    "tiny": Workload("tiny", 1, 256, 4, 64, 64, 1, 64, "f32"),
    # Mamba-2 ~370M layer shape (d_model 1024, expand 2)
    "mamba2-370m": Workload("mamba2-370m", 2, 2048, 32, 64, 128, 1, 256, "f32"),
    # Mamba-2 ~2.7B layer shape (d_model 2560), bf16, random initial state
    "mamba2-2.7b": Workload("mamba2-2.7b", 4, 4096, 80, 64, 128, 1, 256, "bf16", init_state=True),
    # long sequence, large state
    "long-16k-n256": Workload("long-16k-n256", 1, 16384, 32, 64, 256, 1, 256, "f32"),
    **_sweep(),
}


def make_inputs(w: Workload, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Draw the inputs of workload ``w`` (all numpy float32, C-contiguous).

    Returns x[B,L,H,P], dt[B,L,H], A[H], Bm[B,L,G,N], Cm[B,L,G,N], D[H] and,
    when ``w.init_state``, init[B,H,P,N].  For bf16 workloads x, Bm and Cm hold
    bf16-representable values.
    """
    s = w.seed if seed is None else seed
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    if w.dtype not in ("bf16", "f32"):
        raise ValueError(f"unknown dtype {w.dtype!r}")
    low = w.dtype == "bf16"  # x, Bm and Cm stored as bf16 values
    out: Dict[str, np.ndarray] = {}
    out["x"] = normal_f32(s, STREAM_IDS["x"], B * L * H * P, bf16=low).reshape(B, L, H, P)
    z = normal(s, STREAM_IDS["dt"], B * L * H)
    v = z - 4.6
    softplus = np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))
    out["dt"] = np.clip(softplus, 1e-3, 0.1).astype(np.float32).reshape(B, L, H)
    u = uniform01(s, STREAM_IDS["A"], H)
    out["A"] = (-np.exp(u * math.log(16.0))).astype(np.float32)
    scale = 1.0 / math.sqrt(N)
    out["Bm"] = normal_f32(s, STREAM_IDS["Bm"], B * L * G * N, scale, bf16=low).reshape(B, L, G, N)
    out["Cm"] = normal_f32(s, STREAM_IDS["Cm"], B * L * G * N, scale, bf16=low).reshape(B, L, G, N)
    out["D"] = normal(s, STREAM_IDS["D"], H).astype(np.float32)
    if w.init_state:
        out["init"] = normal_f32(s, STREAM_IDS["init"], B * H * P * N, 0.1).reshape(B, H, P, N)
    return out


def custom(name: str = "custom", **kw) -> Workload:
    """A workload with explicit sizes (defaults: the tiny fp32 case)."""
    base = dataclasses.asdict(WORKLOADS["tiny"])
    base.update(kw)
    base["name"] = name
    return Workload(**base)
