"""Helpers shared by the GPU tests: move seeded inputs to the device, run the
CUDA path through the binding, and compare with the fp64 oracle using the
tolerances the workloads state (max|out - ref| / max|ref|)."""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

import oracle
import ssd_synth

TOL = {"f32": 5e-3, "bf16": 2e-2}


def rel_err(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(float(np.max(np.abs(b))), 1e-30)
    return float(np.max(np.abs(a - b))) / scale


def to_device(inp: Dict[str, np.ndarray], dtype: str, device="cuda") -> Dict[str, torch.Tensor]:
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = {}
    for k, v in inp.items():
        t = torch.from_numpy(np.ascontiguousarray(v))
        if k in ("x", "Bm", "Cm"):
            t = t.to(tdt)
        out[k] = t.to(device)
    return out


def run_gpu(inp: Dict[str, np.ndarray], dtype: str, Q: int, with_init: Optional[bool] = None,
            schedule: str = "auto"):
    import mamba_ssd_forward_chunked_gb300 as ssd
    d = to_device(inp, dtype)
    init = d.get("init") if (with_init is None or with_init) else None
    y, fin = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], Q, init_state=init, schedule=schedule)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64), fin.cpu().numpy().astype(np.float64)


def run_gpu_schedule(d: Dict[str, torch.Tensor], Q: int, schedule: str):
    """One forward pass on device tensors ``d`` through the C ABI.  schedule:
    "auto" (ssd_fwd picks), "fused" (the one-pass kernel, ssd_fwd_fused) or
    "staged" (the four step entry points in order: the staged schedule for
    any shape).  Returns (y, final_state) on the device."""
    import mamba_ssd_forward_chunked_gb300 as ssd
    init = d.get("init")
    if schedule in ("auto", "fused"):
        return ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], Q, init_state=init,
                           schedule=schedule)
    assert schedule == "staged", schedule
    shape = ssd.shape_of(d["x"], d["Bm"], Q)
    ws = ssd.new_workspace(shape)
    B, L, H, P = d["x"].shape
    y = torch.empty_like(d["x"])
    fin = torch.empty(B, H, P, d["Bm"].shape[3], dtype=torch.float32, device=d["x"].device)
    ssd.ssd_chunk_cumsum(shape, d["dt"], d["A"], ws)
    ssd.ssd_chunk_state(shape, d["x"], d["Bm"], ws)
    ssd.ssd_state_passing(shape, init, fin, ws)
    ssd.ssd_compute_out(shape, d["x"], d["Bm"], d["Cm"], d["D"], y, ws)
    assert ssd.ssd_fwd_check(ws) == 0
    return y, fin


def pair_rows(y: torch.Tensor, fin: torch.Tensor, pairs: np.ndarray):
    """The sampled (b, h) pairs' outputs, gathered on the device: y[b, :, h]
    stacked as [k, L, P] and final_state[b, h] as [k, P, N], in fp64 on the host."""
    bi = torch.as_tensor(pairs[:, 0], device=y.device)
    hi = torch.as_tensor(pairs[:, 1], device=y.device)
    ys = y[bi, :, hi].float().cpu().numpy().astype(np.float64)
    fs = fin[bi, hi].cpu().numpy().astype(np.float64)
    return ys, fs


def sampled_pairs(B: int, H: int, k: int, seed: int = 0) -> np.ndarray:
    """k (b, h) pairs spread over the batch and heads, always with the first
    and last head and batch."""
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (B - 1, H - 1), (0, H - 1), (B - 1, 0)}
    while len(pairs) < min(k, B * H):
        pairs.add((int(rng.integers(B)), int(rng.integers(H))))
    return np.array(sorted(pairs), dtype=np.int64)


def compare_with_oracle(w: ssd_synth.Workload, inp=None, pairs=None, Q=None, schedule: str = "auto"):
    """Run the GPU on workload ``w`` and the oracle recurrence on all (or the
    sampled) (b, h) pairs.  Returns (err_y, err_final, y_gpu, f_gpu)."""
    inp = ssd_synth.make_inputs(w) if inp is None else inp
    Q = w.chunk_size if Q is None else Q
    y, f = run_gpu(inp, w.dtype, Q, schedule=schedule)
    yr, fr, _ = oracle.recurrence(inp, pairs=pairs)
    if pairs is None:
        return rel_err(y, yr), rel_err(f, fr), y, f
    ys = np.stack([y[b, :, h] for b, h in pairs]); yrs = np.stack([yr[b, :, h] for b, h in pairs])
    fs = np.stack([f[b, h] for b, h in pairs]); frs = np.stack([fr[b, h] for b, h in pairs])
    return rel_err(ys, yrs), rel_err(fs, frs), y, f
