#!/usr/bin/env python3
"""Throughput of the Mamba-2 chunked SSD forward pass on GB300.

One step = one ssd_fwd call (the schedule it picks for the shape: causal_cb then
the one-pass kernel; chunk_state -> state_passing -> compute_out; or the staged
state kernels over long segments, then the one-pass pair) over one batch of
seeded synthetic inputs already resident in HBM.
Prints ONE JSON line (rank 0).  The default workload is the 2.7B-layer shape
(bf16, batch 4 x 4096 tokens, 80 heads, dstate 128).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 runs one rank per GPU (launched under torch.distributed.run, which
bench.py does itself when started without it): every rank solves its own
independent problem of the same size (weak scaling; no collective on the data
path) and the value is all ranks' tokens over the slowest rank's time.

--impl reference times the fp64 CPU oracle (the recurrence) on the host cores
on a bounded sample of the same workload, reported in the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import ssd_synth  # noqa: E402

METRIC = "SSD forward tokens/s and % of roofline (TF32 / bf16), 1xGB300"
DEFAULT_WORKLOAD = "mamba2-2.7b"
L2_FLUSH_BYTES = 256 << 20
# Device-side spin before each timed step (outside its events) so the host has
# enqueued the whole step before the first event fires: the events then time
# the kernels, not the host's launch latency (reported separately).
PRE_STEP_SLEEP_CYCLES = 200_000
# GB300's nominal dense tensor-core rates: TF32 1.1 PFLOP/s against bf16 2.25 PFLOP/s.  Used only
# when the live measurement below cannot run.
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25
KERNELS = ("chunk_state", "state_passing", "compute_out")  # staged schedule (chunk_state forms the cumsum)
FUSED_KERNELS = ("causal_cb", "ssd_onepass")                                 # one-pass schedule
# segmented one-pass schedule: the staged state kernels over segments, then the one-pass pair
SEGMENTED_KERNELS = ("chunk_cumsum", "chunk_state", "state_passing", "causal_cb", "ssd_onepass")


# ------------------------------------------------------------------ model of the work

def algorithmic(w: ssd_synth.Workload):
    """Algorithmic flops and compulsory bytes of one forward pass.

    Flops per (batch, chunk, head): 4*Q*N*P (chunk state and carried-state
    term) + P*Q*(Q+1) (causal intra-chunk product); per (batch, chunk, group):
    N*Q*(Q+1) (causal C B^T, once per group).  Bytes: x read, y write, Bm and
    Cm read, dt read, A and D read, final state write (+ initial state read).
    """
    B, L, H, P, N, G, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk_size
    nc = -(-L // Q)
    es = 2 if w.dtype == "bf16" else 4
    flops = B * nc * H * (4 * Q * N * P + P * Q * (Q + 1)) + B * nc * G * N * Q * (Q + 1)
    x = B * L * H * P * es
    st = B * H * P * N * 4
    by = {"x": x, "y": x, "BmCm": 2 * B * L * G * N * es, "dt": B * L * H * 4, "AD": 2 * H * 4,
          "final": st, "init": st if w.init_state else 0}
    return flops, by


def kernel_model(w: ssd_synth.Workload):
    """Per-kernel algorithmic work: the user-visible bytes each kernel must
    touch and its share of the algorithmic flops (intermediate workspace
    traffic is overhead and not counted)."""
    flops, by = algorithmic(w)
    B, L, H, P, N, G, Q = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk_size
    nc = -(-L // Q)
    f_state = B * nc * H * 2 * Q * N * P
    f_cb = B * nc * G * N * Q * (Q + 1)
    return {
        # segmented schedule only; on the staged one chunk_state reads dt and A itself
        "chunk_cumsum": {"bytes": by["dt"] + by["AD"] // 2, "flops": 0},
        "chunk_state": {"bytes": by["x"] + by["BmCm"] // 2 + by["dt"] + by["AD"] // 2, "flops": f_state},
        "state_passing": {"bytes": by["final"] + by["init"], "flops": 0},
        "compute_out": {"bytes": by["x"] + by["y"] + by["BmCm"] + by["AD"] // 2, "flops": flops - f_state},
        # one-pass schedule: the causal C B^T blocks (Bm, Cm read), then everything of the step
        "causal_cb": {"bytes": by["BmCm"], "flops": f_cb},
        "ssd_onepass": {"bytes": sum(by.values()), "flops": flops - f_cb},
    }


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def tensor_peak(pk, dtype, tf32_ratio=None):
    """Dense tensor-core peak for the problem's MMA type: the measured bf16
    rate, times the TF32/bf16 rate ratio for fp32 problems (measured on this
    device when given, else the nominal one)."""
    base = pk["bf16_tflops"]
    if dtype != "f32":
        return base
    return base * (NOMINAL_TF32_OVER_BF16 if tf32_ratio is None else tf32_ratio)


def measure_tf32_over_bf16(dev, n: int = 8192, reps: int = 10):
    """Ratio of cuBLAS's dense TF32 rate to its bf16 rate on this device: the
    best of ``reps`` n^3 products each (CUDA events), both at the same clocks
    and with the same method as the measured bf16 peak.  The bf16 peak times
    this ratio is the TF32 roofline denominator."""
    import torch
    rates = {}
    old = torch.backends.cuda.matmul.allow_tf32
    try:
        torch.backends.cuda.matmul.allow_tf32 = True
        for name, dt in (("bf16", torch.bfloat16), ("tf32", torch.float32)):
            a = torch.randn(n, n, device=dev, dtype=dt)
            b = torch.randn(n, n, device=dev, dtype=dt)
            for _ in range(3):
                torch.matmul(a, b)
            best = float("inf")
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                torch.matmul(a, b)
                e1.record()
                torch.cuda.synchronize(dev)
                best = min(best, e0.elapsed_time(e1) * 1e-3)
            rates[name] = 2.0 * n ** 3 / best / 1e12
            del a, b
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old
    return rates["tf32"] / rates["bf16"], rates


# ------------------------------------------------------------------ clocks

class ClockMonitor:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [t.strip() for t in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        med = statistics.median(sm) if sm else None
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ multi-rank host logic

def max_over_ranks(values, world: int, device=None):
    """Each value's maximum over all ranks (the slowest rank sets the job's
    time).  world == 1 returns the values unchanged; otherwise every rank must
    call it inside an initialised process group."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_tokens_per_s(tokens_per_rank: int, world: int, ms: float) -> float:
    """Weak scaling: every rank runs the full workload, so the job processes
    world x tokens in the slowest rank's time."""
    return tokens_per_rank * world / (ms * 1e-3)


# ------------------------------------------------------------------ GPU arm

SHARED_HEADERS = ("ptx.cuh", "ssd_internal.cuh")


def kernel_source_digest(kernel: str, root: str = None) -> str:
    """Digest of a kernel's source as compiled: its .cu file and the shared
    device headers every kernel includes (a change to either can change what
    the kernel does)."""
    csrc = os.path.join(root or ROOT, "mamba_ssd_forward_chunked_gb300", "csrc")
    h = hashlib.sha256()
    for name in (kernel + ".cu",) + SHARED_HEADERS:
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def _profile_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        e = rec[workload][kernel]
        if e.get("source_sha256_16") != kernel_source_digest(kernel):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


def run_gpu(args, w: ssd_synth.Workload, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    import mamba_ssd_forward_chunked_gb300 as ssd

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = ssd_synth.make_inputs(w, seed=w.seed + rank)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    host = {k: torch.from_numpy(v) for k, v in inp.items()}
    for k in ("x", "Bm", "Cm"):
        host[k] = host[k].to(tdt)
    host = {k: v.pin_memory() for k, v in host.items()}
    d = {k: v.to(dev) for k, v in host.items()}
    init = d.get("init")
    shape = ssd.shape_of(d["x"], d["Bm"], w.chunk_size)
    ws = ssd.new_workspace(shape, dev)
    y = torch.empty_like(d["x"])
    fin = torch.empty(w.batch, w.nheads, w.headdim, w.dstate, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], w.chunk_size, init_state=init, y=y,
                    final_state=fin, workspace=ws, stream=stream)

    nkern = ssd.ssd_fwd_kernel_count(shape)  # the schedule ssd_fwd takes for this shape
    fused = nkern in (2, 5)
    names = FUSED_KERNELS if nkern == 2 else SEGMENTED_KERNELS if nkern == 5 else KERNELS

    def staged(ev):
        # the same launches ssd_fwd makes, in its order, one ssd_fwd_range call each with events between them
        for i in range(len(names)):
            ev[i].record(stream)
            ssd.ssd_fwd_range(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], w.chunk_size, i, i + 1,
                              init_state=init, y=y, final_state=fin, workspace=ws, stream=stream)
        ev[len(names)].record(stream)

    def barrier():
        if world > 1:
            dist.barrier()

    tf32_ratio, tf32_rates = None, None
    if w.dtype == "f32":  # the TF32 roofline denominator, measured on this device before any timing
        try:
            tf32_ratio, tf32_rates = measure_tf32_over_bf16(dev)
        except Exception:
            tf32_ratio = None
    for _ in range(args.warmup):
        flush.zero_()
        fwd()
    torch.cuda.synchronize(dev)
    if ssd.ssd_fwd_check(ws) != 0:
        raise RuntimeError("device status after warm-up: " + ssd.ssd_status_string(ssd.ssd_fwd_check(ws)))

    with ClockMonitor(local_rank) as clocks:
        # timed region 1: the public call, L2 flushed before every step (outside the events)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        host_s = 0.0
        for a, b in evs:
            flush.zero_()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            a.record(stream)
            h0 = time.perf_counter()
            fwd()
            host_s += time.perf_counter() - h0
            b.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        barrier()
        step_ms = [a.elapsed_time(b) for a, b in evs]

        # timed region 2: the same launches with an event between kernels
        kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize(dev)
        for ev in kev:
            flush.zero_()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            staged(ev)
        torch.cuda.synchronize(dev)
        barrier()
        per_kernel = {n: statistics.median(ev[i].elapsed_time(ev[i + 1]) for ev in kev)
                      for i, n in enumerate(names)}

        # timed region 3: end to end from pinned host memory (copies inside the events)
        out_y = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        out_f = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
        for _ in range(args.warmup):  # untimed: the first calls create the copy streams and buffers
            ssd.ssd_fwd_host(host["x"], host["dt"], host["A"], host["Bm"], host["Cm"], host["D"], w.chunk_size,
                             init_state=host.get("init"), device=dev, out_y=out_y, out_final=out_f, workspace=ws,
                             stream=stream)
        barrier()
        torch.cuda.synchronize(dev)
        for a, b in e2e_ev:
            flush.zero_()
            torch.cuda._sleep(PRE_STEP_SLEEP_CYCLES)
            a.record(stream)
            ssd.ssd_fwd_host(host["x"], host["dt"], host["A"], host["Bm"], host["Cm"], host["D"], w.chunk_size,
                             init_state=host.get("init"), device=dev, out_y=out_y, out_final=out_f, workspace=ws,
                             stream=stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = [a.elapsed_time(b) for a, b in e2e_ev]
    status = ssd.ssd_fwd_check(ws)
    if status != 0:
        raise RuntimeError("device status after timing: " + ssd.ssd_status_string(status))

    ms, ms_e2e = max_over_ranks([statistics.median(step_ms), statistics.median(e2e_ms)], world, dev)
    if rank != 0:
        return None

    flops, by = algorithmic(w)
    total_bytes = sum(by.values())
    pk = peaks()
    tpeak = tensor_peak(pk, w.dtype, tf32_ratio)
    tsrc = pk["source"] if w.dtype != "f32" else (
        pk["source"] + " bf16 x " + ("tf32/bf16 cuBLAS rate ratio measured in this run" if tf32_ratio is not None
                                     else "nominal GB300 tf32/bf16 ratio (1.1/2.25)"))
    t_roof_us = max(flops / (tpeak * 1e12), total_bytes / (pk["hbm_gbs"] * 1e9)) * 1e6
    tokens = w.tokens * world  # whole job (weak scaling)
    km = kernel_model(w)
    dom = max(per_kernel, key=per_kernel.get)
    dk = km[dom]
    t_dom = per_kernel[dom] * 1e-3
    t_mem = dk["bytes"] / (pk["hbm_gbs"] * 1e9)
    t_tc = dk["flops"] / (tpeak * 1e12)
    if t_tc > t_mem:
        roof = {"bound": "tensor", "achieved": dk["flops"] / t_dom / 1e12, "peak": tpeak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": dk["bytes"] / t_dom / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    traffic = _profile_traffic(dom, w.name)
    roof.update({
        "traffic": traffic,
        "kernel": dom,
        "algorithmic_per_launch": dk["flops"] if roof["bound"] == "tensor" else dk["bytes"],
        "peak_source": tsrc if roof["bound"] == "tensor" else pk["source"],
    })
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_y.numel() * out_y.element_size() + out_f.numel() * out_f.element_size()
    line = {
        "metric": METRIC,
        "value": whole_job_tokens_per_s(w.tokens, world, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "tf32" if w.dtype == "f32" else "bf16",
        "data": "synthetic (seeded SplitMix64 inputs with the Mamba-2 layer value recipe)",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads,
                   "headdim": w.headdim, "dstate": w.dstate, "ngroups": w.ngroups, "chunk_size": w.chunk_size,
                   "init_state": w.init_state, "input_dtype": w.dtype, "tokens_per_step_per_gpu": w.tokens,
                   "l2": f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MB write, outside the events)"},
        "tflops": flops * world / (ms * 1e-3) / 1e12,
        "step_roofline": {"t_roof_us": t_roof_us, "t_us": ms * 1e3, "frac": t_roof_us / (ms * 1e3),
                          "flops": flops, "bytes": total_bytes, "tensor_peak_tflops": tpeak,
                          "hbm_peak_gbs": pk["hbm_gbs"], "peak_source": tsrc,
                          "tf32_over_bf16": tf32_ratio, "cublas_tflops": tf32_rates},
        "roofline": roof,
        "kernels_ms": per_kernel,
        "timing": "median over steps (CUDA events on the launching stream)",
        "gpu_launches": ssd.ssd_fwd_kernel_count(shape) * args.steps,
        "schedule": "one-pass" if nkern == 2 else "segmented one-pass" if nkern == 5 else "staged",
        "e2e": {"value": whole_job_tokens_per_s(w.tokens, world, ms_e2e), "unit": "tokens/s", "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "wall_s_timed_region_1": wall,
        "host_us_per_call": host_s / args.steps * 1e6,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, inp=inp)
    return line


# ------------------------------------------------------------------ CPU oracle arm

def _oracle_sample(w: ssd_synth.Workload, seconds: float):
    """(b, h) pairs for a bounded run of the oracle (about `seconds` of CPU work)."""
    import oracle
    threads = oracle.threads_available()
    per_pair = 2.0 * w.seqlen * w.headdim * w.dstate / 1.0e9  # ~1 G multiply-adds / s per thread
    total = w.batch * w.nheads
    k = min(total, max(threads, int(seconds * threads / max(per_pair, 1e-9))))
    rng = np.random.default_rng(0)
    idx = np.sort(rng.choice(total, size=k, replace=False))
    return np.stack([idx // w.nheads, idx % w.nheads], axis=1).astype(np.int64), threads


def cpu_baseline(w: ssd_synth.Workload, seconds: float, inp=None, reps: int = 3):
    import oracle
    inp = ssd_synth.make_inputs(w) if inp is None else inp
    pairs, threads = _oracle_sample(w, seconds / reps)
    times, used = [], threads
    for _ in range(reps):
        t0 = time.perf_counter()
        _, _, used = oracle.recurrence(inp, pairs=pairs)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    frac = len(pairs) / (w.batch * w.nheads)
    return {"value": w.tokens * frac / t, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"fp64 recurrence (C, OpenMP) on {len(pairs)} of {w.batch * w.nheads} (batch, head) pairs "
                      f"of the same workload, median of {reps}; tokens/s scaled by that fraction",
            "seconds_per_run": t}


def run_reference(args, w: ssd_synth.Workload):
    import oracle
    inp = ssd_synth.make_inputs(w)
    pairs, threads = _oracle_sample(w, args.cpu_seconds / max(1, args.steps))
    frac = len(pairs) / (w.batch * w.nheads)
    for _ in range(args.warmup):
        oracle.recurrence(inp, pairs=pairs[: max(1, len(pairs) // 8)])
    times, used = [], threads
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _, _, used = oracle.recurrence(inp, pairs=pairs)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    value = w.tokens * frac / t
    sample = (f"fp64 recurrence (C, OpenMP) on {len(pairs)} of {w.batch * w.nheads} (batch, head) pairs per step; "
              f"tokens/s scaled by that fraction")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 inputs with the Mamba-2 layer value recipe)",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
                   "dstate": w.dstate, "ngroups": w.ngroups, "chunk_size": w.chunk_size, "input_dtype": w.dtype},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------------------------ main

def relaunch_one_rank_per_gpu(n: int, argv) -> int:
    """``--gpus N`` started as a plain process: run this script again under
    torch.distributed.run with N ranks on this node (rendezvous on 127.0.0.1,
    a free port), passing the same arguments.  The ranks print through this
    process's stdout (rank 0 alone prints the line); returns their exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(ssd_synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU work budget of the oracle leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = ssd_synth.WORKLOADS[args.workload]

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world == 1 and args.gpus > 1 and "RANK" not in os.environ:
        return relaunch_one_rank_per_gpu(args.gpus, sys.argv[1:] if argv is None else list(argv))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return 0

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        line = run_gpu(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
