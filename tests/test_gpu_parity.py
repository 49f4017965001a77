"""End-to-end parity of ssd_fwd (through the C ABI) with the fp64 oracle
recurrence, element by element, on seeded inputs.

Tolerance (stated for the workloads): max|out - ref| / max|ref| <= 5e-3 for
fp32 inputs with TF32 products, <= 2e-2 for bf16 inputs with fp32
accumulation, for y and for the final state alike.

Small cases compare every element.  The full-size workloads run in the same
launch configuration the benchmark times and compare every output of a sample
of (batch, head) pairs (the oracle computes a pair's whole sequence at once).
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_synth
from gpu_util import TOL, compare_with_oracle, pair_rows, rel_err, run_gpu, run_gpu_schedule, sampled_pairs, to_device

pytestmark = pytest.mark.gpu
W = ssd_synth.WORKLOADS


@pytest.mark.parametrize("name", ["tiny", "mamba2-370m"])
def test_full_parity(name):
    w = W[name]
    ey, ef, y, _ = compare_with_oracle(w)
    assert np.all(np.isfinite(y))
    assert ey <= TOL[w.dtype] and ef <= TOL[w.dtype], (ey, ef)


@pytest.mark.parametrize("name,k", [("mamba2-2.7b", 8), ("long-16k-n256", 6)])
def test_full_size_sampled(name, k):
    w = W[name]
    pairs = sampled_pairs(w.batch, w.nheads, k)
    ey, ef, y, _ = compare_with_oracle(w, pairs=pairs)
    assert np.all(np.isfinite(y))
    assert ey <= TOL[w.dtype] and ef <= TOL[w.dtype], (ey, ef)


SWEEP = sorted(n for n in W if n.startswith("sweep-"))


@pytest.mark.parametrize("name", SWEEP)
def test_sweep_points_sampled(name):
    """Every point of the 65,536-token shape sweep (bf16, 64 heads in 8 groups),
    at full size, against the oracle on sampled (batch, head) pairs: the
    schedule ssd_fwd picks, and the others too (the one-pass kernel, and the
    staged kernels through the four step calls).  The staged bf16 path stores
    chunk and entering states in bf16; L 32768 at chunk 128 is its longest
    chain (256 chunks).  At L 32768 ssd_fwd takes the segmented one-pass
    schedule (entering states of 2048-token segments from the staged kernels,
    in bf16)."""
    import mamba_ssd_forward_chunked_gb300 as ssd
    w = W[name]
    assert len(SWEEP) == 24
    inp = ssd_synth.make_inputs(w)
    pairs = sampled_pairs(w.batch, w.nheads, 6)
    yr, fr, _ = oracle.recurrence(inp, pairs=pairs)
    yrs = np.stack([yr[b, :, h] for b, h in pairs])
    frs = np.stack([fr[b, h] for b, h in pairs])
    del yr, fr
    d = to_device(inp, w.dtype)
    del inp
    shape = ssd.shape_of(d["x"], d["Bm"], w.chunk_size)
    picked = {2: "fused", 5: "segmented"}.get(ssd.ssd_fwd_kernel_count(shape), "staged")
    others = {"fused": ["staged"], "staged": ["fused"], "segmented": ["fused", "staged"]}[picked]
    for schedule in ["auto"] + others:
        y, f = run_gpu_schedule(d, w.chunk_size, schedule)
        torch.cuda.synchronize()
        ys, fs = pair_rows(y, f, pairs)
        del y, f
        assert np.all(np.isfinite(ys))
        ey, ef = rel_err(ys, yrs), rel_err(fs, frs)
        assert ey <= TOL[w.dtype] and ef <= TOL[w.dtype], (schedule, picked, ey, ef)



def test_segmented_sampled():
    """The segmented one-pass schedule (15 segments of 2048 tokens, two
    sequences, so segment states cross a batch boundary in the reshaped
    batch), bf16 with an initial state and dstate 128, against the oracle on
    sampled (batch, head) pairs, final state included."""
    import mamba_ssd_forward_chunked_gb300 as ssd
    w = ssd_synth.custom("g", dtype="bf16", batch=2, seqlen=30720, nheads=32, ngroups=8, dstate=128,
                         chunk_size=256, init_state=True)
    inp = ssd_synth.make_inputs(w)
    pairs = sampled_pairs(w.batch, w.nheads, 6)
    yr, fr, _ = oracle.recurrence(inp, pairs=pairs)
    yrs = np.stack([yr[b, :, h] for b, h in pairs])
    frs = np.stack([fr[b, h] for b, h in pairs])
    d = to_device(inp, w.dtype)
    shape = ssd.shape_of(d["x"], d["Bm"], w.chunk_size)
    assert ssd.ssd_fwd_kernel_count(shape) == 5
    y, f = run_gpu_schedule(d, w.chunk_size, "auto")
    torch.cuda.synchronize()
    ys, fs = pair_rows(y, f, pairs)
    assert np.all(np.isfinite(ys))
    ey, ef = rel_err(ys, yrs), rel_err(fs, frs)
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"], (ey, ef)


SMALL = [
    dict(seqlen=1),
    dict(seqlen=37),
    dict(seqlen=300, chunk_size=128, dstate=256, init_state=True),
    dict(seqlen=513, chunk_size=256, dstate=128, dtype="bf16", init_state=True),
    dict(batch=3, seqlen=130, chunk_size=64, nheads=8, ngroups=4, dstate=64, dtype="bf16"),
    dict(batch=2, seqlen=1000, chunk_size=256, nheads=6, ngroups=3, dstate=256, dtype="f32", init_state=True),
    dict(batch=2, seqlen=333, chunk_size=128, nheads=8, ngroups=2, dstate=128, dtype="f32", init_state=True),
]


@pytest.mark.parametrize("over", SMALL, ids=[str(i) for i in range(len(SMALL))])
def test_small_and_ragged_shapes(over):
    w = ssd_synth.custom("s", **over)
    ey, ef, _, _ = compare_with_oracle(w)
    assert ey <= TOL[w.dtype] and ef <= TOL[w.dtype], (ey, ef)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_size_invariance(dtype):
    w = ssd_synth.custom("q", seqlen=768, nheads=4, dstate=128, dtype=dtype, init_state=True)
    inp = ssd_synth.make_inputs(w)
    ref = None
    for Q in (64, 128, 256):
        y, f = run_gpu(inp, dtype, Q)
        if ref is None:
            ref = (y, f)
        else:
            assert rel_err(y, ref[0]) <= TOL[dtype] and rel_err(f, ref[1]) <= TOL[dtype]


def _perturbed_after(inp, t, dt_value, seed=3):
    p = {k: v.copy() for k, v in inp.items()}
    rng = np.random.default_rng(seed)
    for k in ("x", "Bm", "Cm"):
        p[k][:, t + 1:] = rng.standard_normal(p[k][:, t + 1:].shape).astype(np.float32)
    p["dt"][:, t + 1:] = dt_value
    return p


def test_causality_bitwise():
    """Perturbing x, Bm, Cm and dt after token t leaves y[:, :t+1] bit-identical:
    masked entries are exact zeros, and every factor a row uses is read from
    tokens up to that row."""
    w = ssd_synth.custom("c", seqlen=600, nheads=4, dstate=128, chunk_size=256)
    inp = ssd_synth.make_inputs(w)
    y1, _ = run_gpu(inp, "f32", 256)
    t = 345
    y2, _ = run_gpu(_perturbed_after(inp, t, 0.002), "f32", 256)
    assert np.array_equal(y1[:, :t + 1], y2[:, :t + 1])


def test_causality_when_decay_switches_form():
    """A strong-decay perturbation after token t can move a tile between the
    rescaled form and the exact form (the choice reads the tile's decay);
    earlier outputs then change only by rounding."""
    w = ssd_synth.custom("c", seqlen=600, nheads=4, dstate=128, chunk_size=256)
    inp = ssd_synth.make_inputs(w)
    y1, _ = run_gpu(inp, "f32", 256)
    t = 345
    y2, _ = run_gpu(_perturbed_after(inp, t, 0.1), "f32", 256)
    assert rel_err(y2[:, :t + 1], y1[:, :t + 1]) <= 1e-5


def test_resume_with_init_state():
    """Running tokens [0, L1) and then [L1, L) from the carried final state
    matches one run over [0, L)."""
    w = ssd_synth.custom("r", seqlen=1024, nheads=4, dstate=128, chunk_size=256, init_state=True)
    inp = ssd_synth.make_inputs(w)
    y, f = run_gpu(inp, "f32", 256)
    L1 = 512
    a = {k: (v[:, :L1] if k in ("x", "dt", "Bm", "Cm") else v) for k, v in inp.items()}
    ya, fa = run_gpu(a, "f32", 256)
    b = {k: (v[:, L1:] if k in ("x", "dt", "Bm", "Cm") else v) for k, v in inp.items()}
    b["init"] = fa.astype(np.float32)
    yb, fb = run_gpu(b, "f32", 256)
    assert rel_err(np.concatenate([ya, yb], axis=1), y) <= TOL["f32"]
    assert rel_err(fb, f) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_extreme_decay_is_finite_and_exact(dtype):
    """A = -16, dt = 0.1: the cumsum falls by 410 per 256-token chunk, so any
    unmasked exp(G_i - G_j) with j > i would overflow."""
    w = ssd_synth.custom("e", seqlen=512, nheads=4, dstate=128, chunk_size=256, dtype=dtype, init_state=True)
    inp = ssd_synth.make_inputs(w)
    inp["A"][:] = -16.0
    inp["dt"][:] = 0.1
    ey, ef, y, f = compare_with_oracle(w, inp=inp)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(f))
    assert ey <= TOL[dtype] and ef <= TOL[dtype]


def test_empty_inputs():
    import mamba_ssd_forward_chunked_gb300 as ssd
    for B, L in ((0, 64), (2, 0)):
        x = torch.empty(B, L, 4, 64, device="cuda")
        dt = torch.empty(B, L, 4, device="cuda")
        Bm = torch.empty(B, L, 1, 64, device="cuda")
        A = torch.full((4,), -1.0, device="cuda")
        D = torch.ones(4, device="cuda")
        init = torch.randn(B, 4, 64, 64, device="cuda")
        y, f = ssd.ssd_fwd(x, dt, A, Bm, Bm.clone(), D, 64, init_state=init)
        torch.cuda.synchronize()
        assert y.numel() == 0 and torch.equal(f, init)


def test_device_timeout_surfaces_as_status_and_context_survives():
    import mamba_ssd_forward_chunked_gb300 as ssd
    w = ssd_synth.WORKLOADS["tiny"]
    inp = ssd_synth.make_inputs(w)
    d = to_device(inp, "f32")
    shape = ssd.shape_of(d["x"], d["Bm"], w.chunk_size)
    ws = ssd.new_workspace(shape)
    ws.zero_()
    ssd.ssd_debug_timeout_probe(ws, 2000)  # 2 ms bound on a barrier nothing arrives at
    torch.cuda.synchronize()
    assert ssd.ssd_fwd_check(ws) == 5
    # the context is still usable and the next forward pass clears the status
    y, f = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], w.chunk_size, workspace=ws)
    torch.cuda.synchronize()
    assert ssd.ssd_fwd_check(ws) == 0
    yr, fr, _ = oracle.recurrence(inp)
    assert rel_err(y.cpu().numpy(), yr) <= TOL["f32"]


def test_host_buffers_end_to_end():
    import mamba_ssd_forward_chunked_gb300 as ssd
    w = ssd_synth.custom("h", seqlen=512, nheads=4, dstate=128, chunk_size=256, dtype="bf16", init_state=True)
    inp = ssd_synth.make_inputs(w)
    h = {k: torch.from_numpy(v).pin_memory() for k, v in inp.items()}
    for k in ("x", "Bm", "Cm"):
        h[k] = h[k].to(torch.bfloat16).pin_memory()
    y, f = ssd.ssd_fwd_host(h["x"], h["dt"], h["A"], h["Bm"], h["Cm"], h["D"], 256, init_state=h["init"])
    torch.cuda.synchronize()
    yr, fr, _ = oracle.recurrence(inp)
    assert rel_err(y.float().numpy(), yr) <= TOL["bf16"] and rel_err(f.numpy(), fr) <= TOL["bf16"]


@pytest.mark.parametrize("batch,seqlen,pieces", [(3, 300, None), (3, 300, 2), (4, 300, 4), (1, 700, 3),
                                                 (1, 700, 8), (2, 700, 4)])
def test_host_buffers_pipelined(batch, seqlen, pieces):
    """The host entry point splits the work into slices whose copies and
    kernels overlap: batch ranges, or for one sequence, segments of whole
    chunks resumed from each other's final state.  Every slice must still
    match the oracle (uneven slices and a ragged last segment included), and
    the result must not depend on the split (bitwise for batch ranges, within
    rounding for segments)."""
    import mamba_ssd_forward_chunked_gb300 as ssd
    w = ssd_synth.custom("hp", batch=batch, seqlen=seqlen, nheads=4, dstate=64, chunk_size=128, dtype="bf16",
                         init_state=True)
    inp = ssd_synth.make_inputs(w)
    h = {k: torch.from_numpy(v).pin_memory() for k, v in inp.items()}
    for k in ("x", "Bm", "Cm"):
        h[k] = h[k].to(torch.bfloat16).pin_memory()
    y, f = ssd.ssd_fwd_host(h["x"], h["dt"], h["A"], h["Bm"], h["Cm"], h["D"], 128, init_state=h["init"],
                            pieces=pieces)
    y1, f1 = ssd.ssd_fwd_host(h["x"], h["dt"], h["A"], h["Bm"], h["Cm"], h["D"], 128, init_state=h["init"],
                              pieces=1)
    torch.cuda.synchronize()
    yr, fr, _ = oracle.recurrence(inp)
    assert rel_err(y.float().numpy(), yr) <= TOL["bf16"] and rel_err(f.numpy(), fr) <= TOL["bf16"]
    if batch > 1:  # batch ranges: the same kernels on the same rows
        assert torch.equal(y, y1) and torch.equal(f, f1)
    else:
        assert rel_err(y.float().numpy(), y1.float().numpy()) <= 1e-2
        assert rel_err(f.numpy(), f1.numpy()) <= 1e-2


def test_argument_errors_raise():
    import mamba_ssd_forward_chunked_gb300 as ssd
    x = torch.randn(1, 64, 4, 32, device="cuda")  # headdim 32: unsupported
    dt = torch.rand(1, 64, 4, device="cuda")
    Bm = torch.randn(1, 64, 1, 64, device="cuda")
    A = -torch.ones(4, device="cuda")
    with pytest.raises(ssd.SSDError) as e:
        ssd.ssd_fwd(x, dt, A, Bm, Bm, A, 64)
    assert e.value.code == 2
