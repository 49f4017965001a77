"""The one-pass schedule (C: ssd_fwd_fused) against the fp64 oracle
recurrence, element by element, on bf16 shapes chosen to reach every branch
of the kernels: windows of 128 tokens whatever the chunk size (64, 128, 256),
dstate 64, 128 and 256 (two carried-state operand buffers, or one), runs of
windows chained through the workspace flags, grouped heads, ragged and
one-token sequences, initial states, windows that take the exact path next
to windows on the rescaled form, and the full-size workloads the benchmark
times (sampled pairs).

Tolerance: max|out - ref| / max|ref| <= 2e-2 for bf16 inputs, on y and on the
final state."""
import numpy as np
import pytest
import torch

import oracle
import ssd_synth
from gpu_util import TOL, compare_with_oracle, rel_err, run_gpu, sampled_pairs, to_device

pytestmark = pytest.mark.gpu

SHAPES = [
    dict(seqlen=1, nheads=2, dstate=64, chunk_size=64),
    dict(seqlen=37, nheads=2, dstate=128, chunk_size=128, init_state=True),
    dict(seqlen=300, nheads=4, dstate=256, chunk_size=128, init_state=True),
    dict(seqlen=513, nheads=4, dstate=128, chunk_size=256, init_state=True),
    dict(batch=3, seqlen=130, chunk_size=64, nheads=8, ngroups=4, dstate=64),
    dict(batch=2, seqlen=1000, chunk_size=256, nheads=6, ngroups=3, dstate=256, init_state=True),
    dict(batch=2, seqlen=1700, chunk_size=128, nheads=4, ngroups=2, dstate=64, init_state=True),
    dict(seqlen=2300, nheads=2, dstate=128, chunk_size=64),  # 36 windows: nine runs chained through the flags
]


@pytest.mark.parametrize("over", SHAPES, ids=[str(i) for i in range(len(SHAPES))])
def test_fused_small_and_ragged(over):
    w = ssd_synth.custom("f", dtype="bf16", **over)
    ey, ef, y, f = compare_with_oracle(w, schedule="fused")
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(f))
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"], (ey, ef)


def test_fused_mixed_fallback_and_rescaled_windows():
    """Heads 0-1 decay so fast that every window takes the exact fallback;
    heads 2-3 stay on the rescaled form; head 4-5 switch between the two
    from window to window (dt jumps to 0.1 in every other 128-token stretch)."""
    w = ssd_synth.custom("m", dtype="bf16", seqlen=1024, nheads=6, dstate=128, chunk_size=256, init_state=True)
    inp = ssd_synth.make_inputs(w)
    inp["A"][0:2] = -16.0
    inp["dt"][:, :, 0:2] = 0.1
    inp["A"][4:6] = -16.0
    stretch = (np.arange(1024) // 128) % 2 == 1
    inp["dt"][:, stretch, 4:6] = 0.1
    ey, ef, y, f = compare_with_oracle(w, inp=inp, schedule="fused")
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(f))
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"], (ey, ef)


def test_fused_causality_bitwise():
    """Perturbing x, Bm, Cm and dt after token t leaves y[:, :t+1] bit-identical
    (moderate decay: every window keeps the rescaled form); with a strong
    decay that may switch a window to the exact form, only rounding changes."""
    w = ssd_synth.custom("c", dtype="bf16", seqlen=600, nheads=4, dstate=128, chunk_size=256)
    inp = ssd_synth.make_inputs(w)
    y1, _ = run_gpu(inp, "bf16", 256, schedule="fused")
    t = 345
    for dt_value, exact in ((0.002, True), (0.1, False)):
        p = {k: v.copy() for k, v in inp.items()}
        rng = np.random.default_rng(3)
        for k in ("x", "Bm", "Cm"):
            p[k][:, t + 1:] = rng.standard_normal(p[k][:, t + 1:].shape).astype(np.float32)
        p["dt"][:, t + 1:] = dt_value
        y2, _ = run_gpu(p, "bf16", 256, schedule="fused")
        if exact:
            assert np.array_equal(y1[:, :t + 1], y2[:, :t + 1])
        else:
            assert rel_err(y2[:, :t + 1], y1[:, :t + 1]) <= 1e-2  # bf16 output rounding


def test_fused_chunk_size_invariance():
    w = ssd_synth.custom("q", dtype="bf16", seqlen=768, nheads=4, dstate=128, init_state=True)
    inp = ssd_synth.make_inputs(w)
    outs = [run_gpu(inp, "bf16", Q, schedule="fused") for Q in (64, 128, 256)]
    for y, f in outs[1:]:
        assert rel_err(y, outs[0][0]) <= TOL["bf16"] and rel_err(f, outs[0][1]) <= TOL["bf16"]


def test_fused_agrees_with_staged():
    """Both schedules on the same inputs: each within tolerance of the oracle
    and of each other."""
    w = ssd_synth.custom("a", dtype="bf16", batch=2, seqlen=1024, nheads=8, dstate=128, chunk_size=256,
                         init_state=True)
    inp = ssd_synth.make_inputs(w)
    import mamba_ssd_forward_chunked_gb300 as ssd
    d = to_device(inp, "bf16")
    yf, ff = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], 256, init_state=d["init"],
                         schedule="fused")
    shape = ssd.shape_of(d["x"], d["Bm"], 256)
    ws = ssd.new_workspace(shape)
    ys = torch.empty_like(d["x"])
    fs = torch.empty_like(ff)
    ssd.ssd_chunk_cumsum(shape, d["dt"], d["A"], ws)
    ssd.ssd_chunk_state(shape, d["x"], d["Bm"], ws)
    ssd.ssd_state_passing(shape, d["init"], fs, ws)
    ssd.ssd_compute_out(shape, d["x"], d["Bm"], d["Cm"], d["D"], ys, ws)
    torch.cuda.synchronize()
    yr, fr, _ = oracle.recurrence(inp)
    yf, ys = yf.float().cpu().numpy(), ys.float().cpu().numpy()
    ff, fs = ff.cpu().numpy(), fs.cpu().numpy()
    assert rel_err(yf, yr) <= TOL["bf16"] and rel_err(ys, yr) <= TOL["bf16"]
    assert rel_err(ff, fr) <= TOL["bf16"] and rel_err(fs, fr) <= TOL["bf16"]
    assert rel_err(yf, ys) <= TOL["bf16"] and rel_err(ff, fs) <= TOL["bf16"]


def test_fused_without_final_state_and_in_place_resume():
    """final_state NULL (the running state lives in the workspace), then a
    second call that resumes from the first half's state with init_state and
    final_state the same buffer."""
    import mamba_ssd_forward_chunked_gb300 as ssd
    w = ssd_synth.custom("r", dtype="bf16", seqlen=1024, nheads=4, dstate=128, chunk_size=128, init_state=True)
    inp = ssd_synth.make_inputs(w)
    yr, fr, _ = oracle.recurrence(inp)
    d = to_device(inp, "bf16")
    y, f = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], 128, init_state=d["init"],
                       want_final_state=False, schedule="fused")
    torch.cuda.synchronize()
    assert f is None and rel_err(y.float().cpu().numpy(), yr) <= TOL["bf16"]
    L1 = 384
    h = d["init"].clone()
    parts = []
    for lo, hi in ((0, L1), (L1, 1024)):
        sl = {k: (v[:, lo:hi].contiguous() if k in ("x", "dt", "Bm", "Cm") else v) for k, v in d.items()}
        yy, _ = ssd.ssd_fwd(sl["x"], sl["dt"], sl["A"], sl["Bm"], sl["Cm"], sl["D"], 128, init_state=h,
                            final_state=h, schedule="fused")
        parts.append(yy)
    torch.cuda.synchronize()
    assert rel_err(torch.cat(parts, 1).float().cpu().numpy(), yr) <= TOL["bf16"]
    assert rel_err(h.cpu().numpy(), fr) <= TOL["bf16"]


@pytest.mark.parametrize("name", ["mamba2-2.7b", "sweep-L32768-N256-Q256", "sweep-L512-N64-Q128"])
def test_fused_full_size_sampled(name):
    w = ssd_synth.WORKLOADS[name]
    pairs = sampled_pairs(w.batch, w.nheads, 6)
    ey, ef, y, _ = compare_with_oracle(w, pairs=pairs, schedule="fused")
    assert np.all(np.isfinite(y))
    assert ey <= TOL["bf16"] and ef <= TOL["bf16"], (ey, ef)


def test_fused_rejects_fp32_and_dispatch():
    import mamba_ssd_forward_chunked_gb300 as ssd
    w = ssd_synth.custom("z", seqlen=64, nheads=2, dstate=64, chunk_size=64)
    d = to_device(ssd_synth.make_inputs(w), "f32")
    with pytest.raises(ssd.SSDError):
        ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], 64, schedule="fused")
    big = ssd.make_shape(batch=4, seqlen=4096, nheads=80, headdim=64, ngroups=1, dstate=128, chunk_size=256,
                         dtype=ssd.SSD_BF16)
    assert ssd.ssd_fwd_kernel_count(big) == 2  # 160 head-pair sequences: one-pass schedule
    few = ssd.make_shape(batch=1, seqlen=4096, nheads=8, headdim=64, ngroups=1, dstate=128, chunk_size=256,
                         dtype=ssd.SSD_BF16)
    assert ssd.ssd_fwd_kernel_count(few) == 3
