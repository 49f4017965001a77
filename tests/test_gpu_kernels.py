"""Each of the four kernels, run alone through its C entry point, against the
fp64 restatement of its step (the chunked form of the oracle), fed with the
same inputs -- including the intermediate results of the previous GPU step, so
that every comparison isolates one kernel."""
import numpy as np
import pytest
import torch

import oracle
import ssd_synth
from gpu_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # (name, workload overrides)
    ("tiny-f32", dict()),
    ("f32-N128-Q256", dict(seqlen=512, nheads=4, dstate=128, chunk_size=256)),
    ("bf16-N128-Q256-init", dict(seqlen=512, nheads=4, dstate=128, chunk_size=256, dtype="bf16", init_state=True)),
    ("f32-N256-Q128-ragged", dict(seqlen=300, nheads=4, dstate=256, chunk_size=128, init_state=True)),
    ("bf16-N64-Q64-G2", dict(batch=2, seqlen=200, nheads=8, ngroups=2, dstate=64, chunk_size=64, dtype="bf16")),
    ("bf16-N256-Q256-G2", dict(seqlen=700, nheads=4, ngroups=2, dstate=256, chunk_size=256, dtype="bf16")),
    # dstate 256 with four heads per group, two groups
    ("bf16-N256-Q128-G2-quad", dict(batch=2, seqlen=400, nheads=8, ngroups=2, dstate=256, chunk_size=128,
                                     dtype="bf16", init_state=True)),
    ("f32-N256-Q64-G2-quad", dict(batch=2, seqlen=200, nheads=8, ngroups=2, dstate=256, chunk_size=64,
                                   init_state=True)),
]


def _setup(over):
    import mamba_ssd_forward_chunked_gb300 as ssd
    w = ssd_synth.custom("k", **over)
    inp = ssd_synth.make_inputs(w)
    d = to_device(inp, w.dtype)
    shape = ssd.shape_of(d["x"], d["Bm"], w.chunk_size)
    ws = ssd.new_workspace(shape)
    ws.zero_()
    return ssd, w, inp, d, shape, ws


@pytest.mark.parametrize("name,over", CASES, ids=[c[0] for c in CASES])
def test_each_kernel_against_its_step(name, over):
    ssd, w, inp, d, shape, ws = _setup(over)
    Q = w.chunk_size
    V = ssd.workspace_views(shape, ws)

    # step 1: cumsum (fp32 sequential sums vs fp64)
    ssd.ssd_chunk_cumsum(shape, d["dt"], d["A"], ws)
    torch.cuda.synchronize()
    G_ref = oracle.chunk_cumsum(inp["dt"], inp["A"], Q)            # [B,H,nc,Q]
    G_gpu = V["cumsum"].cpu().numpy().astype(np.float64).reshape(G_ref.shape)
    assert np.max(np.abs(G_gpu - G_ref)) <= 1e-5 * max(1.0, np.max(np.abs(G_ref)))
    dtT = V["dt_t"].cpu().numpy()
    B, L, H = inp["dt"].shape
    assert np.array_equal(dtT[:, :, :L], inp["dt"].transpose(0, 2, 1))
    assert np.all(dtT[:, :, L:] == 0)
    assert int(V["status"].item()) == 0

    # step 2: chunk states (tensor cores) vs fp64 with the GPU's cumsum
    ssd.ssd_chunk_state(shape, d["x"], d["Bm"], ws)
    torch.cuda.synchronize()
    S_ref = oracle.chunk_state(inp["x"], inp["dt"], inp["Bm"], G_gpu, Q)
    S_gpu = V["states"].float().cpu().numpy().astype(np.float64)
    assert rel_err(S_gpu, S_ref) <= TOL[w.dtype], rel_err(S_gpu, S_ref)

    # step 3: state passing (fp32 elementwise) vs fp64 on the GPU's S
    final = torch.empty(B, H, 64, w.dstate, device="cuda")
    ssd.ssd_state_passing(shape, d.get("init"), final, ws)
    torch.cuda.synchronize()
    hprev_ref, fin_ref = oracle.state_passing(S_gpu, G_gpu, inp.get("init"))
    key = "states_bf16" if w.dtype == "bf16" else "states"
    hprev_gpu = V[key].float().cpu().numpy().astype(np.float64)
    tol3 = 2 ** -8 if w.dtype == "bf16" else 1e-5
    assert rel_err(hprev_gpu, hprev_ref) <= tol3, rel_err(hprev_gpu, hprev_ref)
    assert rel_err(final.cpu().numpy(), fin_ref) <= 1e-5

    # step 4: fused output vs fp64 given the GPU's entering states
    y = torch.empty_like(d["x"])
    ssd.ssd_compute_out(shape, d["x"], d["Bm"], d["Cm"], d["D"], y, ws)
    torch.cuda.synchronize()
    y_ref = oracle.compute_out(inp["x"], inp["dt"], inp["Bm"], inp["Cm"], inp["D"], G_gpu, hprev_gpu, Q)
    y_gpu = y.float().cpu().numpy()
    assert rel_err(y_gpu, y_ref) <= TOL[w.dtype], rel_err(y_gpu, y_ref)
    assert int(V["status"].item()) == 0
    assert ssd.ssd_fwd_check(ws) == 0


def test_compute_out_causal_upper_triangle_is_exactly_zero():
    """With D = 0, y at token t of a chunk depends only on tokens <= t: setting
    later tokens of x to huge values must leave earlier y bit-identical
    (masked entries are selected to 0, so 0 * 1e30 never appears as inf)."""
    ssd, w, inp, d, shape, ws = _setup(dict(seqlen=256, nheads=2, dstate=128, chunk_size=256))
    d["D"].zero_()
    y1, _ = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], 256)
    x2 = d["x"].clone()
    x2[:, 100:] = 1e30
    y2, _ = ssd.ssd_fwd(x2, d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], 256)
    torch.cuda.synchronize()
    assert torch.equal(y1[:, :100], y2[:, :100])
    assert torch.isfinite(y1).all()


@pytest.mark.parametrize("name,over", [CASES[1], CASES[3], CASES[5], CASES[7]],
                         ids=[CASES[1][0], CASES[3][0], CASES[5][0], CASES[7][0]])
def test_full_forward_equals_the_four_steps(name, over):
    """ssd_fwd on the staged schedule (fp32 inputs; bf16 at dstate 256) gives
    bit for bit what the four step calls give in order: the full forward forms
    the chunk cumsum inside chunk_state (three launches, the same scan as the
    chunk_cumsum kernel) and chains the kernels with programmatic dependent
    launch, and neither may change a result."""
    ssd, w, inp, d, shape, ws = _setup(over)
    assert ssd.ssd_fwd_kernel_count(shape) == 3
    B, L, H = inp["dt"].shape
    y1, f1 = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], w.chunk_size,
                         init_state=d.get("init"), workspace=ws)
    torch.cuda.synchronize()
    ws2 = torch.zeros_like(ws)
    y2 = torch.empty_like(d["x"])
    f2 = torch.empty(B, H, 64, w.dstate, device="cuda")
    ssd.ssd_chunk_cumsum(shape, d["dt"], d["A"], ws2)
    ssd.ssd_chunk_state(shape, d["x"], d["Bm"], ws2)
    ssd.ssd_state_passing(shape, d.get("init"), f2, ws2)
    ssd.ssd_compute_out(shape, d["x"], d["Bm"], d["Cm"], d["D"], y2, ws2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert torch.equal(f1, f2)
    v1, v2 = ssd.workspace_views(shape, ws), ssd.workspace_views(shape, ws2)
    assert torch.equal(v1["cumsum"], v2["cumsum"]) and torch.equal(v1["dt_t"], v2["dt_t"])


@pytest.mark.parametrize("over", [CASES[1][1], CASES[3][1], CASES[4][1],
                                  dict(batch=16, seqlen=384, nheads=20, dstate=128, chunk_size=128, dtype="bf16",
                                       init_state=True),
                                  dict(batch=1, seqlen=32768, nheads=64, ngroups=8, dstate=64, chunk_size=128,
                                       dtype="bf16", init_state=True)],
                         ids=["f32-N128", "f32-N256-ragged", "bf16-staged-G2", "bf16-one-pass", "bf16-segmented"])
def test_launch_ranges_equal_the_full_forward(over):
    """ssd_fwd_range over each single launch in turn (how the bench times the
    schedule's kernels) gives bit for bit what one ssd_fwd call gives, on
    every schedule (staged, one-pass, segmented one-pass)."""
    ssd, w, inp, d, shape, ws = _setup(over)
    n = ssd.ssd_fwd_kernel_count(shape)
    B, L, H = inp["dt"].shape
    y1, f1 = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], w.chunk_size,
                         init_state=d.get("init"), workspace=ws)
    ws2 = torch.zeros_like(ws)
    y2 = torch.empty_like(d["x"])
    f2 = torch.empty(B, H, 64, w.dstate, device="cuda")
    for i in range(n):
        ssd.ssd_fwd_range(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], w.chunk_size, i, i + 1,
                          init_state=d.get("init"), y=y2, final_state=f2, workspace=ws2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2)
    assert ssd.ssd_fwd_check(ws2) == 0


@pytest.mark.parametrize("over", [dict(batch=2, seqlen=300, nheads=4, ngroups=2, dstate=128, chunk_size=256),
                                  dict(seqlen=128, nheads=2, dstate=64, chunk_size=64),
                                  dict(seqlen=200, nheads=2, dstate=256, chunk_size=128)],
                         ids=["N128-G2-ragged", "N64", "N256"])
def test_causal_cb_blocks(over):
    """Step 1 of the one-pass schedule alone: every (batch, 128-token window,
    group) block equals C B^T of that window (fp64 product of the same bf16
    inputs) up to bf16 rounding, with the upper triangle exactly zero and
    rows and columns past the sequence zero."""
    ssd, w, inp, d = None, None, None, None
    ssd, w, inp, d, shape, ws = _setup(dict(over, dtype="bf16"))
    ssd.ssd_causal_cb(shape, d["Bm"], d["Cm"], ws)
    torch.cuda.synchronize()
    M = ssd.workspace_views(shape, ws)["cbm"].float().cpu().numpy().astype(np.float64)
    B, L, G, N = inp["Bm"].shape
    nw = -(-L // 128)
    assert M.shape == (B, nw, G, 128, 128)
    Bp = np.zeros((B, nw * 128, G, N))
    Cp = np.zeros((B, nw * 128, G, N))
    Bp[:, :L] = inp["Bm"]
    Cp[:, :L] = inp["Cm"]
    tri = np.tril(np.ones((128, 128), dtype=bool))
    for b in range(B):
        for k in range(nw):
            for g in range(G):
                c = Cp[b, 128 * k:128 * (k + 1), g]
                bb = Bp[b, 128 * k:128 * (k + 1), g]
                ref = np.where(tri, c @ bb.T, 0.0)
                got = M[b, k, g]
                assert np.all(got[~tri] == 0.0)
                assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5), (b, k, g)
    assert int(ssd.workspace_views(shape, ws)["status"].item()) == 0
