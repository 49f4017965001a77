"""The seeded input generator: determinism, counter access and value recipe."""
import math

import numpy as np

import ssd_synth


def test_splitmix_counter_access():
    a = ssd_synth.uniform01(0, 3, 1000)
    b = ssd_synth.uniform01(0, 3, 10, offset=500)
    assert np.array_equal(a[500:510], b)
    assert np.all((a > 0) & (a < 1))


def test_splitmix_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (state += 0x9E3779B97F4A7C15, then the finalizer), as 64-bit integers.
    z = np.array([0x9E3779B97F4A7C15], dtype=np.uint64)
    assert int(ssd_synth._mix64(z)[0]) == 0xE220A8397B1DCDAF
    z = np.array([(2 * 0x9E3779B97F4A7C15) % 2**64], dtype=np.uint64)
    assert int(ssd_synth._mix64(z)[0]) == 0x6E789E6AA1B965F4


def test_deterministic_and_distinct_streams():
    w = ssd_synth.WORKLOADS["tiny"]
    a = ssd_synth.make_inputs(w)
    b = ssd_synth.make_inputs(w)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert not np.allclose(a["Bm"], a["Cm"])


def test_value_recipe():
    w = ssd_synth.WORKLOADS["tiny"].with_(seqlen=4096, init_state=True)
    inp = ssd_synth.make_inputs(w)
    assert abs(inp["x"].mean()) < 0.01 and abs(inp["x"].std() - 1) < 0.01
    assert abs(inp["Bm"].std() * math.sqrt(w.dstate) - 1) < 0.02
    assert inp["dt"].min() >= 1e-3 - 1e-9 and inp["dt"].max() <= 0.1 + 1e-9
    assert 0.008 < np.median(inp["dt"]) < 0.012
    assert np.all(inp["A"] <= -1.0) and np.all(inp["A"] >= -16.0)
    assert abs(inp["init"].std() - 0.1) < 0.01


def test_bf16_rounding():
    v = np.array([1.0, 1.00390625, 1.005859375, -3.3, 1e-3], np.float32)
    r = ssd_synth.round_to_bf16(v)
    bits = r.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)
    assert r[0] == 1.0 and r[1] == 1.0  # tie (1 + 2^-8) rounds to even
    assert r[2] == np.float32(1.0078125)
    w = ssd_synth.WORKLOADS["mamba2-2.7b"].with_(batch=1, seqlen=64, nheads=4)
    inp = ssd_synth.make_inputs(w)
    assert np.all(inp["x"].view(np.uint32) & 0xFFFF == 0)
    assert np.all(inp["dt"].view(np.uint32) & 0xFFFF != 0)  # dt stays fp32


def test_workload_table():
    W = ssd_synth.WORKLOADS
    assert W["mamba2-2.7b"].tokens == 16384 and W["mamba2-2.7b"].nheads == 80
    sweep = [w for k, w in W.items() if k.startswith("sweep-")]
    assert len(sweep) == 24 and all(w.tokens == 65536 and w.ngroups == 8 for w in sweep)
