"""bench.py's host-side arithmetic, on CPU: the per-kernel byte and flop model
adds up to the step's algorithmic totals, the TF32 peak is the bf16 peak times
the measured (else the nominal) TF32/bf16 ratio, the clock summary reads nvidia-smi's CSV lines, and a DRAM
traffic record is used only while its kernel's source file is unchanged."""
import json
import os
import shutil

import pytest

import bench
import ssd_synth

STAGED = ("chunk_state", "state_passing", "compute_out")


@pytest.mark.parametrize("name", ["tiny", "mamba2-370m", "mamba2-2.7b", "long-16k-n256", "sweep-L2048-N256-Q128"])
def test_kernel_model_adds_up(name):
    w = ssd_synth.WORKLOADS[name]
    flops, by = bench.algorithmic(w)
    km = bench.kernel_model(w)
    total = sum(by.values())
    assert km["chunk_state"]["flops"] + km["compute_out"]["flops"] == flops
    assert km["causal_cb"]["flops"] + km["ssd_onepass"]["flops"] == flops and km["chunk_cumsum"]["flops"] == 0
    # one pass: the main kernel touches every byte of the step; the causal C B^T blocks read Bm and Cm once more
    assert km["ssd_onepass"]["bytes"] == total
    assert km["causal_cb"]["bytes"] == by["BmCm"]
    # staged: x and Bm are read twice (chunk_state, then compute_out)
    assert sum(km[k]["bytes"] for k in STAGED) == total + by["x"] + by["BmCm"] // 2
    assert by["init"] == (by["final"] if w.init_state else 0)


def test_tf32_peak_is_the_measured_or_nominal_fraction_of_bf16():
    pk = {"bf16_tflops": 1930.0}
    assert bench.tensor_peak(pk, "bf16") == 1930.0
    assert bench.tensor_peak(pk, "bf16", 0.3) == 1930.0  # the ratio applies to TF32 problems only
    assert bench.tensor_peak(pk, "f32") == pytest.approx(1930.0 * 1.1 / 2.25)
    assert bench.tensor_peak(pk, "f32", 0.5) == pytest.approx(965.0)


def test_clock_summary_parses_nvidia_smi_lines():
    mon = bench.ClockMonitor(0)
    mon.lines = [
        "0, 2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 950.0, 0x0000000000000004, Not Active, Not Active, Not Active, Not Active",
        "0, 2010, 2070, 940.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 940.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    s = mon.summary()
    assert s == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    mon.lines = ["0, 1500, 2070, 990.0, 0x8, Active, Not Active, Active, Not Active"]
    assert mon.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_traffic_record_is_used_only_for_the_source_it_was_taken_on(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")))
    for workload, kernels in rec.items():
        if workload.startswith("_"):
            continue
        for kernel, e in kernels.items():
            same = bench.kernel_source_digest(kernel) == e["source_sha256_16"]
            got = bench._profile_traffic(kernel, workload)
            assert got == (float(e["dram_bytes_per_launch"]) if same else None), (workload, kernel)
    # a record taken on another source of the kernel, or of a header it includes, is ignored
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    csrc = root / "mamba_ssd_forward_chunked_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("compute_out.cu",) + bench.SHARED_HEADERS:
        shutil.copy(os.path.join(bench.ROOT, "mamba_ssd_forward_chunked_gb300", "csrc", name), csrc)
    digest = bench.kernel_source_digest("compute_out", str(root))
    entry = {"dram_bytes_per_launch": 123.0, "source_sha256_16": digest}
    (root / "profiles" / "dram_traffic.json").write_text(json.dumps({"w": {"compute_out": entry}}))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench._profile_traffic("compute_out", "w") == 123.0
    with open(csrc / "ptx.cuh", "a") as f:
        f.write("\n")
    assert bench._profile_traffic("compute_out", "w") is None
