"""The benchmark's host-side contract, on the CPU: the reference arm (the
oracle timed on the host) prints one JSON line with the required keys, other
ranks of a multi-rank launch print nothing, the algorithmic byte count is the
metric's definition, and the all-cores oracle run covers the whole tensor."""
import argparse
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def run_bench(*args, env=None):
    e = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    if env:
        e.update(env)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, cwd=ROOT, env=e)
    assert r.returncode == 0, r.stderr[-2000:]
    return [line for line in r.stdout.splitlines() if line.strip()]


def test_default_workload_is_the_full_linear_layer():
    """The default step is the recipe's largest configuration: X (4/6-MSE),
    W (2D) and dY (Hadamard on the columnwise copy + SR), both copies each."""
    assert bench.DEFAULT_WORKLOAD == "linear_layer"
    parts = bench.parts_of("linear_layer")
    assert parts == ["linear_x_16384x5120", "linear_w_5120x20480", "linear_dy_16384x20480"]
    import synthetic
    assert [synthetic.WORKLOADS[p][1:3] for p in parts] == [(16384, 5120), (5120, 20480), (16384, 20480)]
    assert [synthetic.workload_flags(p) for p in parts] == [(1 | 2 | 64, 1), (1 | 2 | 4, 0), (1 | 2 | 16 | 32, 0)]
    total = sum(bench.algorithmic_bytes(*synthetic.WORKLOADS[p][1:3], synthetic.workload_flags(p)[0]) for p in parts)
    assert total == 262_144_000 + 327_680_000 + 1_048_576_000


def test_philox_roofline_peak_from_unit_counts():
    """152 SMs x 32 wide products per clock / 17 products per call x 2070 MHz."""
    assert abs(bench.philox_peak_gcalls(152, 2070.0) - 152 * 32 / 17 * 2.07) < 1e-9


def test_traffic_is_null_for_a_stale_capture(monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC", {("t", "quantize"): (123, "0" * 16)})
    assert bench.traffic_of("t", "quantize") is None
    monkeypatch.setattr(bench, "TRAFFIC", {("t", "quantize"): (123, bench.source_hash())})
    assert bench.traffic_of("t", "quantize") == 123
    # SR on both copies without 4/6, 2D or a rowwise transform runs in its own kernel
    assert bench.sources_of("quantize", 1 | 2 | 16 | 32) == "quantize_sr"
    assert bench.sources_of("quantize", 1 | 2 | 32 | 64) == "quantize"
    assert bench.sources_of("quantize", 1 | 32) == "quantize"
    assert bench.sources_of("amax", 1 | 2 | 32) == "amax"


def test_reference_arm_prints_one_contract_line():
    lines = run_bench("--impl", "reference", "--steps", "1", "--warmup", "0", "--workload", "act_46mae_8192x5120")
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 0
    assert d["config"]["workload"] == "act_46mae_8192x5120"
    assert d["config"]["M"] == 8192 and d["config"]["N"] == 5120 and d["config"]["flags"] == 67
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    assert run_bench("--impl", "reference", "--steps", "1", "--warmup", "0", env={"RANK": "1"}) == []


@pytest.mark.parametrize("flags,per_elem", [(1, 2.5625), (2, 2.5625), (3, 3.125), (3 | 4, 3.125), (1 | 64, 2.5625)])
def test_algorithmic_bytes_are_the_metric_definition(flags, per_elem):
    M, N = 8192, 5120
    assert bench.algorithmic_bytes(M, N, flags) == int(per_elem * M * N)


def test_all_cores_oracle_run_covers_the_tensor():
    args = argparse.Namespace(workload="rowwise_rn_256x1024", flags=None, sel=None)
    r = bench.run_oracle_all_cores(args)
    assert r is not None
    assert r["kind"] == "oracle" and r["value"] > 0
    assert 1 <= r["cores"] <= min(len(os.sched_getaffinity(0)), 256 // 16)
    assert "256x1024" in r["sample"]


@pytest.mark.gpu
def test_benchmark_line_on_the_gpu():
    """The benchmark's own arm on a GPU (the small rowwise workload, two
    steps): one JSON line with the contract's keys, a roofline for the
    dominant kernel, the end-to-end figure with the bytes it moved, the
    single-pass figure, the clocks and the launch count."""
    lines = run_bench("--workload", "rowwise_rn_256x1024", "--steps", "3", "--warmup", "3",
                      "--no-cpu-baseline", env={"CUDA_VISIBLE_DEVICES": os.environ.get("CUDA_VISIBLE_DEVICES", "0")})
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                "single_pass", "kernels"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["dtype"] == "f32"
    assert d["config"]["workload"] == "rowwise_rn_256x1024"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    r = d["roofline"]
    assert r["bound"] in ("hbm", "alu") and 0 < r["frac"] and r["achieved"] > 0 and r["peak"] > 0
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 2 * 256 * 1024
    assert d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 2 * 3  # amax and quantize per step
    assert d["clocks"]["sm_mhz"] is None or d["clocks"]["sm_mhz"] > 0


def test_kernel_source_lists_cover_their_includes():
    """A traffic capture is keyed by the hash of the sources its kernel is
    built from: every local header that a listed translation unit includes,
    directly or through another header, must be in the list too, or an edit
    to it would leave a stale capture looking valid."""
    import re
    csrc = bench.CSRC
    local = set(os.listdir(csrc))

    def closure(name, seen):
        if name in seen:
            return
        seen.add(name)
        with open(os.path.join(csrc, name)) as f:
            for inc in re.findall(r'#include\s+"([^"]+)"', f.read()):
                if inc in local:
                    closure(inc, seen)

    for kernel, files in bench.KERNEL_SOURCES.items():
        need = set()
        for name in files:
            if name.endswith(".cu"):
                closure(name, need)
        assert need <= set(files), (kernel, sorted(need - set(files)))
