"""bench.py's GPU arm on the 128-token decode workload: one JSON line with the
benchmark contract's keys (roofline, clocks, launch count, end-to-end, CPU
baseline) and, with --graph, the graph-replay step time."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_gpu_line_keys():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "1", "--steps", "5",
                        "--warmup", "3", "--graph", "--cpu-sample-tokens", "128"],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "phases", "roofline", "gpu_launches", "clocks", "e2e",
              "cpu_baseline", "graph"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert abs(rf["frac_nominal"] - rf["achieved"] / rf["peak_nominal"]) < 1e-3
    assert rf["kernel"] == "ll_send_small_kernel"
    assert d["gpu_launches"] == 3 * 5        # one-launch send, receive, combine per step
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    if cb["cores"] > 1:
        assert cb["single_core"]["cores"] == 1 and cb["single_core"]["value"] > 0
    assert "workloads" not in d              # a non-default workload measures itself only
    assert d["graph"]["ms_per_step"] > 0 and d["graph"]["value"] > 0
    assert d["config"]["rows"] == {"received": 1024}


def test_default_line_carries_every_workload():
    """The default run (large prefill) also measures the other four workloads
    and reports each under `workloads` with its phases, dominant kernel's
    fractions, launches, clocks and end-to-end figure."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
                        "--no-cpu-baseline"], capture_output=True, text=True, cwd=ROOT, timeout=1200)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["config"]["workload"].startswith("prefill_large")
    assert d["gpu_launches"] == 3 * 3       # layout, dispatch, combine
    wls = d["workloads"]
    assert sorted(k.split("_n")[0] for k in wls) == ["ll_decode_fp8", "ll_decode_tiny", "prefill_grouped",
                                                     "skewed_zipf"]
    for name, e in wls.items():
        assert e["value"] > 0 and e["ms_per_step"] > 0, name
        assert e["dominant"]["frac"] > 0 and e["dominant"]["frac_nominal"] > 0, name
        assert e["e2e"]["h2d_bytes_per_step"] > 0 and e["e2e"]["value"] > 0, name
        assert e["gpu_launches"] > 0 and "sm_mhz" in e["clocks"], name
        assert any(k.endswith("_frac_nominal") for k in e["phases"]), name
