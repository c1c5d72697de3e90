"""The reference arm of bench.py (the CPU oracle timed on a sample of the
workload) prints one JSON line with every key of the benchmark contract, and
its config is the one the GPU arm prints for the same workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_line_keys():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    c = d["config"]
    assert c["workload"].startswith("ll_decode_tiny") and c["tokens"] == 128 and c["topk"] == 8
    assert c["rows"] == {"received": 1024}   # 128 tokens x 8 routed slots, none masked


def test_default_run_measures_every_workload():
    """bench.py's default run (the large prefill, no variant flag) also measures
    workloads 1, 2, 3 and 5; a chosen workload, a token override or a variant
    flag measures that configuration alone."""
    import sys
    sys.path.insert(0, ROOT)
    import bench

    def extras(*argv):
        old = sys.argv
        sys.argv = ["bench.py", *argv]
        try:
            return bench.extra_workloads(bench.parse())
        finally:
            sys.argv = old

    assert extras() == [1, 2, 3, 5]
    assert extras("--steps", "20", "--warmup", "5") == [1, 2, 3, 5]
    assert extras("--workload", "3") == []
    assert extras("--tokens", "4096") == []
    assert extras("--graph") == []
    assert extras("--fp8-scales", "ue8m0") == []
    assert extras("--extra-workloads", "none") == []
    assert extras("--workload", "1", "--extra-workloads", "2,3") == [2, 3]


def test_cpu_baseline_runs_on_the_whole_workload_by_default():
    """Without --cpu-sample-tokens the oracle baseline takes every token of the
    workload, reusing the host inputs the GPU arm made; a smaller sample is
    drawn afresh from the same seeded generator (its first tokens)."""
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import epinputs as ei

    old = sys.argv
    sys.argv = ["bench.py"]
    try:
        assert bench.parse().cpu_sample_tokens is None
    finally:
        sys.argv = old
    cfg = ei.WORKLOADS[3].scaled(N=64, H=256)
    inp = ei.make_inputs(cfg, seed=0)
    whole = bench._sample(cfg, None, inp)
    assert whole["n_tok"] == 64 and whole["x"] is inp["x"] and whole["topk_idx"] is inp["topk_idx"]
    part = bench._sample(cfg, 16, inp)
    assert part["n_tok"] == 16 and part["x"] is not inp["x"]
    assert np.array_equal(part["x"], inp["x"][:16])
    ll = ei.WORKLOADS[1].scaled(N=64, H=256)
    assert bench._sample(ll, 20, None)["n_tok"] == 16        # whole source ranks (8 ranks)
