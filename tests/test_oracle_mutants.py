"""The oracle's pins catch plausible mistakes.

Each mutant below is one small, believable error planted in a copy of
oracle/ep_oracle.cpp (a reversed or unfused sum, an off-by-one slot, the
wrong expert-to-rank map, a duplicated per-rank copy, the wrong FP8 constant
or rounding, a dropped term, ...). The copy is compiled to its own library in
a temporary directory and the oracle's CPU tests are run against it in a
subprocess (EP_ORACLE_LIB points the oracle at it). Every mutant must make at
least one of them fail. The committed oracle source is never modified.
"""
import concurrent.futures
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ep_oracle.cpp")
sys.path.insert(0, ROOT)
from oracle import build as oracle_build  # noqa: E402

PIN_TESTS = ["tests/test_oracle_encoders.py", "tests/test_oracle_layout.py",
             "tests/test_oracle_dispatch_combine.py"]

# (name, text in the oracle, replacement). Each text occurs exactly once.
MUTANTS = [
    ("combine sums the slots in reverse",
     "    for (int k = 0; k < K; ++k) {\n      const int32_t row = slot[static_cast<int64_t>(t) * K + k];\n"
     "      if (row < 0) continue;\n      if (row >= y_rows) { status |= kCapacity; continue; }\n"
     "      const float wk",
     "    for (int k = K - 1; k >= 0; --k) {\n      const int32_t row = slot[static_cast<int64_t>(t) * K + k];\n"
     "      if (row < 0) continue;\n      if (row >= y_rows) { status |= kCapacity; continue; }\n"
     "      const float wk"),
    ("combine multiplies and adds separately",
     "acc[h] = std::fmaf(wk, f32_from_bf16(yr[h]), acc[h]);",
     "acc[h] = acc[h] + wk * f32_from_bf16(yr[h]);"),
    ("combine drops the bias",
     "acc[h] = acc[h] + f32_from_bf16(bias[static_cast<int64_t>(t) * H + h]);",
     "acc[h] = acc[h];"),
    ("expert to rank by modulo",
     "      const int r = e / L;\n      if (!seen[r])",
     "      const int r = e % R;\n      if (!seen[r])"),
    ("one per-rank copy per slot instead of per rank",
     "if (!seen[r]) { seen[r] = 1; rank_list[r].push_back(t); }",
     "{ rank_list[r].push_back(t); }"),
    ("expert slots off by one",
     "expert_slot[static_cast<int64_t>(t) * K + k] = expert_off[e] + static_cast<int32_t>(j);",
     "expert_slot[static_cast<int64_t>(t) * K + k] = expert_off[e] + static_cast<int32_t>(j) + 1;"),
    ("alignment padding ignored",
     "const int32_t seg = (per_expert[e] + A - 1) / A * A;",
     "const int32_t seg = per_expert[e];"),
    ("FP8 scale over 224 instead of 448",
     "float s = amax / 448.0f;",
     "float s = amax / 224.0f;"),
    ("FP8 multiplies by the reciprocal of the scale",
     "e4m3_from_f32(xi / s)",
     "e4m3_from_f32(xi * (1.0f / s))"),
    ("E4M3 ties away from zero",
     "return std::fmod(f, 2.0) == 0.0 ? f : f + 1.0;",
     "return f + 1.0;"),
    ("BF16 truncates",
     "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;",
     "(void)lower;"),
    ("power-of-two scale rounded down",
     "return static_cast<float>(m == 0.5 ? static_cast<double>(s) : std::ldexp(1.0, e));",
     "return static_cast<float>(m == 0.5 ? static_cast<double>(s) : std::ldexp(1.0, e - 1));"),
    ("per-rank top-k ids not made local",
     "here ? e - r * L : -1;",
     "here ? e : -1;"),
    ("expert-major source index is the token",
     "if (exp_src) exp_src[row] = t * K + k;",
     "if (exp_src) exp_src[row] = t;"),
    ("rank pre-sum takes experts of every rank",
     "if (!valid_expert(e, E) || e / L != r) continue;",
     "if (!valid_expert(e, E)) continue;"),
    ("combine backward drops the weight",
     "bf16_from_f32(w[tk] * f32_from_bf16(g[h]))",
     "bf16_from_f32(f32_from_bf16(g[h]))"),
    ("low-latency ranges by token modulo ranks",
     "const int s = (n_s > 0) ? t / n_s : 0;",
     "const int s = t % R;"),
    ("shrink mode keeps a masked rank's own tokens",
     "      if (!valid_expert(e, E)) continue;\n      const int src = n_s > 0 ? t / n_s : 0;\n"
     "      if (rank_mask[e / L] != 0 || (src < R && rank_mask[src] != 0)) out[tk] = -1;",
     "      if (!valid_expert(e, E)) continue;\n      const int src = n_s > 0 ? t / n_s : 0;\n"
     "      if (rank_mask[e / L] != 0) out[tk] = -1;"),
]


def _build_mutant(tmp, i, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutant {i}: anchor not unique in the oracle"
    src = os.path.join(tmp, f"mutant{i}.cpp")
    lib = os.path.join(tmp, f"libmutant{i}.so")
    open(src, "w").write(text.replace(old, new))
    subprocess.check_call(["g++", *oracle_build.FLAGS, src, "-o", lib])
    return lib


def _pins_fail(lib):
    env = dict(os.environ, EP_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *PIN_TESTS, "-x", "-q", "-m", "not gpu",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    tail = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else r.stderr[-300:]
    return r.returncode == 1 and " failed" in tail, tail


def test_every_mutant_fails_a_pin(tmp_path):
    libs = [_build_mutant(str(tmp_path), i, old, new) for i, (_, old, new) in enumerate(MUTANTS)]
    workers = max(1, min(len(libs), os.cpu_count() or 1, 8))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(_pins_fail, libs))
    survivors = [(name, tail) for (name, _, _), (ok, tail) in zip(MUTANTS, results) if not ok]
    assert not survivors, survivors


def test_unmutated_copy_passes(tmp_path):
    """The harness itself: the oracle compiled the same way passes its pins."""
    text = open(SRC).read()
    src = os.path.join(str(tmp_path), "same.cpp")
    lib = os.path.join(str(tmp_path), "libsame.so")
    open(src, "w").write(text)
    subprocess.check_call(["g++", *oracle_build.FLAGS, src, "-o", lib])
    env = dict(os.environ, EP_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_encoders.py", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-500:]
