"""Compile the CPU oracle (test infrastructure).

oracle/libep_oracle.so: plain g++, no CUDA, single-threaded, strict IEEE
arithmetic: -ffp-contract=off keeps the compiler from fusing multiplies and
adds on its own, so the only fused multiply-add is the explicit std::fmaf of
the combine.

oracle/libep_oracle_omp.so: the same source with -fopenmp, whose row loops
run on every host core (identical results). It is built when the compiler
supports OpenMP and is used only to time the oracle on all cores.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ep_oracle.cpp")
LIB = os.path.join(HERE, "libep_oracle.so")
LIB_OMP = os.path.join(HERE, "libep_oracle_omp.so")
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def _compile(out: str, extra, force: bool) -> str:
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", *FLAGS, *extra, SRC, "-o", tmp])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    return _compile(LIB, [], force)


def build_omp(force: bool = False):
    """The all-core build, or None when the compiler has no OpenMP."""
    try:
        return _compile(LIB_OMP, ["-fopenmp"], force)
    except (subprocess.CalledProcessError, OSError):
        return None


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
    print(build_omp(force="--force" in sys.argv))
