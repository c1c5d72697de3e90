"""Compile the CPU oracle into oracle/libep_oracle.so (test infrastructure).

Plain g++, no CUDA, strict IEEE arithmetic: -ffp-contract=off keeps the
compiler from fusing multiplies and adds on its own, so the only fused
multiply-add is the explicit std::fmaf of the combine.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ep_oracle.cpp")
LIB = os.path.join(HERE, "libep_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", *FLAGS, SRC, "-o", tmp])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
