"""Compile the CPU oracle into oracle/libskv_oracle.so.

TEST INFRASTRUCTURE: the oracle is the checker of the CUDA library, loaded
only by the tests, the smoke check and the benchmark's CPU-baseline leg.
Plain gcc, C11, -O2, no FMA contraction, no fast-math, so
the binary32 steps of SKV v1 format §5 round exactly as written on x86-64
and on aarch64 alike.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "skv_oracle.c")
LIB = os.path.join(HERE, "libskv_oracle.so")
FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fno-finite-math-only",
         "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    deps = [SRC, os.path.join(HERE, "phi_q24.inc")]
    if not force and os.path.exists(LIB) and all(
            os.path.getmtime(LIB) >= os.path.getmtime(d) for d in deps):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *FLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
