"""Compile the CPU oracle (plain C) into ``oracle/_build/liboracle.so``.

Test infrastructure only: the library built here is the checker for the CUDA
path and is never linked into it.  Binary32 arithmetic must stay exact IEEE,
so the flags forbid fast-math and floating-point contraction.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rarn_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-pthread"]


def compile_source(src: str, out: str) -> str:
    """Compile one oracle source file into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out) or ".", exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    return compile_source(SRC, LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
