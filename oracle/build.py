"""Compile the CPU oracle (plain C) into oracle/liboracle.so with the host gcc.

Test infrastructure: the library built here is loaded only by the tests, the
smoke check and the benchmark's CPU-baseline / reference leg.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

# Portable flags only (the library is rebuilt on both x86-64 and aarch64 hosts):
# no -march, no fast-math, no contraction of a*b+c, IEEE subnormals kept.
CFLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
          "-Wall", "-Wextra", "-Werror"]


def needs_build() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its source; return its path."""
    if force or needs_build():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
