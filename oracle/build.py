"""Compile the C oracle into ``oracle/libdc_oracle.so`` with gcc.

Test infrastructure: only the tests, the smoke check and the benchmark's
CPU-baseline leg load the result.  Flags keep binary32 arithmetic IEEE:
no fast-math, no contraction, no FTZ/DAZ.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dc_oracle.c")
LIB = os.path.join(HERE, "libdc_oracle.so")

CFLAGS = ["-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
          "-fno-strict-aliasing", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its sources."""
    srcs = [SRC, os.path.join(HERE, "dc_oracle.h")]
    if not force and os.path.exists(LIB):
        lib_mtime = os.path.getmtime(LIB)
        if all(os.path.getmtime(s) <= lib_mtime for s in srcs):
            return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    compile_source(SRC, tmp)
    os.replace(tmp, LIB)
    return LIB


def compile_source(c_path: str, out_path: str) -> str:
    """Compile one C source (the oracle, or a deliberately broken copy of it
    that a test writes to a temporary folder) with the oracle's flags."""
    cc = os.environ.get("CC", "gcc")
    subprocess.run([cc, *CFLAGS, "-I", HERE, "-o", out_path, c_path], check=True)
    return out_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
