"""Compile the CPU oracle into oracle/libmmq_oracle.so with gcc.

Test infrastructure only.  Built with -ffp-contract=off so that every f32
product and sum in the method form is rounded exactly as written (GCC
contracts a*b+c into an FMA by default on some targets, aarch64 included).
OpenMP only divides the output columns among threads (orc_gemm_mt); every
output is computed by the same single-thread code.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mmq_oracle.c")
LIB = os.path.join(HERE, "libmmq_oracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
           "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
