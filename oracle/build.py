"""Compile the fp64 CPU oracle (``mac_oracle.c``) into ``oracle/_build/libmacoracle.so``.

Test infrastructure: the oracle is built so the test suite and the benchmark's
CPU leg can run it; the CUDA library never links it.  Plain gcc, ``-O2``, no
fast-math, no FMA contraction, OpenMP over (request, head).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mac_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmacoracle.so")


def build(force: bool = False) -> str:
    """Build the oracle shared library if it is missing or older than its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
