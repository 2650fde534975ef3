"""Builds the fp64 C oracle (test infrastructure) with gcc.

The oracle is only loaded by the tests, by the smoke check and by the
CPU-baseline leg of the benchmark.  Building it is not using it: the product
build compiles it so that the checker exists on the machine that runs checks.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
LIB = os.path.join(HERE, "libpa_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Compile oracle/pa_oracle.c to oracle/libpa_oracle.so (OpenMP, -O2)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
