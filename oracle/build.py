"""Build the oracle's shared library (plain C, gcc, OpenMP).

Test infrastructure only: the tests, the smoke check and the bench's CPU
baseline load the library this builds; the CUDA library never does.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cba_ref.c")
LIB = os.path.join(HERE, "libcba_ref.so")


def build(force: bool = False) -> str:
    """Compile cba_ref.c into libcba_ref.so next to it; return the path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
