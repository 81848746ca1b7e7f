"""Compile the CPU oracle (oracle.c) into liboracle.so next to this file.

Test infrastructure: building the checker is not using it.  Plain gcc, no
fast-math and no floating-point contraction, so that every float addition in
the oracle is one IEEE binary32 addition on any host (x86-64 or aarch64).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile liboracle.so (with OpenMP for the *_mt entry points when gcc
    offers it; without, they run on one thread)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    res = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if res.returncode != 0:
        subprocess.run(base, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
