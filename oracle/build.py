"""Compile the fp64 CPU oracle (oracle.c) into a host shared library.

Test infrastructure: the oracle is the checker for the CUDA path. Building it
is part of the package build step so that the tests, the smoke check and the
benchmark's CPU baseline find it, but nothing in the product calls it.

Plain gcc, -O2 (no -ffast-math: the oracle must keep IEEE semantics for inf
and NaN), OpenMP, and no machine-specific flags, so the same source gives the
same results on x86-64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "_build", "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
