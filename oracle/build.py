"""Compile the fp64 CPU oracle (attn_oracle.c) into oracle/libattn_oracle.so.

Test infrastructure only: the oracle judges the CUDA kernels and is never
linked into, or called by, the product library.  Plain gcc with OpenMP; no
machine-specific flags, so it builds the same way on x86_64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "libattn_oracle.so")


def build(force: bool = False) -> str:
    """Build the oracle shared library if missing or stale; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-fno-fast-math", "-fPIC", "-shared", "-fopenmp",
           "-std=c11", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
