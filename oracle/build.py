"""Compile the fp64 C oracle (test infrastructure) into ``oracle/libgma_oracle.so``.

Plain gcc with OpenMP; no architecture-specific flags, so the same source builds on x86_64 and
aarch64 hosts and gives the same results on both.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gma_oracle.c")
LIB = os.path.join(HERE, "libgma_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Build the oracle shared library if it is missing or older than its source; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
