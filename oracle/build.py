"""Builds the C oracle into ``oracle/_build/liboracle.so`` (test infrastructure only).

Plain gcc, no intrinsics, no fused multiply-add contraction (``-ffp-contract=off``) so
that every fp32 decision the oracle takes is one IEEE operation, on x86-64 and on
aarch64 alike.  OpenMP is used only to split independent output rows across cores.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bq8_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or older than its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [
        "gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
        "-fopenmp", SRC, "-o", tmp, "-lm",
    ]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
