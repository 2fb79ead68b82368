"""Compile the CPU fp64 oracle (test infrastructure only) with gcc.

The shared library lands in ``oracle/_build/`` next to this file.  It is rebuilt
whenever the C source is newer than the library, so a checkout on another
machine (or another CPU architecture) builds its own copy.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attention_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    """Build liboracle.so if missing or stale; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -O2 without -ffast-math: gcc keeps IEEE double semantics (no reassociation).
    cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
           "-std=c11", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
