"""Compile the float64 CPU oracle (test infrastructure) into oracle/_build/liboracle.so.

Plain gcc, no CUDA.  OpenMP is used when the compiler supports it; without it
the oracle runs single-threaded and gives the same results (every row is
computed independently, in a fixed order).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Build liboracle.so if missing or older than its source; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", SRC, "-o", tmp, "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose:
            print(" ".join(cmd), r.stdout, r.stderr, file=sys.stderr)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            return LIB
    raise RuntimeError(f"oracle build failed:\n{r.stderr}")


if __name__ == "__main__":
    print(build(force=True, verbose=True))
