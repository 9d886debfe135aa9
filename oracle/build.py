"""Compile the float64 CPU oracle (test infrastructure) into a shared library.

Plain gcc, no fast-math and no floating-point contraction, so that every
operation in ``rmsnorm_oracle.c`` is one IEEE double operation on any host.
OpenMP parallelises over independent rows (or columns for the weight gradient);
if the compiler has no OpenMP runtime the same source builds single-threaded.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rmsnorm_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle_rmsnorm.so")

_BASE_FLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    last_err = ""
    for extra in (["-fopenmp"], []):
        cmd = ["gcc", *_BASE_FLAGS, *extra, SRC, "-o", tmp, "-lm"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        if res.returncode == 0:
            os.replace(tmp, LIB)
            return LIB
        last_err = res.stderr
    raise RuntimeError(f"oracle build failed:\n{last_err}")


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
