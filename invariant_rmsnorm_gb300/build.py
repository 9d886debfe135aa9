"""Build the sm_103a shared library ``_build/librmsnorm_gb300.so`` in-tree.

Each ``csrc/*.cu`` translation unit is compiled in parallel with nvcc for
``sm_103a`` only, then linked into one shared library exporting the C ABI of
``include/rmsnorm.h``. ``-fmad=false`` forbids contraction of a multiply and
an add into one FMA anywhere, on top of the kernels' explicitly rounded
arithmetic.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from typing import List, Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "librmsnorm_gb300.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-fmad=false", "-DNDEBUG"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources() -> List[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> List[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def lib_path(out_dir: Optional[str] = None) -> str:
    return os.path.join(out_dir or OUT_DIR, LIB_NAME)


def build(force: bool = False, extra_flags: Sequence[str] = (), out_dir: Optional[str] = None,
          verbose: bool = False) -> str:
    """Compile and link the library if any input is newer than it; return its path."""
    out_dir = out_dir or OUT_DIR
    lib = lib_path(out_dir)
    if not force and not extra_flags and os.path.exists(lib):
        newest = max(os.path.getmtime(p) for p in _inputs())
        if os.path.getmtime(lib) >= newest:
            return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, "-I", INCLUDE, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"--- {src}\n{out}")
        elif verbose and out.strip():
            print(out, file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n" + res.stdout + res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
