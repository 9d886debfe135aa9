"""The boundary is a plain C ABI: a C11 program (no C++, no CUDA headers)
includes ``include/rmsnorm.h``, links the library and calls it.

The program is generated from the header's own declarations: it takes the
address of every entry point (so each one must link with C linkage and the
declared signature), then calls the calls that need no GPU (the workspace
queries, the status strings, host validation) and prints what they return,
which must equal what the Python binding gets from the same library. Built
with gcc -std=c11 -Wall -Wextra -Werror -pedantic into the package's build
folder; runs on a machine without a GPU.
"""
from __future__ import annotations

import os
import subprocess

import pytest

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import build as cuda_build
from tests._helpers import header_declarations

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(cuda_build.OUT_DIR, "c_consumer")

_BODY = r"""
#include <stdio.h>

#include "rmsnorm.h"

typedef void (*entry_point)(void);
static const entry_point every_entry_point[] = {
%(addresses)s
};

int main(void) {
    /* every declared entry point links */
    printf("entry_points %%zu\n", sizeof every_entry_point / sizeof every_entry_point[0]);
    /* queries */
    printf("ws %%zu\n", rmsnorm_bwd_workspace_bytes(32768, 4096));
    printf("ws_max %%zu\n", rmsnorm_bwd_workspace_bytes_max(32768, 4096));
    printf("ws_narrow %%zu\n", rmsnorm_bwd_workspace_bytes(1000, 128));
    printf("step_work %%zu\n", rmsnorm_residual_step_host_work_bytes(32768, 4096, 0));
    printf("status %%s\n", rmsnorm_status_string(RMSN_EWORKSPACE));
    /* host validation, before any CUDA call */
    printf("fwd_null %%d\n", rmsnorm_fwd(NULL, 4096, NULL, NULL, 4096, NULL, 16, 4096, 1e-6f, 0, NULL));
    printf("fwd_width %%d\n", rmsnorm_fwd(NULL, 4100, NULL, NULL, 4100, NULL, 16, 4100, 1e-6f, 0, NULL));
    printf("fwd_empty %%d\n", rmsnorm_fwd(NULL, 4096, NULL, NULL, 4096, NULL, 0, 4096, 1e-6f, 0, NULL));
    printf("flags_arg %%d\n", rmsnorm_device_error(NULL, 0) == RMSN_EINVAL ? 1 : 0);
    return 0;
}
"""


def _program() -> str:
    names = sorted(n for _, n, _ in header_declarations())
    return _BODY % {"addresses": "\n".join(f"    (entry_point){n}," for n in names)}


@pytest.fixture(scope="module")
def consumer():
    lib = cuda_build.build()
    os.makedirs(OUT, exist_ok=True)
    src = os.path.join(OUT, "consumer.c")
    exe = os.path.join(OUT, "consumer")
    with open(src, "w") as f:
        f.write(_program())
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           src, "-o", exe, "-L", libdir, "-l:" + os.path.basename(lib), "-Wl,-rpath," + libdir]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_program_links_every_entry_point_and_matches_the_binding(consumer):
    run = subprocess.run([consumer], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    got = dict(line.split(" ", 1) for line in run.stdout.strip().splitlines())
    assert int(got["entry_points"]) == len(rn.EXPORTED_SYMBOLS)
    assert int(got["ws"]) == rn.rmsnorm_bwd_workspace_bytes(32768, 4096)
    assert int(got["ws_max"]) == rn.rmsnorm_bwd_workspace_bytes_max(32768, 4096)
    assert int(got["ws_narrow"]) == rn.rmsnorm_bwd_workspace_bytes(1000, 128)
    assert int(got["step_work"]) == rn.rmsnorm_residual_step_host_work_bytes(32768, 4096)
    assert got["status"] == rn.rmsnorm_status_string(-5)
    assert int(got["fwd_null"]) == -1        # RMSN_EINVAL: null pointers
    assert int(got["fwd_width"]) == -3       # RMSN_EUNSUPPORTED: D not a multiple of 8
    assert int(got["fwd_empty"]) == 0        # T == 0: nothing to do
    assert got["flags_arg"] == "1"
