"""Host-side checks of the C-ABI library (no GPU needed, no compute calls).

The library must load on a machine without a GPU, export every entry point
that include/rmsnorm.h declares, answer the workspace query, and reject
invalid arguments on the host, before touching the CUDA runtime.
"""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import build as cuda_build
from tests._helpers import header_declarations

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return rn.load()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names |= set(re.findall(r"\b(rmsnorm_\w+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert declared, "no declarations found in include/*.h"
    assert declared == set(rn.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


_SCALARS = {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "float": ctypes.c_float, "size_t": ctypes.c_size_t,
            "unsigned long long": ctypes.c_ulonglong, "rmsn_stream": ctypes.c_void_p}


def _matches(c_type, ct):
    if c_type.endswith("*"):
        return ct in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(ct, ctypes._Pointer)
    return ct is _SCALARS[c_type]


def test_binding_signatures_match_the_header(lib):
    """Every ctypes prototype of the binding has the header's parameter count
    and, position by position, a type of the same kind and width (a pointer, or
    the same integer / float type), and the same return type: a mismatch would
    pass garbage through the C ABI without any error."""
    decls = header_declarations()
    assert {n for _, n, _ in decls} == set(rn.EXPORTED_SYMBOLS)
    for ret, name, types in decls:
        res, args = rn._SIGS[name]
        assert len(args) == len(types), (name, len(args), len(types))
        for i, (c_type, ct) in enumerate(zip(types, args)):
            assert _matches(c_type, ct), (name, i, c_type, ct)
        assert _matches(ret, res), (name, ret, res)
        fn = getattr(lib, name)
        assert fn.restype is res and list(fn.argtypes) == list(args), name


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5):
        assert rn.rmsnorm_status_string(st).startswith("RMSN_")
    assert "unknown" in rn.rmsnorm_status_string(17)


@pytest.mark.parametrize("T,D", [(1, 128), (16, 128), (32768, 4096), (262144, 128), (131072, 7168), (33, 8)])
def test_workspace_query(lib, T, D):
    b = rn.rmsnorm_bwd_workspace_bytes(T, D)
    assert b > 0 and b % (4 * D) == 0
    assert b // (4 * D) < T + 64  # at most one partial row per chunk
    assert rn.rmsnorm_bwd_workspace_bytes(0, D) == 0
    assert rn.rmsnorm_bwd_workspace_bytes(T, 7) == 0


def _fwd(lib, x=16, ldx=128, w=16, y=16, ldy=128, r=16, T=4, D=128, eps=1e-6):
    return lib.rmsnorm_fwd(ctypes.c_void_p(x), ldx, ctypes.c_void_p(w), ctypes.c_void_p(y), ldy,
                           ctypes.c_void_p(r), T, D, eps, 0, None)


def test_host_validation_rejects_before_launch(lib):
    # Fake, never-dereferenced addresses: every case fails validation first.
    A = 1 << 20
    assert _fwd(lib, x=A, y=A, w=A, r=A, D=7) == -3          # D not a multiple of 8
    assert _fwd(lib, x=A, y=A, w=A, r=A, D=16392, ldx=16392, ldy=16392) == -3  # D too large
    assert _fwd(lib, x=0, y=A, w=A, r=A) == -1               # null input
    assert _fwd(lib, x=A + 2, y=A, w=A, r=A) == -2           # misaligned pointer
    assert _fwd(lib, x=A, y=A, w=A, r=A, ldx=132) == -2      # row stride not 16-byte aligned
    assert _fwd(lib, x=A, y=A, w=A, r=A, ldx=120) == -1      # ld < D
    assert _fwd(lib, x=A, y=A, w=A, r=A, eps=-1.0) == -1     # negative eps
    assert _fwd(lib, x=A, y=A, w=A, r=A, eps=float("nan")) == -1
    assert _fwd(lib, x=A, y=A, w=A, r=A, T=-1) == -1
    assert _fwd(lib, x=0, y=0, w=0, r=0, T=0) == 0           # empty: OK, nothing launched
    # backward: missing / short workspace
    need = rn.rmsnorm_bwd_workspace_bytes(4, 128)
    st = lib.rmsnorm_bwd(A, 128, A, 128, A, A, A, 128, A, None, need, 4, 128, 0, None)
    assert st == -5
    st = lib.rmsnorm_bwd(A, 128, A, 128, A, A, A, 128, A, A, need - 4, 4, 128, 0, None)
    assert st == -5
    st = lib.rmsnorm_gated_bwd(A, 128, A, 128, 0, 128, A, A, A, 128, A, 128, A, A, need, 4, 128, 1, None)
    assert st == -1
    st = lib.rmsnorm_dgamma_reduce(A, need - 1, 4, 128, A, None)
    assert st == -5
    assert lib.rmsnorm_device_error(None, 0) == -1


def test_noalloc_checks_arguments_in_the_backward_order(lib):
    """rmsnorm_bwd_noalloc fails with the status rmsnorm_bwd gives for the same
    bad argument, also when the problem is too large for its array; a NULL
    dgamma and then the array's size come after those checks. Fake addresses:
    every case fails before the device is touched."""
    A = 1 << 20
    big_T, D = 32769, 8192                      # one chunk past the 32 MiB array
    assert rn.rmsnorm_bwd_workspace_bytes(big_T, D) > 32 << 20
    assert rn.rmsnorm_bwd_workspace_bytes(32768, D) == 32 << 20

    def call(g=A, x=A, w=A, r=A, dx=A, ld=D, dg=A, T=big_T):
        return lib.rmsnorm_bwd_noalloc(g, ld, x, ld, w, r, dx, ld, dg, T, D, 0, None)

    def ref(g=A, x=A, w=A, r=A, dx=A, ld=D, dg=A, T=big_T):
        return lib.rmsnorm_bwd(g, ld, x, ld, w, r, dx, ld, dg, A, 1 << 40, T, D, 0, None)

    for bad in (dict(g=0), dict(x=A + 2), dict(dx=0), dict(w=A + 4), dict(r=0), dict(dg=A + 8), dict(ld=D + 4),
                dict(ld=D - 8), dict(T=-1)):
        st = call(**bad)
        assert st in (-1, -2) and st == ref(**bad), bad
    assert call(dg=0) == -1                      # NULL dgamma: the partials cannot stay in the shared array
    assert call() == -5                          # valid arguments, too large for the array
    assert call(T=0) == 0 and call(g=0, x=0, w=0, r=0, dx=0, dg=0, T=0) == 0
    assert lib.rmsnorm_bwd_noalloc(A, 8, A, 8, A, A, A, 8, A, 4, 7, 0, None) == -3  # D not a multiple of 8


def test_ex_options_are_validated_on_the_host(lib):
    """Unknown activation formats and gates are rejected before anything else;
    known ones reach the ordinary validation (here: a null input)."""
    A = 1 << 20
    fwd = lambda dt, x=A: lib.rmsnorm_fwd_ex(x, 128, A, A, 128, A, 4, 128, 1e-6, 0, dt, None)
    assert fwd(2) == -1 and fwd(-1) == -1
    assert fwd(0, x=0) == -1 and fwd(1, x=0) == -1
    assert fwd(1, x=A + 2) == -2
    gfwd = lambda gate, dt=0: lib.rmsnorm_gated_fwd_ex(A, 128, A, 128, A, A, 128, A, 4, 128, 1e-6, 1, gate, dt,
                                                       None)
    assert gfwd(2) == -1 and gfwd(0, dt=3) == -1
    need = rn.rmsnorm_bwd_workspace_bytes(4, 128)
    assert lib.rmsnorm_gated_bwd_ex(A, 128, A, 128, A, 128, A, A, A, 128, A, 128, A, None, need, 4, 128, 1,
                                    1, 1, None) == -5
    assert lib.rmsnorm_gated_bwd_ex(A, 128, A, 128, A, 128, A, A, A, 128, A, 128, A, A, need, 4, 128, 1,
                                    5, 1, None) == -1
    assert lib.rmsnorm_fused_add_bwd_ex(A, 128, A, 128, A, 128, A, A, None, 128, A, 128, A, A, need, 4, 128,
                                        0, 9, None) == -1
    assert lib.rmsnorm_residual_fwd_ex(0, 0, 0, 0, 0, 0, 0, 0, 0, 128, 1e-6, 0, 1, None) == 0  # T = 0


def test_library_chunk_rule_matches_the_test_model(lib):
    """The workspace query reveals the library's weight-gradient chunk count for
    any T; it must be the count of the chunk rule the bit-for-bit tests model
    (tests/_helpers.py wide_chunk_rows), over widths inside and outside the band
    where chunks are shortened."""
    from tests._helpers import wide_chunk_rows
    rng = __import__("numpy").random.default_rng(4)
    Ts = sorted(set([1, 31, 32, 33, 9728, 9729, 10000, 19456, 19457, 20000, 27360, 32768, 38912, 78784, 78785, 87552,
                     87553, 97280, 131072, 262144] + [int(t) for t in rng.integers(1, 300000, 200)]))
    for D in (264, 2048, 2056, 4096, 7168, 7176, 8192, 16384):
        for T in Ts:
            n = rn.rmsnorm_bwd_workspace_bytes(T, D) // (4 * D)
            assert n == -(-T // wide_chunk_rows(T, D)), (T, D, n)


def test_workspace_size_is_not_monotone_and_the_max_query_covers_it(lib):
    """The chunk rule makes the per-T size non-monotone at 2048 < D <= 7168; the
    max query bounds every T up to its argument and equals the per-T size where
    the size grows with T."""
    q, qmax = rn.rmsnorm_bwd_workspace_bytes, rn.rmsnorm_bwd_workspace_bytes_max
    assert q(20000, 4096) > q(27360, 4096)
    for D in (4096, 7168):
        sizes = [q(t, D) for t in range(1, 40001, 7)]
        m = qmax(40000, D)
        assert m >= max(sizes) and m >= q(40000, D)
        assert m == max(q(t, D) for t in range(1, 40001))
    for T, D in ((100000, 2048), (70000, 128), (50000, 8192), (200000, 4096)):
        assert qmax(T, D) == q(T, D)  # the size grows with T here
    assert qmax(0, 4096) == 0 and qmax(100, 7) == 0


def test_workspace_max_closed_form_matches_scan(lib):
    """The max query is a closed form, not a scan: for every T_max up to 131072
    (past the last row count whose chunks are shortened) it equals the running
    maximum of the per-T size, at widths inside and at the edges of the band
    where chunks are shortened; far beyond it, it is the per-T size."""
    q, qmax = rn.rmsnorm_bwd_workspace_bytes, rn.rmsnorm_bwd_workspace_bytes_max
    for D in (2056, 4096, 7168):
        run = 0
        for t in range(1, 131073):
            run = max(run, q(t, D))
            assert qmax(t, D) == run, (t, D)
    for D in (2048, 4096, 7168, 7176):
        for T in (10 ** 6, 10 ** 9, 2 ** 31 - 1):
            assert qmax(T, D) == q(T, D)


@pytest.mark.parametrize("T,D", [(1, 128), (100, 64), (32768, 4096), (4097, 4096), (70000, 8)])
def test_host_step_work_query(lib, T, D):
    """The host-buffer step's device work buffer: the weight-gradient partials
    of all T rows, plus up to three slab slots of six activation buffers and
    one fp32 buffer; slabs are whole chunks, capped at T; 0 = the default."""
    q = rn.rmsnorm_residual_step_host_work_bytes
    part = rn.rmsnorm_bwd_workspace_bytes(T, D)
    b = q(T, D)
    assert b == q(T, D, 4096) and b % 256 == 0
    slab = min(4096, T)
    slots = min(3, -(-T // 4096))
    assert b >= part + slots * (6 * slab * D * 2 + slab * 4)
    assert b < part + slots * (6 * (slab + 256) * D * 2 + (slab + 256) * 4) + 8 * D + 4096
    assert q(T, D, 10 ** 9) == q(T, D, T)                 # capped at T
    assert q(T, D, 2 ** 63 - 1) == q(T, D, T)             # no overflow in the rounding
    assert q(T, D, 1) <= b                                # one chunk per slab
    assert q(0, D) == 0 and q(T, 7) == 0 and q(T, D, -1) == 0


def test_host_step_validation_rejects_before_launch(lib):
    """The host-buffer step checks every argument before it enqueues anything."""
    A = 1 << 20
    need = rn.rmsnorm_residual_step_host_work_bytes(64, 128)

    def step(x=A, dt=0, T=64, D=128, eps=1e-6, slab=0, work=A * 16, wb=need, gres=A):
        return lib.rmsnorm_residual_step_host(x, A, gres, A, A, A, A, A, A, T, D, eps, 0, dt, slab, work, wb, None)

    assert step(dt=2) == -1                    # unknown activation format
    assert step(D=7) == -3 and step(D=16392) == -3
    assert step(eps=float("nan")) == -1 and step(eps=-1.0) == -1
    assert step(T=-1) == -1 and step(slab=-4) == -1
    assert step(x=0, T=0, work=0, wb=0) == 0   # empty: OK, nothing enqueued
    assert step(x=0) == -1                     # null host input
    assert step(work=0) == -5 and step(wb=need - 1) == -5
    assert step(work=A * 16 + 16) == -2        # work not 256-byte aligned


def test_selftest_wait_validation_rejects_before_launch(lib):
    """The wait self-test takes a limit of 1 ns .. 1 s and an 8-byte-aligned
    output pointer; anything else is refused before any launch."""
    A = 1 << 20
    st = lambda limit, out=None: lib.rmsnorm_selftest_wait_timeout(limit, out, None)
    assert st(0) == -1 and st(1_000_000_001) == -1
    assert st(1000, A + 4) == -2
    assert rn.DEVICE_ERR_WAIT_TIMEOUT == 1


def test_product_sources_never_reach_the_oracle():
    """No file of the package (Python, CUDA, headers) imports, includes or
    loads anything under oracle/, and the oracle includes nothing of the
    library: the two share no code."""
    import ast
    pkg = os.path.join(ROOT, "invariant_rmsnorm_gb300")
    for path in glob.glob(os.path.join(pkg, "*.py")):
        for node in ast.walk(ast.parse(open(path).read())):
            if isinstance(node, ast.Import):
                assert not any(a.name.split(".")[0] == "oracle" for a in node.names), path
            if isinstance(node, ast.ImportFrom):
                assert (node.module or "").split(".")[0] != "oracle", path
    for path in glob.glob(os.path.join(pkg, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h")):
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', open(path).read()):
            assert "oracle" not in inc, (path, inc)
    for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', open(os.path.join(ROOT, "oracle", "rmsnorm_oracle.c")).read()):
        assert inc in ("math.h", "stdint.h", "string.h", "omp.h"), inc


def test_package_has_no_non_cuda_path():
    """The binding refuses to run without the built library (no fallback)."""
    import importlib
    src = open(os.path.join(ROOT, "invariant_rmsnorm_gb300", "__init__.py")).read()
    assert "oracle" not in src and "import numpy" not in src
    mod = importlib.import_module("invariant_rmsnorm_gb300")
    with pytest.raises(RuntimeError):
        mod._lib, saved = None, mod._lib
        try:
            mod.load(path=os.path.join(ROOT, "does-not-exist.so"))
        finally:
            mod._lib = saved
