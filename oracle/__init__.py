"""Float64 CPU oracle for batch-invariant RMSNorm — TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline may import this package. The CUDA library never calls it and shares
no code with it; the product path fails loudly when its CUDA extension is
missing instead of falling back to anything here.

The arithmetic lives in ``rmsnorm_oracle.c`` (plain C, IEEE double). This module
only marshals numpy arrays into it. All arrays are float64, C-contiguous,
row-major ``[T, D]`` for activations, ``[D]`` for the weight and ``[T]`` for the
inverse RMS. Callers convert bf16 tensors to float64 exactly before calling.

``rounded=True`` applies the method's rounding points (fp32 inverse RMS and
weight gradient, fp32 zero-centred offset, round-to-nearest-even activation
outputs in the format ``fmt``: ``"bf16"``, the default, or ``"f16"``); the
returned values then lie exactly on those grids. ``rounded=False`` is the
unrounded mathematical function, used by finite-difference pins.

The gated functions take ``gate``: ``"silu"`` (the default) or ``"sigmoid"``.

``eps`` is an fp32 argument of the library, so in rounded mode it is first
rounded to fp32; in unrounded mode it is used as given.

Sources (short keys used in the C file):
  [Megatron]  Megatron-LM pull request 6859, "Fix the batch-invariant RMSNorm
              forward and its input gradient"
  [ZC-norm]   RL-Kernel pull request 467, "[WS1][CUDA][Qwen3-Next] C1:
              zero-centred RMSNorm references and CUDA kernel"
  [Residual]  RL-Kernel pull request 414, "[DSv4][P1-5] rmsnorm_residual"

Every function here has a finite-difference, closed-form or brute-force pin
in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

__all__ = [
    "round_bf16", "round_f16", "num_threads",
    "rmsnorm_fwd", "rmsnorm_bwd", "residual_fwd", "residual_bwd",
    "gated_fwd", "gated_bwd", "weight_grad", "fused_add_fwd", "fused_add_bwd", "gated_hf_fwd",
    "gated_hf_apply",
]

_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64
_INT = ctypes.c_int


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # RMSN_ORACLE_LIB names another build of the oracle source: the
            # planted-mistake test loads altered copies through it.
            lib = ctypes.CDLL(os.environ.get("RMSN_ORACLE_LIB") or _build.build())
            lib.orc_num_threads.restype = _INT
            lib.orc_round_bf16.restype = ctypes.c_double
            lib.orc_round_bf16.argtypes = [ctypes.c_double]
            lib.orc_round_f16.restype = ctypes.c_double
            lib.orc_round_f16.argtypes = [ctypes.c_double]
            lib.orc_rmsnorm_fwd.argtypes = [_I64, _I64, _D, _D, ctypes.c_double, _INT, _INT, _D, _D]
            lib.orc_rmsnorm_bwd.argtypes = [_I64, _I64, _D, _D, _D, _D, _D, _INT, _INT, _D, _D, _D, _D, _D]
            lib.orc_gated_fwd.argtypes = [_I64, _I64, _D, _D, _D, ctypes.c_double, _INT, _INT, _INT, _D, _D]
            lib.orc_gated_bwd.argtypes = [_I64, _I64, _D, _D, _D, _D, _D, _INT, _INT, _INT, _D, _D, _D,
                                          _D, _D, _D, _D, _D]
            lib.orc_weight_grad.argtypes = [_I64, _I64, _D, _D, _INT, _D, _D, _INT, _D, _D]
            lib.orc_gated_hf_fwd.argtypes = [_I64, _I64, _D, _D, _D, ctypes.c_double, _INT, _INT, _D, _D]
            lib.orc_gated_hf_fwd.restype = None
            lib.orc_gated_hf_apply.argtypes = [_I64, _I64, _D, _D, _D, _D, _INT, _INT, _D]
            lib.orc_gated_hf_apply.restype = None
            lib.orc_fused_add_fwd.argtypes = [_I64, _I64, _D, _D, _D, ctypes.c_double, _INT, _INT, _D, _D, _D]
            lib.orc_fused_add_bwd.argtypes = [_I64, _I64, _D, _D, _D, _D, _D, _D, _INT, _INT, _D, _D, _D,
                                              _D, _D, _D]
            for f in ("orc_rmsnorm_fwd", "orc_rmsnorm_bwd", "orc_gated_fwd", "orc_gated_bwd",
                      "orc_weight_grad", "orc_fused_add_fwd", "orc_fused_add_bwd"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _arr(a, shape=None) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def _eps(eps: float, rounded: bool) -> float:
    return float(np.float32(eps)) if rounded else float(eps)


_FMT = {"bf16": 1, "f16": 2}
_GATE = {"silu": 0, "sigmoid": 1}


def _rnd(rounded: bool, fmt: str) -> int:
    """The C side's `rounded` argument: 0 (unrounded) or the output format code."""
    if fmt not in _FMT:
        raise ValueError(f"fmt must be one of {sorted(_FMT)}, got {fmt!r}")
    return _FMT[fmt] if rounded else 0


def _gate(gate: str) -> int:
    if gate not in _GATE:
        raise ValueError(f"gate must be one of {sorted(_GATE)}, got {gate!r}")
    return _GATE[gate]


def num_threads() -> int:
    """Threads the oracle's parallel loops use (1 if built without OpenMP)."""
    return int(_load().orc_num_threads())


def round_bf16(v) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even) in one step; returns float64."""
    lib = _load()
    v = np.asarray(v, dtype=np.float64)
    return np.vectorize(lib.orc_round_bf16, otypes=[np.float64])(v) if v.size else v.copy()


def round_f16(v) -> np.ndarray:
    """Round float64 values to IEEE fp16 (nearest, ties to even) in one step; returns float64."""
    lib = _load()
    v = np.asarray(v, dtype=np.float64)
    return np.vectorize(lib.orc_round_f16, otypes=[np.float64])(v) if v.size else v.copy()


def rmsnorm_fwd(x, w, eps: float, zero_centered_gamma: bool = False, rounded: bool = True, fmt: str = "bf16"):
    """Plain / zero-centred forward. Returns ``(y [T,D], rstd [T])``."""
    x = _arr(x)
    T, D = x.shape
    w = _arr(w, (D,))
    y = np.empty((T, D))
    rstd = np.empty((T,))
    _load().orc_rmsnorm_fwd(T, D, _p(x), _p(w), _eps(eps, rounded), int(zero_centered_gamma),
                            _rnd(rounded, fmt), _p(y), _p(rstd))
    return y, rstd


def rmsnorm_bwd(g, x, w, rstd, zero_centered_gamma: bool = False, g_res=None,
                rounded: bool = True, diagnostics: bool = False, fmt: str = "bf16"):
    """Plain / zero-centred backward (``g_res`` adds the residual branch's gradient).

    ``rstd`` is the forward's saved inverse RMS. Returns ``(dx [T,D], dgamma [D])``,
    plus, with ``diagnostics``, a dict with ``dx_pre`` (dx before its final
    rounding), ``dx_scale`` (magnitude of dx's terms before cancellation) and
    ``dw_abs`` (sum of |terms| of each weight-gradient column).
    """
    x = _arr(x)
    T, D = x.shape
    g = _arr(g, (T, D))
    w = _arr(w, (D,))
    rstd = _arr(rstd, (T,))
    gr = None if g_res is None else _arr(g_res, (T, D))
    dx = np.empty((T, D))
    dw = np.empty((D,))
    diag = {k: np.empty(s) for k, s in (("dx_pre", (T, D)), ("dx_scale", (T, D)), ("dw_abs", (D,)))} \
        if diagnostics else {}
    _load().orc_rmsnorm_bwd(T, D, _p(g), _p(x), _p(w), _p(rstd), _p(gr),
                            int(zero_centered_gamma), _rnd(rounded, fmt), _p(dx), _p(dw),
                            _p(diag.get("dx_pre")), _p(diag.get("dx_scale")), _p(diag.get("dw_abs")))
    return (dx, dw, diag) if diagnostics else (dx, dw)


def residual_fwd(x, w, eps: float, zero_centered_gamma: bool = False, rounded: bool = True, fmt: str = "bf16"):
    """``rmsnorm_residual`` forward: the normalised output plus a copy of the input.

    The copy is the input itself, unchanged ([Residual], Summary: the op returns
    the RMS-normalised output and a copy of the original input, not
    RMSNorm(x + residual)). Returns ``(y, rstd, x_copy)``.
    """
    x = _arr(x)
    y, rstd = rmsnorm_fwd(x, w, eps, zero_centered_gamma, rounded, fmt)
    return y, rstd, x.copy()


def residual_bwd(g, x, w, rstd, g_res, zero_centered_gamma: bool = False, rounded: bool = True,
                 diagnostics: bool = False, fmt: str = "bf16"):
    """``rmsnorm_residual`` backward: ``dx`` gains the copy branch's gradient ``g_res``
    before its single rounding ([Residual], reviewer's "for dx": ``+ d_residual``)."""
    return rmsnorm_bwd(g, x, w, rstd, zero_centered_gamma, g_res=g_res, rounded=rounded,
                       diagnostics=diagnostics, fmt=fmt)


def gated_fwd(x, z, w, eps: float, zero_centered_gamma: bool = True, rounded: bool = True,
              gate: str = "silu", fmt: str = "bf16"):
    """Gated forward ``y = ((x r) w_eff) q(z)``, q = silu or sigmoid. Returns ``(y, rstd)``."""
    x = _arr(x)
    T, D = x.shape
    z = _arr(z, (T, D))
    w = _arr(w, (D,))
    y = np.empty((T, D))
    rstd = np.empty((T,))
    _load().orc_gated_fwd(T, D, _p(x), _p(z), _p(w), _eps(eps, rounded), int(zero_centered_gamma),
                          _gate(gate), _rnd(rounded, fmt), _p(y), _p(rstd))
    return y, rstd


def gated_bwd(g, x, z, w, rstd, zero_centered_gamma: bool = True, rounded: bool = True,
              diagnostics: bool = False, gate: str = "silu", fmt: str = "bf16"):
    """Gated backward. Returns ``(dx [T,D], dz [T,D], dw [D])``, plus with
    ``diagnostics`` a dict as in ``rmsnorm_bwd`` with ``dz_pre`` and ``dz_scale``
    (|g u| times q' with its cancelling term in absolute value) added."""
    x = _arr(x)
    T, D = x.shape
    g = _arr(g, (T, D))
    z = _arr(z, (T, D))
    w = _arr(w, (D,))
    rstd = _arr(rstd, (T,))
    dx = np.empty((T, D))
    dz = np.empty((T, D))
    dw = np.empty((D,))
    names = (("dx_pre", (T, D)), ("dx_scale", (T, D)), ("dz_pre", (T, D)), ("dz_scale", (T, D)),
             ("dw_abs", (D,)))
    diag = {k: np.empty(s) for k, s in names} if diagnostics else {}
    _load().orc_gated_bwd(T, D, _p(g), _p(x), _p(z), _p(w), _p(rstd), int(zero_centered_gamma),
                          _gate(gate), _rnd(rounded, fmt), _p(dx), _p(dz), _p(dw),
                          *[_p(diag.get(k)) for k, _ in names])
    return (dx, dz, dw, diag) if diagnostics else (dx, dz, dw)


def weight_grad(g, x, rstd, z=None, rounded: bool = True, with_abs: bool = False, gate: str = "silu"):
    """Weight gradient alone, ``sum_t g_tj [q(z_tj)] x_tj r_t`` per column.

    Columns are independent, so this may be called on any subset of columns
    (with all T rows) to check sampled columns of a large problem; pass the
    gate ``z`` for the gated variant. Returns ``[D]`` (and, with ``with_abs``,
    the per-column sum of |terms| as a second array).
    """
    x = _arr(x)
    T, D = x.shape
    g = _arr(g, (T, D))
    rstd = _arr(rstd, (T,))
    zz = None if z is None else _arr(z, (T, D))
    dw = np.empty((D,))
    dwa = np.empty((D,)) if with_abs else None
    _load().orc_weight_grad(T, D, _p(g), _p(zz), _gate(gate), _p(x), _p(rstd), int(rounded), _p(dw), _p(dwa))
    return (dw, dwa) if with_abs else dw


def fused_add_fwd(x, res, w, eps: float, zero_centered_gamma: bool = False, rounded: bool = True,
                  fmt: str = "bf16"):
    """Fused add + norm forward on h = x + res (fp32 sum). Returns ``(y, rstd, res_out)``
    with ``res_out`` = h rounded to ``fmt`` (rounded mode) or h (unrounded)."""
    x = _arr(x)
    T, D = x.shape
    res = _arr(res, (T, D))
    w = _arr(w, (D,))
    y = np.empty((T, D))
    rstd = np.empty((T,))
    ro = np.empty((T, D))
    _load().orc_fused_add_fwd(T, D, _p(x), _p(res), _p(w), _eps(eps, rounded), int(zero_centered_gamma),
                              _rnd(rounded, fmt), _p(y), _p(rstd), _p(ro))
    return y, rstd, ro


def fused_add_bwd(g, x, res, w, rstd, g_res=None, zero_centered_gamma: bool = False, rounded: bool = True,
                  diagnostics: bool = False, fmt: str = "bf16"):
    """Fused add + norm backward. Returns ``(dh [T,D], dgamma [D])`` (+ diagnostics as in
    ``rmsnorm_bwd``); ``dh`` is the gradient of both x and res."""
    x = _arr(x)
    T, D = x.shape
    g = _arr(g, (T, D))
    res = _arr(res, (T, D))
    w = _arr(w, (D,))
    rstd = _arr(rstd, (T,))
    gr = None if g_res is None else _arr(g_res, (T, D))
    dh = np.empty((T, D))
    dw = np.empty((D,))
    hs = np.empty((T, D))
    diag = {k: np.empty(s) for k, s in (("dx_pre", (T, D)), ("dx_scale", (T, D)), ("dw_abs", (D,)))} \
        if diagnostics else {}
    _load().orc_fused_add_bwd(T, D, _p(g), _p(x), _p(res), _p(w), _p(rstd), _p(gr), int(zero_centered_gamma),
                              _rnd(rounded, fmt), _p(dh), _p(dw), _p(hs), _p(diag.get("dx_pre")),
                              _p(diag.get("dx_scale")), _p(diag.get("dw_abs")))
    return (dh, dw, diag) if diagnostics else (dh, dw)


def gated_hf_fwd(x, z, w, eps: float, zero_centered_gamma: bool = False, rounded: bool = True):
    """Gated forward in the HF/transformers convention (normalised value and weight
    multiply in bf16). Returns ``(y, rstd)``."""
    x = _arr(x)
    T, D = x.shape
    z = _arr(z, (T, D))
    w = _arr(w, (D,))
    y = np.empty((T, D))
    rstd = np.empty((T,))
    _load().orc_gated_hf_fwd(T, D, _p(x), _p(z), _p(w), _eps(eps, rounded), int(zero_centered_gamma),
                             int(rounded), _p(y), _p(rstd))
    return y, rstd


def gated_hf_apply(x, z, w, rstd, zero_centered_gamma: bool = False, rounded: bool = True):
    """The HF-convention gated output for given inverse RMS values (the second half
    of ``gated_hf_fwd``). Returns ``y``."""
    x = _arr(x)
    T, D = x.shape
    z = _arr(z, (T, D))
    w = _arr(w, (D,))
    rstd = _arr(rstd, (T,))
    y = np.empty((T, D))
    _load().orc_gated_hf_apply(T, D, _p(x), _p(z), _p(w), _p(rstd), int(zero_centered_gamma), int(rounded), _p(y))
    return y
