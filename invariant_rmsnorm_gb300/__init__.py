"""Python binding of the GB300 batch-invariant RMSNorm library (C ABI in
``include/rmsnorm.h``).

Argument marshalling only: every function here takes torch tensors that the
caller allocated on a CUDA device, checks dtypes/shapes/devices, and passes raw
pointers, row strides and sizes to the ``extern "C"`` entry point of the same
name in ``_build/librmsnorm_gb300.so``. All arithmetic runs in the library's
sm_103a kernels. If the library has not been built, ``load()`` raises; there is
no other implementation to fall back to.

Activations are bf16 ``[T, D]`` (bf16 or fp16 for the ``*_ex`` calls, which take
the format from ``x``) with unit column stride (any row stride that is a
multiple of 8 elements); weights and weight gradients fp32 ``[D]``;
inverse RMS fp32 ``[T]``. Work is enqueued on ``stream`` (default: the current
torch stream of the tensors' device).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "load", "lib_path", "RmsNormError", "workspace_bytes",
    "rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_residual_fwd", "rmsnorm_residual_bwd",
    "rmsnorm_gated_fwd", "rmsnorm_gated_bwd", "rmsnorm_dgamma_reduce",
    "rmsnorm_bwd_workspace_bytes", "rmsnorm_status_string", "rmsnorm_device_error",
    "rmsnorm_bwd_noalloc", "rmsnorm_fused_add_fwd", "rmsnorm_fused_add_bwd", "rmsnorm_bwd_recompute",
    "rmsnorm_gated_bwd_recompute", "rmsnorm_gated_hf_fwd", "EXPORTED_SYMBOLS",
    "rmsnorm_fwd_ex", "rmsnorm_bwd_ex", "rmsnorm_residual_fwd_ex", "rmsnorm_residual_bwd_ex",
    "rmsnorm_gated_fwd_ex", "rmsnorm_gated_bwd_ex", "rmsnorm_fused_add_fwd_ex", "rmsnorm_fused_add_bwd_ex",
    "rmsnorm_bwd_recompute_ex", "rmsnorm_gated_bwd_recompute_ex", "DTYPE_CODES", "GATE_CODES",
    "rmsnorm_residual_step_host", "rmsnorm_residual_step_host_work_bytes", "rmsnorm_selftest_wait_timeout",
    "DEVICE_ERR_WAIT_TIMEOUT", "rmsnorm_bwd_workspace_bytes_max",
]

EXPORTED_SYMBOLS = (
    "rmsnorm_status_string", "rmsnorm_fwd", "rmsnorm_bwd_workspace_bytes", "rmsnorm_bwd",
    "rmsnorm_residual_fwd", "rmsnorm_residual_bwd", "rmsnorm_gated_fwd", "rmsnorm_gated_bwd",
    "rmsnorm_dgamma_reduce", "rmsnorm_device_error", "rmsnorm_bwd_noalloc",
    "rmsnorm_fused_add_fwd", "rmsnorm_fused_add_bwd", "rmsnorm_bwd_recompute", "rmsnorm_gated_bwd_recompute",
    "rmsnorm_gated_hf_fwd",
    "rmsnorm_fwd_ex", "rmsnorm_bwd_ex", "rmsnorm_residual_fwd_ex", "rmsnorm_residual_bwd_ex",
    "rmsnorm_gated_fwd_ex", "rmsnorm_gated_bwd_ex", "rmsnorm_fused_add_fwd_ex", "rmsnorm_fused_add_bwd_ex",
    "rmsnorm_bwd_recompute_ex", "rmsnorm_gated_bwd_recompute_ex",
    "rmsnorm_residual_step_host_work_bytes", "rmsnorm_residual_step_host", "rmsnorm_selftest_wait_timeout",
    "rmsnorm_bwd_workspace_bytes_max",
)

# RMSN_DEVICE_ERR_WAIT_TIMEOUT of include/rmsnorm.h: the flag a wait that ran out of time raises
DEVICE_ERR_WAIT_TIMEOUT = 1

# enum rmsn_dtype / enum rmsn_gate of include/rmsnorm.h
DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1}
GATE_CODES = {"silu": 0, "sigmoid": 1}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "rmsnorm_status_string": (ctypes.c_char_p, [_INT]),
    "rmsnorm_fwd": (_INT, [_P, _I64, _P, _P, _I64, _P, _I64, _I64, _F, _INT, _P]),
    "rmsnorm_bwd_workspace_bytes": (_SZ, [_I64, _I64]),
    "rmsnorm_bwd": (_INT, [_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _P, _SZ, _I64, _I64, _INT, _P]),
    "rmsnorm_residual_fwd": (_INT, [_P, _I64, _P, _P, _I64, _P, _P, _I64, _I64, _I64, _F, _INT, _P]),
    "rmsnorm_residual_bwd": (_INT, [_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I64, _P, _P, _SZ,
                                    _I64, _I64, _INT, _P]),
    "rmsnorm_gated_fwd": (_INT, [_P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _I64, _F, _INT, _P]),
    "rmsnorm_gated_hf_fwd": (_INT, [_P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _I64, _F, _INT, _P]),
    "rmsnorm_gated_bwd": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I64, _P, _P,
                                 _SZ, _I64, _I64, _INT, _P]),
    "rmsnorm_dgamma_reduce": (_INT, [_P, _SZ, _I64, _I64, _P, _P]),
    "rmsnorm_device_error": (_INT, [ctypes.POINTER(ctypes.c_uint), _INT]),
    "rmsnorm_bwd_noalloc": (_INT, [_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I64, _I64, _INT, _P]),
    "rmsnorm_fused_add_fwd": (_INT, [_P, _I64, _P, _I64, _P, _P, _I64, _P, _P, _I64, _I64, _I64, _F, _INT, _P]),
    "rmsnorm_fused_add_bwd": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I64, _P, _P, _SZ,
                                     _I64, _I64, _INT, _P]),
    "rmsnorm_bwd_recompute": (_INT, [_P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I64, _P, _P, _I64, _P, _SZ,
                                     _I64, _I64, _INT, _P]),
    "rmsnorm_gated_bwd_recompute": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I64, _P, _I64, _P, _P, _I64,
                                           _P, _SZ, _I64, _I64, _INT, _P]),
}
_SIGS["rmsnorm_residual_step_host_work_bytes"] = (_SZ, [_I64, _I64, _I64])
_SIGS["rmsnorm_bwd_workspace_bytes_max"] = (_SZ, [_I64, _I64])
_SIGS["rmsnorm_selftest_wait_timeout"] = (_INT, [ctypes.c_ulonglong, _P, _P])
_SIGS["rmsnorm_residual_step_host"] = (_INT, [_P] * 9 + [_I64, _I64, _F, _INT, _INT, _I64, _P, _SZ, _P])
# Each *_ex call: the unsuffixed signature with `int dtype` (gated: `int gate, int dtype`) before the stream.
for _name in ("rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_residual_fwd", "rmsnorm_residual_bwd",
              "rmsnorm_fused_add_fwd", "rmsnorm_fused_add_bwd", "rmsnorm_gated_fwd", "rmsnorm_gated_bwd",
              "rmsnorm_bwd_recompute", "rmsnorm_gated_bwd_recompute"):
    _res, _args = _SIGS[_name]
    _extra = [_INT, _INT] if "gated" in _name else [_INT]
    _SIGS[_name + "_ex"] = (_res, _args[:-1] + _extra + [_P])
del _name, _res, _args, _extra

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class RmsNormError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {rmsnorm_status_string(status)} (status {status})")


def lib_path() -> str:
    return _build.lib_path()


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or lib_path()
            if not os.path.exists(p):
                raise RuntimeError(
                    f"CUDA library not built ({p} missing): run `python -c \"import __graft_entry__ as g; "
                    f"g.build()\"` first. There is no non-CUDA implementation.")
            lib = ctypes.CDLL(p)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _act(t: torch.Tensor, name: str, T: int, D: int, dtype: torch.dtype = torch.bfloat16) -> int:
    if t.dtype != dtype or not t.is_cuda or t.dim() != 2:
        raise TypeError(f"{name}: expected a 2-D {dtype} CUDA tensor, got {t.dtype} {t.device} {tuple(t.shape)}")
    if tuple(t.shape) != (T, D):
        raise ValueError(f"{name}: expected shape {(T, D)}, got {tuple(t.shape)}")
    if D > 1 and t.stride(1) != 1:
        raise ValueError(f"{name}: columns must be contiguous")
    return t.stride(0) if T > 1 else max(t.stride(0), D)


def _f32(t: torch.Tensor, name: str, n: int):
    if t.dtype != torch.float32 or not t.is_cuda or t.dim() != 1 or t.shape[0] != n or (n > 1 and t.stride(0) != 1):
        raise TypeError(f"{name}: expected a contiguous fp32 CUDA tensor of shape ({n},)")


def _stream(stream, dev) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    return ctypes.c_void_p(stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream))


def _check(fn: str, status: int):
    if status != 0:
        raise RmsNormError(fn, status)


def _dtype_code(x: torch.Tensor) -> int:
    if x.dtype not in DTYPE_CODES:
        raise TypeError(f"activations must be bf16 or fp16, got {x.dtype}")
    return DTYPE_CODES[x.dtype]


def _gate_code(gate: str) -> int:
    if gate not in GATE_CODES:
        raise ValueError(f"gate must be one of {sorted(GATE_CODES)}, got {gate!r}")
    return GATE_CODES[gate]


def _ws(ws: torch.Tensor):
    if not ws.is_cuda:
        raise TypeError("ws: expected a CUDA tensor")
    return ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size()


# --------------------------------------------------------------------------
# entry points (same names as the C ABI)
# --------------------------------------------------------------------------
def rmsnorm_status_string(status: int) -> str:
    return load().rmsnorm_status_string(int(status)).decode()


def rmsnorm_bwd_workspace_bytes(T: int, D: int) -> int:
    return int(load().rmsnorm_bwd_workspace_bytes(int(T), int(D)))


workspace_bytes = rmsnorm_bwd_workspace_bytes


def rmsnorm_bwd_workspace_bytes_max(T_max: int, D: int) -> int:
    """Bytes of one workspace that serves every T up to T_max (the per-T size is
    not monotone in T at some widths)."""
    return int(load().rmsnorm_bwd_workspace_bytes_max(int(T_max), int(D)))


def rmsnorm_fwd(x, w, y, rstd, eps: float = 1e-6, zero_centered_gamma: bool = False, stream=None):
    T, D = x.shape
    ldx, ldy = _act(x, "x", T, D), _act(y, "y", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_fwd", load().rmsnorm_fwd(_ptr(x), ldx, _ptr(w), _ptr(y), ldy, _ptr(rstd), T, D,
                                             float(eps), int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_residual_fwd(x, w, y, rstd, x_copy, eps: float = 1e-6, zero_centered_gamma: bool = False,
                         stream=None):
    T, D = x.shape
    ldx, ldy, ldc = _act(x, "x", T, D), _act(y, "y", T, D), _act(x_copy, "x_copy", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_residual_fwd", load().rmsnorm_residual_fwd(
        _ptr(x), ldx, _ptr(w), _ptr(y), ldy, _ptr(rstd), _ptr(x_copy), ldc, T, D, float(eps),
        int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_gated_fwd(x, z, w, y, rstd, eps: float = 1e-6, zero_centered_gamma: bool = True, stream=None):
    T, D = x.shape
    ldx, ldz, ldy = _act(x, "x", T, D), _act(z, "z", T, D), _act(y, "y", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_gated_fwd", load().rmsnorm_gated_fwd(
        _ptr(x), ldx, _ptr(z), ldz, _ptr(w), _ptr(y), ldy, _ptr(rstd), T, D, float(eps),
        int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_gated_hf_fwd(x, z, w, y, rstd, eps: float = 1e-6, zero_centered_gamma: bool = False, stream=None):
    """Gated forward in the HF convention (bf16 casts around the weight multiply)."""
    T, D = x.shape
    ldx, ldz, ldy = _act(x, "x", T, D), _act(z, "z", T, D), _act(y, "y", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_gated_hf_fwd", load().rmsnorm_gated_hf_fwd(
        _ptr(x), ldx, _ptr(z), ldz, _ptr(w), _ptr(y), ldy, _ptr(rstd), T, D, float(eps),
        int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_bwd(g, x, w, rstd, dx, dgamma, ws, zero_centered_gamma: bool = False, stream=None):
    """``dgamma`` may be None: pass 1 only (partials stay in ``ws``)."""
    T, D = x.shape
    ldg, ldx, lddx = _act(g, "g", T, D), _act(x, "x", T, D), _act(dx, "dx", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_bwd", load().rmsnorm_bwd(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(w), _ptr(rstd), _ptr(dx), lddx, _ptr(dgamma), wp, wb, T, D,
        int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_residual_bwd(g, x, w, rstd, g_res, dx, dgamma, ws, zero_centered_gamma: bool = False,
                         stream=None):
    """``g_res`` may be None (zero); ``dgamma`` may be None (pass 1 only)."""
    T, D = x.shape
    ldg, ldx, lddx = _act(g, "g", T, D), _act(x, "x", T, D), _act(dx, "dx", T, D)
    ldgr = _act(g_res, "g_res", T, D) if g_res is not None else D
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_residual_bwd", load().rmsnorm_residual_bwd(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(w), _ptr(rstd), _ptr(g_res), ldgr, _ptr(dx), lddx, _ptr(dgamma),
        wp, wb, T, D, int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_gated_bwd(g, x, z, w, rstd, dx, dz, dw, ws, zero_centered_gamma: bool = True, stream=None):
    """``dw`` may be None (pass 1 only)."""
    T, D = x.shape
    ldg, ldx, ldz = _act(g, "g", T, D), _act(x, "x", T, D), _act(z, "z", T, D)
    lddx, lddz = _act(dx, "dx", T, D), _act(dz, "dz", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dw is not None:
        _f32(dw, "dw", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_gated_bwd", load().rmsnorm_gated_bwd(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(z), ldz, _ptr(w), _ptr(rstd), _ptr(dx), lddx, _ptr(dz), lddz,
        _ptr(dw), wp, wb, T, D, int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_fused_add_fwd(x, res, w, y, rstd, res_out, eps: float = 1e-6, zero_centered_gamma: bool = False,
                          stream=None):
    """Norm of h = x + res (fp32); also writes bf16(h) to ``res_out``."""
    T, D = x.shape
    ldx, ldr, ldy, ldo = _act(x, "x", T, D), _act(res, "res", T, D), _act(y, "y", T, D), _act(res_out, "res_out", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_fused_add_fwd", load().rmsnorm_fused_add_fwd(
        _ptr(x), ldx, _ptr(res), ldr, _ptr(w), _ptr(y), ldy, _ptr(rstd), _ptr(res_out), ldo, T, D, float(eps),
        int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_fused_add_bwd(g, x, res, w, rstd, g_res, dh, dgamma, ws, zero_centered_gamma: bool = False,
                          stream=None):
    """Gradient of h = x + res (that of both x and res); ``g_res`` may be None."""
    T, D = x.shape
    ldg, ldx, ldr, ldd = _act(g, "g", T, D), _act(x, "x", T, D), _act(res, "res", T, D), _act(dh, "dh", T, D)
    ldgr = _act(g_res, "g_res", T, D) if g_res is not None else D
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_fused_add_bwd", load().rmsnorm_fused_add_bwd(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(res), ldr, _ptr(w), _ptr(rstd), _ptr(g_res), ldgr, _ptr(dh), ldd,
        _ptr(dgamma), wp, wb, T, D, int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_bwd_recompute(g, x, w, rstd, g_res, dx, dgamma, y, ws, zero_centered_gamma: bool = False,
                          stream=None):
    """rmsnorm_residual_bwd (``g_res`` may be None) that also writes the forward's y."""
    T, D = x.shape
    ldg, ldx, lddx, ldy = _act(g, "g", T, D), _act(x, "x", T, D), _act(dx, "dx", T, D), _act(y, "y", T, D)
    ldgr = _act(g_res, "g_res", T, D) if g_res is not None else D
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_bwd_recompute", load().rmsnorm_bwd_recompute(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(w), _ptr(rstd), _ptr(g_res), ldgr, _ptr(dx), lddx, _ptr(dgamma),
        _ptr(y), ldy, wp, wb, T, D, int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_gated_bwd_recompute(g, x, z, w, rstd, dx, dz, dw, y, ws, zero_centered_gamma: bool = True,
                                stream=None):
    """rmsnorm_gated_bwd that also writes the gated forward's y."""
    T, D = x.shape
    ldg, ldx, ldz = _act(g, "g", T, D), _act(x, "x", T, D), _act(z, "z", T, D)
    lddx, lddz, ldy = _act(dx, "dx", T, D), _act(dz, "dz", T, D), _act(y, "y", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dw is not None:
        _f32(dw, "dw", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_gated_bwd_recompute", load().rmsnorm_gated_bwd_recompute(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(z), ldz, _ptr(w), _ptr(rstd), _ptr(dx), lddx, _ptr(dz), lddz, _ptr(dw),
        _ptr(y), ldy, wp, wb, T, D, int(zero_centered_gamma), _stream(stream, x.device)))


# --------------------------------------------------------------------------
# activation dtype (bf16 / fp16, from x) and gate (silu / sigmoid) options
# --------------------------------------------------------------------------
def rmsnorm_fwd_ex(x, w, y, rstd, eps: float = 1e-6, zero_centered_gamma: bool = False, stream=None):
    T, D = x.shape
    dt = x.dtype
    ldx, ldy = _act(x, "x", T, D, dt), _act(y, "y", T, D, dt)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_fwd_ex", load().rmsnorm_fwd_ex(
        _ptr(x), ldx, _ptr(w), _ptr(y), ldy, _ptr(rstd), T, D, float(eps), int(zero_centered_gamma),
        _dtype_code(x), _stream(stream, x.device)))


def rmsnorm_bwd_ex(g, x, w, rstd, dx, dgamma, ws, zero_centered_gamma: bool = False, stream=None):
    T, D = x.shape
    dt = x.dtype
    ldg, ldx, lddx = _act(g, "g", T, D, dt), _act(x, "x", T, D, dt), _act(dx, "dx", T, D, dt)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_bwd_ex", load().rmsnorm_bwd_ex(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(w), _ptr(rstd), _ptr(dx), lddx, _ptr(dgamma), wp, wb, T, D,
        int(zero_centered_gamma), _dtype_code(x), _stream(stream, x.device)))


def rmsnorm_residual_fwd_ex(x, w, y, rstd, x_copy, eps: float = 1e-6, zero_centered_gamma: bool = False,
                            stream=None):
    T, D = x.shape
    dt = x.dtype
    ldx, ldy, ldc = _act(x, "x", T, D, dt), _act(y, "y", T, D, dt), _act(x_copy, "x_copy", T, D, dt)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_residual_fwd_ex", load().rmsnorm_residual_fwd_ex(
        _ptr(x), ldx, _ptr(w), _ptr(y), ldy, _ptr(rstd), _ptr(x_copy), ldc, T, D, float(eps),
        int(zero_centered_gamma), _dtype_code(x), _stream(stream, x.device)))


def rmsnorm_residual_bwd_ex(g, x, w, rstd, g_res, dx, dgamma, ws, zero_centered_gamma: bool = False,
                            stream=None):
    T, D = x.shape
    dt = x.dtype
    ldg, ldx, lddx = _act(g, "g", T, D, dt), _act(x, "x", T, D, dt), _act(dx, "dx", T, D, dt)
    ldgr = _act(g_res, "g_res", T, D, dt) if g_res is not None else D
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_residual_bwd_ex", load().rmsnorm_residual_bwd_ex(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(w), _ptr(rstd), _ptr(g_res), ldgr, _ptr(dx), lddx, _ptr(dgamma),
        wp, wb, T, D, int(zero_centered_gamma), _dtype_code(x), _stream(stream, x.device)))


def rmsnorm_gated_fwd_ex(x, z, w, y, rstd, eps: float = 1e-6, zero_centered_gamma: bool = True,
                         gate: str = "silu", stream=None):
    T, D = x.shape
    dt = x.dtype
    ldx, ldz, ldy = _act(x, "x", T, D, dt), _act(z, "z", T, D, dt), _act(y, "y", T, D, dt)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_gated_fwd_ex", load().rmsnorm_gated_fwd_ex(
        _ptr(x), ldx, _ptr(z), ldz, _ptr(w), _ptr(y), ldy, _ptr(rstd), T, D, float(eps),
        int(zero_centered_gamma), _gate_code(gate), _dtype_code(x), _stream(stream, x.device)))


def rmsnorm_gated_bwd_ex(g, x, z, w, rstd, dx, dz, dw, ws, zero_centered_gamma: bool = True,
                         gate: str = "silu", stream=None):
    T, D = x.shape
    dt = x.dtype
    ldg, ldx, ldz = _act(g, "g", T, D, dt), _act(x, "x", T, D, dt), _act(z, "z", T, D, dt)
    lddx, lddz = _act(dx, "dx", T, D, dt), _act(dz, "dz", T, D, dt)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dw is not None:
        _f32(dw, "dw", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_gated_bwd_ex", load().rmsnorm_gated_bwd_ex(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(z), ldz, _ptr(w), _ptr(rstd), _ptr(dx), lddx, _ptr(dz), lddz,
        _ptr(dw), wp, wb, T, D, int(zero_centered_gamma), _gate_code(gate), _dtype_code(x),
        _stream(stream, x.device)))


def rmsnorm_fused_add_fwd_ex(x, res, w, y, rstd, res_out, eps: float = 1e-6, zero_centered_gamma: bool = False,
                             stream=None):
    T, D = x.shape
    dt = x.dtype
    ldx, ldr = _act(x, "x", T, D, dt), _act(res, "res", T, D, dt)
    ldy, ldo = _act(y, "y", T, D, dt), _act(res_out, "res_out", T, D, dt)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    _check("rmsnorm_fused_add_fwd_ex", load().rmsnorm_fused_add_fwd_ex(
        _ptr(x), ldx, _ptr(res), ldr, _ptr(w), _ptr(y), ldy, _ptr(rstd), _ptr(res_out), ldo, T, D, float(eps),
        int(zero_centered_gamma), _dtype_code(x), _stream(stream, x.device)))


def rmsnorm_fused_add_bwd_ex(g, x, res, w, rstd, g_res, dh, dgamma, ws, zero_centered_gamma: bool = False,
                             stream=None):
    T, D = x.shape
    dt = x.dtype
    ldg, ldx = _act(g, "g", T, D, dt), _act(x, "x", T, D, dt)
    ldr, ldd = _act(res, "res", T, D, dt), _act(dh, "dh", T, D, dt)
    ldgr = _act(g_res, "g_res", T, D, dt) if g_res is not None else D
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_fused_add_bwd_ex", load().rmsnorm_fused_add_bwd_ex(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(res), ldr, _ptr(w), _ptr(rstd), _ptr(g_res), ldgr, _ptr(dh), ldd,
        _ptr(dgamma), wp, wb, T, D, int(zero_centered_gamma), _dtype_code(x), _stream(stream, x.device)))


def rmsnorm_bwd_recompute_ex(g, x, w, rstd, g_res, dx, dgamma, y, ws, zero_centered_gamma: bool = False,
                             stream=None):
    T, D = x.shape
    dt = x.dtype
    ldg, ldx, lddx, ldy = _act(g, "g", T, D, dt), _act(x, "x", T, D, dt), _act(dx, "dx", T, D, dt), _act(y, "y", T, D, dt)
    ldgr = _act(g_res, "g_res", T, D, dt) if g_res is not None else D
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_bwd_recompute_ex", load().rmsnorm_bwd_recompute_ex(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(w), _ptr(rstd), _ptr(g_res), ldgr, _ptr(dx), lddx, _ptr(dgamma),
        _ptr(y), ldy, wp, wb, T, D, int(zero_centered_gamma), _dtype_code(x), _stream(stream, x.device)))


def rmsnorm_gated_bwd_recompute_ex(g, x, z, w, rstd, dx, dz, dw, y, ws, zero_centered_gamma: bool = True,
                                   gate: str = "silu", stream=None):
    T, D = x.shape
    dt = x.dtype
    ldg, ldx, ldz = _act(g, "g", T, D, dt), _act(x, "x", T, D, dt), _act(z, "z", T, D, dt)
    lddx, lddz, ldy = _act(dx, "dx", T, D, dt), _act(dz, "dz", T, D, dt), _act(y, "y", T, D, dt)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dw is not None:
        _f32(dw, "dw", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_gated_bwd_recompute_ex", load().rmsnorm_gated_bwd_recompute_ex(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(z), ldz, _ptr(w), _ptr(rstd), _ptr(dx), lddx, _ptr(dz), lddz, _ptr(dw),
        _ptr(y), ldy, wp, wb, T, D, int(zero_centered_gamma), _gate_code(gate), _dtype_code(x),
        _stream(stream, x.device)))


def rmsnorm_dgamma_reduce(ws, T: int, D: int, dgamma, stream=None):
    _f32(dgamma, "dgamma", D)
    wp, wb = _ws(ws)
    _check("rmsnorm_dgamma_reduce", load().rmsnorm_dgamma_reduce(
        wp, wb, int(T), int(D), _ptr(dgamma), _stream(stream, dgamma.device)))


def rmsnorm_bwd_noalloc(g, x, w, rstd, dx, dgamma, zero_centered_gamma: bool = False, stream=None):
    """Backward for callers that cannot allocate device memory: the library's own
    fixed scratch array replaces the workspace (see include/rmsnorm.h)."""
    T, D = x.shape
    ldg, ldx, lddx = _act(g, "g", T, D), _act(x, "x", T, D), _act(dx, "dx", T, D)
    _f32(w, "w", D)
    _f32(rstd, "rstd", T)
    if dgamma is not None:
        _f32(dgamma, "dgamma", D)
    _check("rmsnorm_bwd_noalloc", load().rmsnorm_bwd_noalloc(
        _ptr(g), ldg, _ptr(x), ldx, _ptr(w), _ptr(rstd), _ptr(dx), lddx, _ptr(dgamma), T, D,
        int(zero_centered_gamma), _stream(stream, x.device)))


def rmsnorm_device_error(clear: bool = True) -> int:
    """Device-side error flags since the last clear (0 = none). Synchronises."""
    flags = ctypes.c_uint(0)
    _check("rmsnorm_device_error", load().rmsnorm_device_error(ctypes.byref(flags), int(clear)))
    return int(flags.value)


def _host(t: torch.Tensor, name: str, shape, dtype: torch.dtype):
    if t.dtype != dtype or t.is_cuda or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous host {dtype} tensor of shape {tuple(shape)}, got "
                        f"{t.dtype} {t.device} {tuple(t.shape)}")


def rmsnorm_residual_step_host_work_bytes(T: int, D: int, slab_rows: int = 0) -> int:
    return int(load().rmsnorm_residual_step_host_work_bytes(int(T), int(D), int(slab_rows)))


def rmsnorm_residual_step_host(x, g, g_res, w, y, x_copy, rstd, dx, dgamma, work, eps: float = 1e-6,
                               zero_centered_gamma: bool = False, slab_rows: int = 0, stream=None):
    """rmsnorm_residual forward + backward on HOST tensors (pinned for overlap):
    one call copies the inputs in, runs both kernels and copies every output
    back, pipelined in row slabs inside the library. ``work`` is a CUDA byte
    buffer of ``rmsnorm_residual_step_host_work_bytes(T, D, slab_rows)`` bytes;
    the host tensors must not be touched until ``stream`` has completed."""
    T, D = x.shape
    dt = x.dtype
    for t, n in ((x, "x"), (g, "g"), (y, "y"), (x_copy, "x_copy"), (dx, "dx")):
        _host(t, n, (T, D), dt)
    if g_res is not None:
        _host(g_res, "g_res", (T, D), dt)
    _host(w, "w", (D,), torch.float32)
    _host(dgamma, "dgamma", (D,), torch.float32)
    _host(rstd, "rstd", (T,), torch.float32)
    wp, wb = _ws(work)
    _check("rmsnorm_residual_step_host", load().rmsnorm_residual_step_host(
        _ptr(x), _ptr(g), _ptr(g_res), _ptr(w), _ptr(y), _ptr(x_copy), _ptr(rstd), _ptr(dx), _ptr(dgamma),
        T, D, float(eps), int(zero_centered_gamma), _dtype_code(x), int(slab_rows), wp, wb,
        _stream(stream, work.device)))


def rmsnorm_selftest_wait_timeout(limit_ns: int, waited_ns: Optional[torch.Tensor] = None, device=None, stream=None):
    """Runs the bounded-wait error path on purpose: one thread waits, with the
    kernels' own wait and a limit of ``limit_ns``, on a barrier nothing completes,
    then raises DEVICE_ERR_WAIT_TIMEOUT (read it with rmsnorm_device_error). If
    ``waited_ns`` (a CUDA int64 tensor of one element) is given, the time the wait
    took is written there."""
    if waited_ns is not None and (not waited_ns.is_cuda or waited_ns.dtype != torch.int64 or waited_ns.numel() != 1):
        raise TypeError("waited_ns: expected a one-element int64 CUDA tensor")
    dev = waited_ns.device if waited_ns is not None else (device or torch.device("cuda", torch.cuda.current_device()))
    _check("rmsnorm_selftest_wait_timeout", load().rmsnorm_selftest_wait_timeout(
        ctypes.c_ulonglong(int(limit_ns)), _ptr(waited_ns), _stream(stream, dev)))
