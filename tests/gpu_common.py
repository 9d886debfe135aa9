"""Helpers for the GPU parity tests: run a variant through the C-ABI binding,
run the oracle on the same inputs, compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import invariant_rmsnorm_gb300 as rn
import oracle
from tests._helpers import assert_bf16_parity, assert_dgamma_parity, assert_rel, to_f64

DEV = torch.device("cuda")


def empty_act(T, D, ld=None, fill=None, dtype=torch.bfloat16):
    """A [T, D] 16-bit output view; with ``ld`` its rows sit ld apart and the gap
    columns hold ``fill`` so that stray writes can be detected."""
    if ld is None or ld == D:
        return torch.empty((T, D), dtype=dtype, device=DEV)
    base = torch.full((max(T, 1), ld), fill if fill is not None else 3.0, dtype=dtype, device=DEV)
    return base[:T, :D]


_FMT = {torch.bfloat16: "bf16", torch.float16: "f16"}


def chunk_rows_hint(T, D):
    n = rn.workspace_bytes(T, D) // (4 * D)
    return T if n <= 1 else -(-T // (n - 1)) - 1, n


def run_fwd(variant, x, w, eps, zc, z=None, ld_out=None, res=None, ex=False, gate="silu"):
    """One forward through the binding. ``ex`` calls the *_ex entry point (the
    activation format is x's dtype; gated calls take ``gate``)."""
    T, D = x.shape
    dt = x.dtype
    y = empty_act(T, D, ld_out, dtype=dt)
    rstd = torch.empty(T, dtype=torch.float32, device=DEV)
    out = {"y": y, "rstd": rstd}
    if variant == "plain":
        (rn.rmsnorm_fwd_ex if ex else rn.rmsnorm_fwd)(x, w, y, rstd, eps, zc)
    elif variant == "residual":
        xc = empty_act(T, D, ld_out, dtype=dt)
        (rn.rmsnorm_residual_fwd_ex if ex else rn.rmsnorm_residual_fwd)(x, w, y, rstd, xc, eps, zc)
        out["x_copy"] = xc
    elif variant == "gated":
        if ex:
            rn.rmsnorm_gated_fwd_ex(x, z, w, y, rstd, eps, zc, gate=gate)
        else:
            rn.rmsnorm_gated_fwd(x, z, w, y, rstd, eps, zc)
    elif variant == "fused":
        ro = empty_act(T, D, ld_out, dtype=dt)
        (rn.rmsnorm_fused_add_fwd_ex if ex else rn.rmsnorm_fused_add_fwd)(x, res, w, y, rstd, ro, eps, zc)
        out["res_out"] = ro
    else:
        raise ValueError(variant)
    return out


def run_bwd(variant, g, x, w, rstd, zc, z=None, g_res=None, ld_out=None, split=False, res=None, ex=False,
            gate="silu"):
    T, D = x.shape
    dt = x.dtype
    dx = empty_act(T, D, ld_out, dtype=dt)
    dg = torch.empty(D, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(rn.workspace_bytes(T, D), 16), dtype=torch.uint8, device=DEV)
    out = {"dx": dx, "dgamma": dg, "ws": ws}
    target = None if split else dg
    if variant == "plain":
        (rn.rmsnorm_bwd_ex if ex else rn.rmsnorm_bwd)(g, x, w, rstd, dx, target, ws, zc)
    elif variant == "residual":
        (rn.rmsnorm_residual_bwd_ex if ex else rn.rmsnorm_residual_bwd)(g, x, w, rstd, g_res, dx, target, ws, zc)
    elif variant == "gated":
        dz = empty_act(T, D, ld_out, dtype=dt)
        if ex:
            rn.rmsnorm_gated_bwd_ex(g, x, z, w, rstd, dx, dz, target, ws, zc, gate=gate)
        else:
            rn.rmsnorm_gated_bwd(g, x, z, w, rstd, dx, dz, target, ws, zc)
        out["dz"] = dz
    elif variant == "fused":
        (rn.rmsnorm_fused_add_bwd_ex if ex else rn.rmsnorm_fused_add_bwd)(g, x, res, w, rstd, g_res, dx, target,
                                                                          ws, zc)
    if split:
        rn.rmsnorm_dgamma_reduce(ws, T, D, dg)
    return out


def oracle_fwd(variant, x, w, eps, zc, z=None, res=None, gate="silu"):
    fmt = _FMT[x.dtype]
    if variant == "fused":
        y, r, ro = oracle.fused_add_fwd(to_f64(x), to_f64(res), to_f64(w), eps, zc, fmt=fmt)
        return y, r
    if variant == "gated":
        y, r = oracle.gated_fwd(to_f64(x), to_f64(z), to_f64(w), eps, zc, gate=gate, fmt=fmt)
    else:
        y, r = oracle.rmsnorm_fwd(to_f64(x), to_f64(w), eps, zc, fmt=fmt)
    return y, r


def check_fwd(variant, x, w, eps, zc, out, z=None, name="", res=None, gate="silu"):
    """Compare a forward's outputs with the oracle in x's activation format."""
    fmt = _FMT[x.dtype]
    y_ref, r_ref = oracle_fwd(variant, x, w, eps, zc, z, res, gate)
    assert_rel(f"{name} rstd", to_f64(out["rstd"]), r_ref, 1e-5)
    assert_bf16_parity(f"{name} y", to_f64(out["y"]), y_ref, fmt=fmt)
    if variant == "fused":
        _, _, ro = oracle.fused_add_fwd(to_f64(x), to_f64(res), to_f64(w), eps, zc, fmt=fmt)
        np.testing.assert_array_equal(to_f64(out["res_out"]), ro, err_msg=f"{name} res_out")
    if variant == "residual":
        assert torch.equal(out["x_copy"].view(torch.int16), x.view(torch.int16)), f"{name} x_copy"


def check_bwd(variant, g, x, w, rstd, zc, out, z=None, g_res=None, name="", res=None, gate="silu"):
    """Compare against the oracle run with the same saved rstd. Returns the number
    of elements accepted by the cancellation clause (dx, dz, dgamma)."""
    T, D = x.shape
    fmt = _FMT[x.dtype]
    r64 = to_f64(rstd)
    if variant == "fused":
        gr = None if g_res is None else to_f64(g_res)
        dx_ref, dw_ref, diag = oracle.fused_add_bwd(to_f64(g), to_f64(x), to_f64(res), to_f64(w), r64, gr, zc,
                                                    diagnostics=True, fmt=fmt)
    elif variant == "gated":
        dx_ref, dz_ref, dw_ref, diag = oracle.gated_bwd(to_f64(g), to_f64(x), to_f64(z), to_f64(w), r64, zc,
                                                        diagnostics=True, gate=gate, fmt=fmt)
    else:
        gr = None if g_res is None else to_f64(g_res)
        dx_ref, dw_ref, diag = oracle.rmsnorm_bwd(to_f64(g), to_f64(x), to_f64(w), r64, zc, g_res=gr,
                                                  diagnostics=True, fmt=fmt)
    n2 = assert_bf16_parity(f"{name} dx", to_f64(out["dx"]), dx_ref, diag["dx_pre"], diag["dx_scale"], fmt=fmt)
    if variant == "gated":
        n2 += assert_bf16_parity(f"{name} dz", to_f64(out["dz"]), dz_ref, diag["dz_pre"], diag["dz_scale"],
                                 fmt=fmt)
    C, n = chunk_rows_hint(T, D)
    n2 += assert_dgamma_parity(f"{name} dgamma", to_f64(out["dgamma"]), dw_ref, diag["dw_abs"], C, n)
    return n2
