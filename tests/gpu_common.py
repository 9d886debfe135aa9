"""Helpers for the GPU parity tests: run a variant through the C-ABI binding,
run the oracle on the same inputs, compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import invariant_rmsnorm_gb300 as rn
import oracle
from tests._helpers import assert_bf16_parity, assert_dgamma_parity, assert_rel, to_f64

DEV = torch.device("cuda")


def empty_act(T, D, ld=None, fill=None):
    """A [T, D] bf16 output view; with ``ld`` its rows sit ld apart and the gap
    columns hold ``fill`` so that stray writes can be detected."""
    if ld is None or ld == D:
        return torch.empty((T, D), dtype=torch.bfloat16, device=DEV)
    base = torch.full((max(T, 1), ld), fill if fill is not None else 3.0, dtype=torch.bfloat16, device=DEV)
    return base[:T, :D]


def chunk_rows_hint(T, D):
    n = rn.workspace_bytes(T, D) // (4 * D)
    return T if n <= 1 else -(-T // (n - 1)) - 1, n


def run_fwd(variant, x, w, eps, zc, z=None, ld_out=None, res=None):
    T, D = x.shape
    y = empty_act(T, D, ld_out)
    rstd = torch.empty(T, dtype=torch.float32, device=DEV)
    out = {"y": y, "rstd": rstd}
    if variant == "plain":
        rn.rmsnorm_fwd(x, w, y, rstd, eps, zc)
    elif variant == "residual":
        xc = empty_act(T, D, ld_out)
        rn.rmsnorm_residual_fwd(x, w, y, rstd, xc, eps, zc)
        out["x_copy"] = xc
    elif variant == "gated":
        rn.rmsnorm_gated_fwd(x, z, w, y, rstd, eps, zc)
    elif variant == "fused":
        ro = empty_act(T, D, ld_out)
        rn.rmsnorm_fused_add_fwd(x, res, w, y, rstd, ro, eps, zc)
        out["res_out"] = ro
    else:
        raise ValueError(variant)
    return out


def run_bwd(variant, g, x, w, rstd, zc, z=None, g_res=None, ld_out=None, split=False, res=None):
    T, D = x.shape
    dx = empty_act(T, D, ld_out)
    dg = torch.empty(D, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(rn.workspace_bytes(T, D), 16), dtype=torch.uint8, device=DEV)
    out = {"dx": dx, "dgamma": dg, "ws": ws}
    target = None if split else dg
    if variant == "plain":
        rn.rmsnorm_bwd(g, x, w, rstd, dx, target, ws, zc)
    elif variant == "residual":
        rn.rmsnorm_residual_bwd(g, x, w, rstd, g_res, dx, target, ws, zc)
    elif variant == "gated":
        dz = empty_act(T, D, ld_out)
        rn.rmsnorm_gated_bwd(g, x, z, w, rstd, dx, dz, target, ws, zc)
        out["dz"] = dz
    elif variant == "fused":
        rn.rmsnorm_fused_add_bwd(g, x, res, w, rstd, g_res, dx, target, ws, zc)
    if split:
        rn.rmsnorm_dgamma_reduce(ws, T, D, dg)
    return out


def oracle_fwd(variant, x, w, eps, zc, z=None, res=None):
    if variant == "fused":
        y, r, ro = oracle.fused_add_fwd(to_f64(x), to_f64(res), to_f64(w), eps, zc)
        return y, r
    if variant == "gated":
        y, r = oracle.gated_fwd(to_f64(x), to_f64(z), to_f64(w), eps, zc)
    else:
        y, r = oracle.rmsnorm_fwd(to_f64(x), to_f64(w), eps, zc)
    return y, r


def check_fwd(variant, x, w, eps, zc, out, z=None, name="", res=None):
    y_ref, r_ref = oracle_fwd(variant, x, w, eps, zc, z, res)
    assert_rel(f"{name} rstd", to_f64(out["rstd"]), r_ref, 1e-5)
    assert_bf16_parity(f"{name} y", to_f64(out["y"]), y_ref)
    if variant == "fused":
        _, _, ro = oracle.fused_add_fwd(to_f64(x), to_f64(res), to_f64(w), eps, zc)
        np.testing.assert_array_equal(to_f64(out["res_out"]), ro, err_msg=f"{name} res_out")
    if variant == "residual":
        assert torch.equal(out["x_copy"].view(torch.int16), x.view(torch.int16)), f"{name} x_copy"


def check_bwd(variant, g, x, w, rstd, zc, out, z=None, g_res=None, name="", res=None):
    """Compare against the oracle run with the same saved rstd. Returns the number
    of elements accepted by the cancellation clause (dx, dz, dgamma)."""
    T, D = x.shape
    r64 = to_f64(rstd)
    if variant == "fused":
        gr = None if g_res is None else to_f64(g_res)
        dx_ref, dw_ref, diag = oracle.fused_add_bwd(to_f64(g), to_f64(x), to_f64(res), to_f64(w), r64, gr, zc,
                                                    diagnostics=True)
    elif variant == "gated":
        dx_ref, dz_ref, dw_ref, diag = oracle.gated_bwd(to_f64(g), to_f64(x), to_f64(z), to_f64(w), r64, zc,
                                                        diagnostics=True)
    else:
        gr = None if g_res is None else to_f64(g_res)
        dx_ref, dw_ref, diag = oracle.rmsnorm_bwd(to_f64(g), to_f64(x), to_f64(w), r64, zc, g_res=gr,
                                                  diagnostics=True)
    n2 = assert_bf16_parity(f"{name} dx", to_f64(out["dx"]), dx_ref, diag["dx_pre"], diag["dx_scale"])
    if variant == "gated":
        n2 += assert_bf16_parity(f"{name} dz", to_f64(out["dz"]), dz_ref, diag["dz_pre"], diag["dz_scale"])
    C, n = chunk_rows_hint(T, D)
    n2 += assert_dgamma_parity(f"{name} dgamma", to_f64(out["dgamma"]), dw_ref, diag["dw_abs"], C, n)
    return n2
