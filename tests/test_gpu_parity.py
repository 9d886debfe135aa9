"""GPU parity: the sm_103a kernels against the float64 oracle, element by element.

Tolerances (from the arithmetic): bf16 outputs within 1 bf16 ulp of the
oracle's correctly rounded value, or — only for outputs whose terms cancel —
within 1/2 ulp + 96 * 2^-24 * (magnitude of the terms); fp32 rstd within 1e-5
relative; fp32 weight gradient within 1e-4 relative, or within the fixed
reduction tree's forward-error bound for columns whose sum cancels.
Every input is seeded and synthetic (invariant_rmsnorm_gb300.synth).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from invariant_rmsnorm_gb300 import synth
from tests._helpers import assert_bf16_parity, assert_dgamma_parity, assert_rel, to_f64
from tests.gpu_common import DEV, check_bwd, check_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

VARIANTS = ("plain", "residual", "gated")


def _inputs(variant, T, D, seed, zc=None, ld_in=None):
    zc = (variant == "gated") if zc is None else zc
    x = synth.normal_bf16((T, D), seed, DEV)
    g = synth.normal_bf16((T, D), seed + 1, DEV)
    w = synth.gamma_f32(D, seed + 2, DEV, mean=0.0 if zc else 1.0, std=0.1 if zc else 0.2)
    z = synth.normal_bf16((T, D), seed + 3, DEV) if variant == "gated" else None
    gr = synth.normal_bf16((T, D), seed + 4, DEV) if variant == "residual" else None
    if ld_in is not None:
        x = synth.strided(x, ld_in)
        g = synth.strided(g, ld_in + 8)
        z = synth.strided(z, ld_in + 16) if z is not None else None
        gr = synth.strided(gr, ld_in + 24) if gr is not None else None
    return dict(x=x, g=g, w=w, z=z, g_res=gr, zc=zc)


def _full_check(variant, T, D, seed, eps=1e-6, ld_in=None, ld_out=None, name=""):
    a = _inputs(variant, T, D, seed, ld_in=ld_in)
    fo = run_fwd(variant, a["x"], a["w"], eps, a["zc"], z=a["z"], ld_out=ld_out)
    bo = run_bwd(variant, a["g"], a["x"], a["w"], fo["rstd"], a["zc"], z=a["z"], g_res=a["g_res"], ld_out=ld_out)
    torch.cuda.synchronize()
    check_fwd(variant, a["x"], a["w"], eps, a["zc"], fo, z=a["z"], name=name)
    return check_bwd(variant, a["g"], a["x"], a["w"], fo["rstd"], a["zc"], bo, z=a["z"], g_res=a["g_res"],
                     name=name)


# ---------------------------------------------------------------------------
# Config: tiny plain RMSNorm, T=16, D=128, zero_centered_gamma False / True
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("zc", [False, True])
def test_tiny_plain(zc):
    wl = synth.tiny_plain(DEV, seed=0, zero_centered_gamma=zc)
    fo = run_fwd("plain", wl.x, wl.w, wl.eps, zc)
    bo = run_bwd("plain", wl.g, wl.x, wl.w, fo["rstd"], zc)
    torch.cuda.synchronize()
    check_fwd("plain", wl.x, wl.w, wl.eps, zc, fo, name="tiny")
    check_bwd("plain", wl.g, wl.x, wl.w, fo["rstd"], zc, bo, name="tiny")


def test_zero_centred_differs_and_equals_offset_weight():
    """y(zc=True, w) == y(zc=False, fp32 w+1) bitwise, and differs from y(zc=False, w)."""
    wl = synth.tiny_plain(DEV, seed=3, zero_centered_gamma=True, T=64, D=4096)
    a = run_fwd("plain", wl.x, wl.w, wl.eps, True)
    b = run_fwd("plain", wl.x, wl.w + 1.0, wl.eps, False)
    c = run_fwd("plain", wl.x, wl.w, wl.eps, False)
    assert torch.equal(a["y"].view(torch.int16), b["y"].view(torch.int16))
    assert (a["y"].float() - c["y"].float()).abs().max().item() > 0.5


# ---------------------------------------------------------------------------
# Shapes: several tiles and a ragged tail, narrow to maximum D
# ---------------------------------------------------------------------------
SHAPES = [(D, T) for D in (8, 24, 128, 200, 256, 264, 512, 1032, 2048, 4096, 7168)
          for T in (1, 70, 333)] + [(8192, 1), (8192, 70), (16384, 1), (16384, 45),
                                    (8200, 33), (9216, 5), (12296, 64)]  # CTA pairs; 12296: unequal halves


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("D,T", SHAPES)
def test_shapes(variant, D, T):
    _full_check(variant, T, D, seed=D + T, name=f"{variant} T={T} D={D}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("D", [128, 4096, 9216])
def test_strided_rows(variant, D):
    """Row strides larger than D on every input and output; the gap columns of the
    outputs must be left untouched."""
    T = 77
    n2 = _full_check(variant, T, D, seed=7, ld_in=D + 64, ld_out=D + 8, name=f"strided {variant}")
    assert n2 >= 0
    fo = run_fwd(variant, synth.strided(synth.normal_bf16((T, D), 1, DEV), D + 40),
                 synth.gamma_f32(D, 2, DEV), 1e-6, False,
                 z=synth.normal_bf16((T, D), 3, DEV) if variant == "gated" else None, ld_out=D + 8)
    torch.cuda.synchronize()
    base = fo["y"].as_strided((T, D + 8), (D + 8, 1))
    assert torch.all(base[:, D:] == 3.0), "a kernel wrote outside the rows"


# ---------------------------------------------------------------------------
# Config: rmsnorm_residual fwd+bwd at T=32768, D=4096 (the benchmark's workload)
# ---------------------------------------------------------------------------
def test_residual_full_size():
    wl = synth.residual(DEV, seed=0)
    fo = run_fwd("residual", wl.x, wl.w, wl.eps, False)
    bo = run_bwd("residual", wl.g, wl.x, wl.w, fo["rstd"], False, g_res=wl.g_res)
    torch.cuda.synchronize()
    check_fwd("residual", wl.x, wl.w, wl.eps, False, fo, name="residual 32768x4096")
    n2 = check_bwd("residual", wl.g, wl.x, wl.w, fo["rstd"], False, bo, g_res=wl.g_res,
                   name="residual 32768x4096")
    print(f"residual full size: {n2} elements accepted by the cancellation clause")
    # run-to-run bitwise, and the split pass-2 entry point gives the same bits
    bo2 = run_bwd("residual", wl.g, wl.x, wl.w, fo["rstd"], False, g_res=wl.g_res, split=True)
    torch.cuda.synchronize()
    assert torch.equal(bo2["dgamma"].view(torch.int32), bo["dgamma"].view(torch.int32))
    assert torch.equal(bo2["dx"].view(torch.int16), bo["dx"].view(torch.int16))


# ---------------------------------------------------------------------------
# Config: gated zero-centred (Qwen3-Next), 262144 rows x 128
# ---------------------------------------------------------------------------
def test_gated_full_size():
    wl = synth.gated(DEV, seed=0)
    fo = run_fwd("gated", wl.x, wl.w, wl.eps, True, z=wl.z)
    bo = run_bwd("gated", wl.g, wl.x, wl.w, fo["rstd"], True, z=wl.z)
    torch.cuda.synchronize()
    check_fwd("gated", wl.x, wl.w, wl.eps, True, fo, z=wl.z, name="gated 262144x128")
    check_bwd("gated", wl.g, wl.x, wl.w, fo["rstd"], True, bo, z=wl.z, name="gated 262144x128")
    bo2 = run_bwd("gated", wl.g, wl.x, wl.w, fo["rstd"], True, z=wl.z)
    torch.cuda.synchronize()
    assert torch.equal(bo2["dgamma"].view(torch.int32), bo["dgamma"].view(torch.int32))


# ---------------------------------------------------------------------------
# Config: large sweep with outliers; 4096 sampled rows (y, rstd, dx) and every
# weight-gradient column vs the oracle, and the weight gradient run-to-run bitwise
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,D", [(131072, 2048), (131072, 4096), (131072, 7168), (131072, 8192),
                                 (262144, 4096)])
def test_large_sweep(T, D):
    import oracle
    wl = synth.large(DEV, seed=1, T=T, D=D)
    fo = run_fwd("plain", wl.x, wl.w, wl.eps, False)
    bo = run_bwd("plain", wl.g, wl.x, wl.w, fo["rstd"], False)
    bo2 = run_bwd("plain", wl.g, wl.x, wl.w, fo["rstd"], False)
    torch.cuda.synchronize()
    assert torch.equal(bo2["dgamma"].view(torch.int32), bo["dgamma"].view(torch.int32)), "dgamma not bitwise"
    assert torch.equal(bo2["dx"].view(torch.int16), bo["dx"].view(torch.int16))
    gen = torch.Generator().manual_seed(T + D)
    rows = torch.cat([torch.tensor([0, T - 1]), torch.randint(0, T, (4094,), generator=gen)]).to(DEV)
    sub = {k: v.index_select(0, rows) for k, v in (("x", wl.x), ("g", wl.g), ("y", fo["y"]),
                                                     ("rstd", fo["rstd"]), ("dx", bo["dx"]))}
    y_ref, r_ref = oracle.rmsnorm_fwd(to_f64(sub["x"]), to_f64(wl.w), wl.eps, False)
    assert_rel("large rstd", to_f64(sub["rstd"]), r_ref, 1e-5)
    assert_bf16_parity("large y", to_f64(sub["y"]), y_ref)
    dx_ref, _, diag = oracle.rmsnorm_bwd(to_f64(sub["g"]), to_f64(sub["x"]), to_f64(wl.w), to_f64(sub["rstd"]),
                                         False, diagnostics=True)
    assert_bf16_parity("large dx", to_f64(sub["dx"]), dx_ref, diag["dx_pre"], diag["dx_scale"])
    # every weight-gradient column against the oracle, over all T rows (in column blocks)
    from tests.gpu_common import chunk_rows_hint
    C, n = chunk_rows_hint(T, D)
    r64 = to_f64(fo["rstd"])
    for c0 in range(0, D, 512):
        dw_ref, dw_abs = oracle.weight_grad(to_f64(wl.g[:, c0:c0 + 512]), to_f64(wl.x[:, c0:c0 + 512]), r64,
                                            with_abs=True)
        assert_dgamma_parity(f"large dgamma [{c0}:{c0 + 512}]", to_f64(bo["dgamma"][c0:c0 + 512]), dw_ref, dw_abs,
                             C, n)


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------
def test_empty_batch_launches_nothing():
    import invariant_rmsnorm_gb300 as rn
    D = 4096
    x = torch.empty((0, D), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(D, device=DEV)
    y = torch.empty((0, D), dtype=torch.bfloat16, device=DEV)
    r = torch.empty(0, device=DEV)
    rn.rmsnorm_fwd(x, w, y, r, 1e-6, False)
    dg = torch.full((D,), 7.0, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    rn.rmsnorm_bwd(x, x, w, r, y, dg, ws, False)
    torch.cuda.synchronize()
    assert torch.all(dg == 7.0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_zero_rows_and_outliers(variant):
    """Zero (padding) rows give r = eps^-1/2 and y = 0; rows with x100 outliers."""
    T, D = 96, 4096 if variant != "gated" else 128
    a = _inputs(variant, T, D, seed=5)
    x = a["x"].clone()
    x[10:20] = 0
    x = synth.with_outliers(x, seed=6, frac=0.01)
    fo = run_fwd(variant, x, a["w"], 1e-6, a["zc"], z=a["z"])
    bo = run_bwd(variant, a["g"], x, a["w"], fo["rstd"], a["zc"], z=a["z"], g_res=a["g_res"])
    torch.cuda.synchronize()
    assert torch.all(fo["y"][10:20] == 0)
    check_fwd(variant, x, a["w"], 1e-6, a["zc"], fo, z=a["z"], name="zero rows")
    check_bwd(variant, a["g"], x, a["w"], fo["rstd"], a["zc"], bo, z=a["z"], g_res=a["g_res"], name="zero rows")


def test_eps_zero_and_large_eps():
    for eps in (0.0, 0.5):
        _full_check("plain", 50, 1024, seed=9, eps=eps, name=f"eps={eps}")


def test_residual_without_residual_gradient_is_plain_bwd():
    a = _inputs("plain", 100, 2048, seed=12)
    fo = run_fwd("plain", a["x"], a["w"], 1e-6, False)
    b1 = run_bwd("plain", a["g"], a["x"], a["w"], fo["rstd"], False)
    b2 = run_bwd("residual", a["g"], a["x"], a["w"], fo["rstd"], False, g_res=None)
    torch.cuda.synchronize()
    assert torch.equal(b1["dx"].view(torch.int16), b2["dx"].view(torch.int16))
    assert torch.equal(b1["dgamma"].view(torch.int32), b2["dgamma"].view(torch.int32))


def test_no_device_wait_ever_timed_out():
    import invariant_rmsnorm_gb300 as rn
    _full_check("residual", 256, 4096, seed=1)
    assert rn.rmsnorm_device_error(clear=True) == 0


@pytest.mark.parametrize("D", [128, 2048])
def test_gated_extreme_gates(D):
    """Gates far out in both tails (|z| up to 100, where exp over- or underflows
    in fp32) and exactly zero: the kernels' sigmoid stays finite and within the
    tolerance of the oracle's double-precision one."""
    T = 96
    a = _inputs("gated", T, D, seed=21)
    zf = torch.linspace(-100.0, 100.0, T * D, device=DEV).reshape(T, D)
    zf[::7] = 0.0
    z = zf[torch.randperm(T, generator=torch.Generator().manual_seed(3)).to(DEV)].to(torch.bfloat16)
    fo = run_fwd("gated", a["x"], a["w"], 1e-6, True, z=z)
    bo = run_bwd("gated", a["g"], a["x"], a["w"], fo["rstd"], True, z=z)
    torch.cuda.synchronize()
    assert torch.isfinite(fo["y"].float()).all() and torch.isfinite(bo["dz"].float()).all()
    check_fwd("gated", a["x"], a["w"], 1e-6, True, fo, z=z, name="extreme gates")
    check_bwd("gated", a["g"], a["x"], a["w"], fo["rstd"], True, bo, z=z, name="extreme gates")
