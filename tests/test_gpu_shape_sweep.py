"""Seeded sweep over row widths and batch sizes.

The kernels pick their launch shape from D alone (narrow lane groups of 1 to
32 lanes, wide rows of 1, 2 or 4 vectors per thread on 224, 256 or 512
threads) and from the mode (which fixes registers and CTAs per SM). This
sweep draws widths across the whole supported range, 8 to 16384 in steps of
8, with ragged batch sizes, and checks every variant in both activation
formats against the oracle: outputs within one ulp (or the cancellation
bound), rstd within 1e-5 relative, the weight gradient within 1e-4 relative
(or the fixed tree's bound). Widths at each launch-shape boundary are
always included.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from invariant_rmsnorm_gb300 import synth
from tests.gpu_common import DEV, check_bwd, check_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

# Boundaries of the launch shapes (in elements): narrow groups (<= 256), wide
# VPT 1 (<= 2048 at 256 threads), VPT 2 (<= 4096), VPT 4 on <= 224 threads
# (<= 7168), then up to 8192 the forward's VPT 4 on 256 threads and the
# backward's VPT 2 on 512; beyond, the forward's VPT 4 on 512 threads and the
# backward on CTA pairs (the plain mode up to 9216, then VPT 4 on 512 threads).
BOUNDARY_D = [8, 16, 136, 256, 264, 2048, 2056, 4096, 4104, 7168, 7176, 8192, 8200, 9216, 9224, 16384]


def _draws(n, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        D = int(rng.integers(1, 2049)) * 8
        T = int(rng.integers(1, 200)) if D <= 4096 else int(rng.integers(1, 60))
        out.append((D, T))
    return out


CASES = [(D, 37 if D <= 4096 else 19) for D in BOUNDARY_D] + _draws(24)
VARIANTS = ["plain", "residual", "gated", "fused"]


@pytest.mark.parametrize("D,T", CASES)
def test_shape_sweep(D, T):
    rng = np.random.default_rng(D * 7919 + T)
    variant = VARIANTS[int(rng.integers(0, 4))]
    dtype = torch.float16 if rng.integers(0, 2) else torch.bfloat16
    gate = "sigmoid" if rng.integers(0, 2) else "silu"
    zc = bool(rng.integers(0, 2))
    seed = int(rng.integers(0, 1 << 20))
    x = synth.normal16((T, D), seed, DEV, dtype=dtype)
    g = synth.normal16((T, D), seed + 1, DEV, dtype=dtype)
    w = synth.gamma_f32(D, seed + 2, DEV, mean=0.0 if zc else 1.0, std=0.1)
    z = synth.normal16((T, D), seed + 3, DEV, std=2.0, dtype=dtype) if variant == "gated" else None
    gr = synth.normal16((T, D), seed + 4, DEV, dtype=dtype) if variant in ("residual", "fused") else None
    res = synth.normal16((T, D), seed + 5, DEV, std=4.0, dtype=dtype) if variant == "fused" else None
    name = f"{variant} {dtype} {gate} zc={zc} T={T} D={D}"
    fo = run_fwd(variant, x, w, 1e-6, zc, z=z, res=res, ex=True, gate=gate)
    bo = run_bwd(variant, g, x, w, fo["rstd"], zc, z=z, g_res=gr, res=res, ex=True, gate=gate)
    torch.cuda.synchronize()
    check_fwd(variant, x, w, 1e-6, zc, fo, z=z, res=res, gate=gate, name=name)
    check_bwd(variant, g, x, w, fo["rstd"], zc, bo, z=z, g_res=gr, res=res, gate=gate, name=name)


@pytest.mark.parametrize("D,T", _draws(12, seed=77) + [(7168, 21), (8192, 13), (16384, 9)])
def test_shape_sweep_strided_recompute(D, T):
    """Random widths with padded row strides on every input and output, through
    the recompute backward: its y is the forward's bit for bit, its dx and
    weight gradient the plain backward's, and the pad columns stay untouched."""
    import invariant_rmsnorm_gb300 as rn
    from tests.gpu_common import empty_act
    rng = np.random.default_rng(D + 31 * T)
    dtype = torch.float16 if rng.integers(0, 2) else torch.bfloat16
    zc = bool(rng.integers(0, 2))
    ld_in, ld_out = D + 8 * int(rng.integers(1, 9)), D + 8 * int(rng.integers(1, 9))
    x = synth.strided(synth.normal16((T, D), D, DEV, dtype=dtype), ld_in)
    g = synth.strided(synth.normal16((T, D), D + 1, DEV, dtype=dtype), ld_in + 8)
    gr = synth.strided(synth.normal16((T, D), D + 2, DEV, dtype=dtype), ld_in + 16)
    w = synth.gamma_f32(D, D + 3, DEV, mean=0.0 if zc else 1.0, std=0.1)
    fo = run_fwd("plain", x, w, 1e-6, zc, ld_out=ld_out, ex=True)
    ref = run_bwd("residual", g, x, w, fo["rstd"], zc, g_res=gr, ld_out=ld_out, ex=True)
    y = empty_act(T, D, ld_out, fill=5.0, dtype=dtype)
    dx = empty_act(T, D, ld_out, fill=5.0, dtype=dtype)
    dg = torch.empty(D, device=DEV)
    ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=DEV)
    rn.rmsnorm_bwd_recompute_ex(g, x, w, fo["rstd"], gr, dx, dg, y, ws, zc)
    torch.cuda.synchronize()
    bits = lambda t: t.contiguous().view(torch.int16)
    assert torch.equal(bits(y), bits(fo["y"])) and torch.equal(bits(dx), bits(ref["dx"]))
    assert torch.equal(dg.view(torch.int32), ref["dgamma"].view(torch.int32))
    for t in (y, dx):  # the pad columns of the padded outputs are untouched
        full = t.as_strided((T, ld_out), (ld_out, 1))
        assert torch.all(full[:, D:].float() == 5.0)
    name = f"strided {dtype} zc={zc} T={T} D={D}"
    check_fwd("plain", x, w, 1e-6, zc, fo, name=name)
    check_bwd("residual", g, x, w, fo["rstd"], zc, ref, g_res=gr, name=name)
