"""dx and y, bit for bit against float32 models of their stated arithmetic.

The backward's row sum s = sum_i (g_i w_i) x_i goes through the fixed tree
(Megatron-LM pull request 6859, items 1-2; RL-Kernel pull request 414,
Implementation: ascending fp32 reductions, separately rounded operations):
each consumer thread adds its elements in order, a warp (or lane-group)
butterfly, the warp totals in order. dx = ((g w) r) - x (((r^3)/D) s) [+ g_res]
with every operation rounded to fp32 and one rounding to the activation format.
The forward's y = (x r) w with the saved rstd r (its rsqrt is the hardware's,
so r is taken from the kernel rather than modelled). The models are in
tests/_helpers.py (row_sums_model, dx_model); the gated mode is left out
because its gate uses the hardware exponential.

Widths cover the narrow lane groups and every wide launch shape, including
the first width past each shape boundary.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import synth
from tests._helpers import dx_model, f32_round_act
from tests.gpu_common import DEV, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

WIDTHS = [8, 40, 128, 200, 256, 264, 1000, 2048, 2056, 4096, 4104, 7168, 7176, 8192, 8200, 16384]


def _f32(t):
    return t.detach().float().cpu().numpy().astype(np.float32)


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


@pytest.mark.parametrize("variant", ["plain", "residual", "fused"])
@pytest.mark.parametrize("D", WIDTHS)
def test_dx_and_y_bits(D, variant):
    T = 77 if D <= 4096 else 23
    seed = 3 * D + len(variant)
    rng = np.random.default_rng(seed)
    dtype = torch.float16 if rng.integers(0, 2) else torch.bfloat16
    fmt = "f16" if dtype == torch.float16 else "bf16"
    zc = bool(rng.integers(0, 2))
    x = synth.normal16((T, D), seed, DEV, dtype=dtype)
    g = synth.normal16((T, D), seed + 1, DEV, dtype=dtype)
    w = synth.gamma_f32(D, seed + 2, DEV, mean=0.0 if zc else 1.0, std=0.1)
    gr = synth.normal16((T, D), seed + 3, DEV, dtype=dtype) if variant in ("residual", "fused") else None
    res = synth.normal16((T, D), seed + 4, DEV, std=4.0, dtype=dtype) if variant == "fused" else None
    fo = run_fwd(variant, x, w, 1e-6, zc, res=res, ex=True)
    bo = run_bwd(variant, g, x, w, fo["rstd"], zc, g_res=gr, res=res, ex=True)
    torch.cuda.synchronize()
    w_eff = _f32(w)
    if zc:
        w_eff = w_eff + np.float32(1.0)
    h = _f32(x) if variant != "fused" else _f32(x) + _f32(res)
    r = _f32(fo["rstd"])
    want_y = f32_round_act((h * r[:, None]) * w_eff[None, :], fmt)
    want_dx = dx_model(_f32(g), h, w_eff, r, variant, None if gr is None else _f32(gr), fmt)
    name = f"{variant} D={D} {dtype} zc={zc}"
    for what, got, want in (("y", _f32(fo["y"]), want_y), ("dx", _f32(bo["dx"]), want_dx)):
        bad = np.flatnonzero(_bits(got) != _bits(want))
        assert bad.size == 0, f"{name}: {what} differs at {bad.size} elements, first {bad[:4].tolist()}"
    if variant == "fused":
        assert np.array_equal(_bits(_f32(fo["res_out"])), _bits(f32_round_act(h, fmt))), name
