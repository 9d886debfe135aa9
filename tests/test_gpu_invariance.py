"""Batch invariance: one fixed anchor row gives bitwise-identical y, rstd, dx
(and dz) whatever batch it sits in — batch size T in {1,2,17,33,128,257,1000,
1024}, position first / middle / last / shuffled, fresh neighbours, zero padding
rows, a different row stride — and across repeated runs.

Rows wider than 8192 (12296, 16384, and 9216 in the plain mode) run their
backward on CTA pairs, whose chunk assignment changes with T; their rows are
held to the same bar.

Methodology from Expose Batch Invariant Kernels (TransformerEngine issue 2986:
anchor row at several offsets in batches of different M, output bytes compared
exactly) and from the zero-centred RMSNorm PR (RL-Kernel pull request 467:
bitwise gates under batch-size, chunk, padding and permutation transforms).
"""
from __future__ import annotations

import pytest
import torch

from invariant_rmsnorm_gb300 import synth
from tests.gpu_common import DEV, check_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).clone()


@pytest.mark.parametrize("variant,D", [("plain", 4096), ("residual", 4096), ("gated", 128), ("plain", 7168),
                                       ("plain", 128), ("residual", 12296), ("gated", 16384), ("plain", 9216)])
def test_anchor_row_bitwise_across_batches(variant, D):
    zc = variant == "gated"
    anchor_x = synth.normal_bf16((D,), 100, DEV)
    anchor_g = synth.normal_bf16((D,), 101, DEV)
    anchor_z = synth.normal_bf16((D,), 102, DEV)
    anchor_gr = synth.normal_bf16((D,), 103, DEV)
    w = synth.gamma_f32(D, 104, DEV, mean=0.0 if zc else 1.0, std=0.1)
    ref = None
    n_cases = 0
    for T in synth.INVARIANCE_T:
        for pos in synth.INVARIANCE_POSITIONS:
            seed = 1000 + 10 * T + synth.INVARIANCE_POSITIONS.index(pos)
            x, g, idx = synth.invariance_batch(anchor_x, anchor_g, T, pos, seed)
            z = gr = None
            if variant == "gated":
                z = synth.normal_bf16((T, D), seed + 7, DEV)
                z[idx] = anchor_z
            if variant == "residual":
                gr = synth.normal_bf16((T, D), seed + 8, DEV)
                gr[idx] = anchor_gr
            for ld in (None, D + 64):   # also a different padding layout (row stride)
                xx = x if ld is None else synth.strided(x, ld)
                fo = run_fwd(variant, xx, w, 1e-6, zc, z=z)
                bo = run_bwd(variant, g, xx, w, fo["rstd"], zc, z=z, g_res=gr)
                got = {"y": _bits(fo["y"][idx]), "rstd": fo["rstd"][idx].view(torch.int32).clone(),
                       "dx": _bits(bo["dx"][idx])}
                if variant == "gated":
                    got["dz"] = _bits(bo["dz"][idx])
                if variant == "residual":
                    got["x_copy"] = _bits(fo["x_copy"][idx])
                if ref is None:
                    ref = got
                    # the anchor itself matches the oracle
                    torch.cuda.synchronize()
                    check_fwd(variant, xx[idx:idx + 1], w, 1e-6, zc, {k: v[idx:idx + 1] for k, v in fo.items()},
                              z=None if z is None else z[idx:idx + 1], name="anchor")
                for k in ref:
                    assert torch.equal(got[k], ref[k]), f"{variant} D={D}: anchor {k} differs at T={T} pos={pos} ld={ld}"
                n_cases += 1
    assert n_cases == len(synth.INVARIANCE_T) * len(synth.INVARIANCE_POSITIONS) * 2


def test_prefix_and_slice_invariance():
    """Rows computed in a batch of 512 equal the same rows computed as prefixes
    n in {1,2,8,16,32,48,64,256} and as the x[3:5] / x[:1] slices (RL-Kernel pull
    request 467, prefix-slice probes)."""
    D = 2048
    x = synth.normal_bf16((512, D), 7, DEV)
    g = synth.normal_bf16((512, D), 8, DEV)
    w = synth.gamma_f32(D, 9, DEV, mean=0.0, std=0.1)
    full_f = run_fwd("plain", x, w, 1e-6, True)
    full_b = run_bwd("plain", g, x, w, full_f["rstd"], True)
    for sl in [slice(0, n) for n in (1, 2, 8, 16, 32, 48, 64, 256)] + [slice(3, 5), slice(0, 1)]:
        f = run_fwd("plain", x[sl], w, 1e-6, True)
        b = run_bwd("plain", g[sl], x[sl], w, f["rstd"], True)
        assert torch.equal(_bits(f["y"]), _bits(full_f["y"][sl]))
        assert torch.equal(_bits(b["dx"]), _bits(full_b["dx"][sl]))


def test_repeated_runs_bitwise():
    wl = synth.residual(DEV, seed=4, T=4096, D=4096)
    outs = []
    for _ in range(3):
        fo = run_fwd("residual", wl.x, wl.w, wl.eps, False)
        bo = run_bwd("residual", wl.g, wl.x, wl.w, fo["rstd"], False, g_res=wl.g_res)
        outs.append((_bits(fo["y"]), fo["rstd"].clone(), _bits(bo["dx"]), bo["dgamma"].clone()))
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1])
        assert torch.equal(o[2], outs[0][2]) and torch.equal(o[3].view(torch.int32), outs[0][3].view(torch.int32))
