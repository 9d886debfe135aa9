"""The allocation-free backward entry point (rmsnorm_bwd_noalloc).

It is meant for callers that cannot call cudaMalloc — code that may only use
the tensors it is given, or a runtime whose device footprint must not grow
after start-up — so it keeps the weight-gradient scratch in a fixed array in
the library's device image instead of a caller workspace. This test calls it
through the C ABI and checks that its dx and dgamma equal those of the regular
rmsnorm_bwd (caller workspace) on the same inputs, bit for bit, on consecutive
calls of different sizes: one that fills the whole array exactly
(T = 32768, D = 8192: 1024 chunks of 32 rows x 8192 x 4 bytes = 32 MiB), one
that uses part of it, and smaller ones that follow them and find their
leftovers. A problem one chunk past the array is refused. This file is collected last so that a failure here cannot
hide the results of the other GPU tests.
"""
from __future__ import annotations

import pytest
import torch

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


def _inputs(T, D, seed, zc):
    x = synth.normal_bf16((T, D), seed, DEV)
    g = synth.normal_bf16((T, D), seed + 1, DEV)
    w = synth.gamma_f32(D, seed + 2, DEV, mean=0.0 if zc else 1.0, std=0.1)
    y = torch.empty_like(x)
    rstd = torch.empty(T, device=DEV)
    rn.rmsnorm_fwd(x, w, y, rstd, 1e-6, zc)
    return g, x, w, rstd


LIMIT = 32 << 20  # RMSN_NOALLOC_SCRATCH_BYTES


def test_noalloc_backward_matches_workspace_backward():
    # T = 32768 at D = 8192 fills the array exactly; at D = 4096 (27-row chunks:
    # 1214 partial rows) it takes 19.9 MB of it.
    assert rn.workspace_bytes(32768, 8192) == LIMIT
    assert 16 << 20 < rn.workspace_bytes(32768, 4096) <= LIMIT
    cases = [(4096, 4096, 1, False), (32768, 8192, 4, False), (32768, 4096, 2, False), (100, 2048, 3, True)]
    for T, D, seed, zc in cases:
        g, x, w, rstd = _inputs(T, D, seed, zc)
        dx_ref = torch.empty_like(x)
        dg_ref = torch.empty(D, device=DEV)
        ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=DEV)
        rn.rmsnorm_bwd(g, x, w, rstd, dx_ref, dg_ref, ws, zc)
        dx = torch.full_like(x, 5.0)
        dg = torch.full((D,), 5.0, device=DEV)
        rn.rmsnorm_bwd_noalloc(g, x, w, rstd, dx, dg, zc)
        torch.cuda.synchronize()
        assert torch.equal(dx.view(torch.int16), dx_ref.view(torch.int16)), f"dx differs at T={T} D={D}"
        assert torch.equal(dg.view(torch.int32), dg_ref.view(torch.int32)), f"dgamma differs at T={T} D={D}"


def test_noalloc_refuses_problems_larger_than_its_array():
    D, T = 4096, 100000  # 30-row chunks: 3334 partial rows, 54.6 MB
    assert rn.workspace_bytes(T, D) > LIMIT
    x = torch.zeros((T, D), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(D, device=DEV)
    rstd = torch.ones(T, device=DEV)
    dg = torch.empty(D, device=DEV)
    with pytest.raises(rn.RmsNormError) as err:
        rn.rmsnorm_bwd_noalloc(x, x, w, rstd, x.clone(), dg, False)
    assert err.value.status == -5
    with pytest.raises(rn.RmsNormError) as err:
        rn.rmsnorm_bwd_noalloc(x[:8], x[:8], w, rstd[:8], x[:8].clone(), None, False)
    assert err.value.status == -1
    # one chunk past the array at D = 8192
    D, T = 8192, 32769
    assert rn.workspace_bytes(T, D) == LIMIT + D * 4
    x = torch.zeros((T, D), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(D, device=DEV)
    rstd = torch.ones(T, device=DEV)
    dg = torch.empty(D, device=DEV)
    with pytest.raises(rn.RmsNormError) as err:
        rn.rmsnorm_bwd_noalloc(x, x, w, rstd, torch.empty_like(x), dg, False)
    assert err.value.status == -5
