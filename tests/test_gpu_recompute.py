"""Backward with recomputation of the forward output (one pass that writes y
again for activation recomputation, instead of a separate forward): the y it
writes is the forward's y bit for bit, and its dx / dz / dgamma are those of
the plain backward bit for bit; the gated recompute is also compared with the
oracle element by element, in both formats and with both gates."""
from __future__ import annotations

import pytest
import torch

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import synth
from tests.gpu_common import DEV, check_bwd, check_fwd, empty_act, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16)


@pytest.mark.parametrize("with_gres", [False, True])
@pytest.mark.parametrize("zc", [False, True])
@pytest.mark.parametrize("D,T", [(128, 333), (200, 70), (2048, 333), (4096, 1000), (7168, 70)])
def test_bwd_recompute_matches_forward_and_backward(D, T, zc, with_gres):
    x = synth.normal_bf16((T, D), D, DEV)
    g = synth.normal_bf16((T, D), D + 1, DEV)
    gr = synth.normal_bf16((T, D), D + 2, DEV) if with_gres else None
    w = synth.gamma_f32(D, D + 3, DEV, mean=0.0 if zc else 1.0, std=0.1)
    fo = run_fwd("plain", x, w, 1e-6, zc)
    ref = run_bwd("residual" if with_gres else "plain", g, x, w, fo["rstd"], zc, g_res=gr)
    dx, dg = torch.empty_like(x), torch.empty(D, device=DEV)
    y = empty_act(T, D, D + 8)
    ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=DEV)
    rn.rmsnorm_bwd_recompute(g, x, w, fo["rstd"], gr, dx, dg, y, ws, zc)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(fo["y"]))
    assert torch.equal(_bits(dx), _bits(ref["dx"]))
    assert torch.equal(dg.view(torch.int32), ref["dgamma"].view(torch.int32))


@pytest.mark.parametrize("D,T", [(128, 1000), (2048, 70)])
def test_gated_bwd_recompute_matches_forward_and_backward(D, T):
    x = synth.normal_bf16((T, D), 1, DEV)
    z = synth.normal_bf16((T, D), 2, DEV)
    g = synth.normal_bf16((T, D), 3, DEV)
    w = synth.gamma_f32(D, 4, DEV, mean=0.0, std=0.1)
    fo = run_fwd("gated", x, w, 1e-6, True, z=z)
    ref = run_bwd("gated", g, x, w, fo["rstd"], True, z=z)
    dx, dz, dw, y = torch.empty_like(x), torch.empty_like(x), torch.empty(D, device=DEV), torch.empty_like(x)
    ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=DEV)
    rn.rmsnorm_gated_bwd_recompute(g, x, z, w, fo["rstd"], dx, dz, dw, y, ws, True)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(fo["y"]))
    assert torch.equal(_bits(dx), _bits(ref["dx"])) and torch.equal(_bits(dz), _bits(ref["dz"]))
    assert torch.equal(dw.view(torch.int32), ref["dgamma"].view(torch.int32))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("gate", ["silu", "sigmoid"])
@pytest.mark.parametrize("D,T", [(128, 1000), (4096, 97)])
def test_recompute_ex_matches_forward_and_backward(D, T, gate, dtype):
    """The *_ex recompute calls, in both activation formats and both gates:
    y bit for bit the *_ex forward's, dx / dz / weight gradient bit for bit the
    *_ex backward's."""
    x, z, g, gr = (synth.normal16((T, D), D + s, DEV, dtype=dtype) for s in (10, 11, 12, 13))
    w = synth.gamma_f32(D, D + 14, DEV, mean=0.0, std=0.1)
    # gated
    fo = run_fwd("gated", x, w, 1e-6, True, z=z, ex=True, gate=gate)
    ref = run_bwd("gated", g, x, w, fo["rstd"], True, z=z, ex=True, gate=gate)
    dx, dz, dw = torch.empty_like(x), torch.empty_like(x), torch.empty(D, device=DEV)
    y = empty_act(T, D, D + 8, dtype=dtype)
    ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=DEV)
    rn.rmsnorm_gated_bwd_recompute_ex(g, x, z, w, fo["rstd"], dx, dz, dw, y, ws, True, gate=gate)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(fo["y"]))
    assert torch.equal(_bits(dx), _bits(ref["dx"])) and torch.equal(_bits(dz), _bits(ref["dz"]))
    assert torch.equal(dw.view(torch.int32), ref["dgamma"].view(torch.int32))
    # plain / residual gradient
    fo = run_fwd("plain", x, w, 1e-6, False, ex=True)
    ref = run_bwd("residual", g, x, w, fo["rstd"], False, g_res=gr, ex=True)
    dx, dg = torch.empty_like(x), torch.empty(D, device=DEV)
    y = empty_act(T, D, D + 8, dtype=dtype)
    rn.rmsnorm_bwd_recompute_ex(g, x, w, fo["rstd"], gr, dx, dg, y, ws, False)
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(fo["y"]))
    assert torch.equal(_bits(dx), _bits(ref["dx"]))
    assert torch.equal(dg.view(torch.int32), ref["dgamma"].view(torch.int32))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("gate", ["silu", "sigmoid"])
@pytest.mark.parametrize("D,T,zc,pad", [(128, 333, True, 0), (64, 1000, False, 8), (200, 70, True, 16),
                                        (2048, 100, True, 0), (4096, 97, False, 24), (7168, 33, True, 8)])
def test_gated_bwd_recompute_against_the_oracle(D, T, zc, pad, gate, dtype):
    """rmsnorm_gated_bwd_recompute (bf16, silu) and rmsnorm_gated_bwd_recompute_ex
    on narrow and wide rows, some with padded row strides: y, the saved rstd it
    reads, dx, dz and the weight gradient each against the oracle's gated
    forward and backward (1 ulp of the activation format, or the cancellation
    clause; dw 1e-4 relative or the fixed tree's bound), not only against the
    gated kernels."""
    x, z, g = (synth.normal16((T, D), D + s, DEV, dtype=dtype) for s in (20, 21, 22))
    if pad:
        x, z, g = (synth.strided(t, D + pad) for t in (x, z, g))
    w = synth.gamma_f32(D, D + 23, DEV, mean=0.0 if zc else 1.0, std=0.1)
    ex = dtype != torch.bfloat16 or gate != "silu"
    fo = run_fwd("gated", x, w, 1e-6, zc, z=z, ex=ex, gate=gate)
    ld_out = D + pad if pad else None
    dx, dz, y = (empty_act(T, D, ld_out, fill=5.0, dtype=dtype) for _ in range(3))
    dw = torch.empty(D, device=DEV)
    ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=DEV)
    if ex:
        rn.rmsnorm_gated_bwd_recompute_ex(g, x, z, w, fo["rstd"], dx, dz, dw, y, ws, zc, gate=gate)
    else:
        rn.rmsnorm_gated_bwd_recompute(g, x, z, w, fo["rstd"], dx, dz, dw, y, ws, zc)
    torch.cuda.synchronize()
    name = f"gated recompute {gate} {dtype} T={T} D={D} zc={zc}"
    check_fwd("gated", x, w, 1e-6, zc, {"y": y, "rstd": fo["rstd"]}, z=z, name=name, gate=gate)
    check_bwd("gated", g, x, w, fo["rstd"], zc, {"dx": dx, "dz": dz, "dgamma": dw}, z=z, name=name, gate=gate)
    if pad:  # the pad columns of the padded outputs are untouched
        for t in (y, dx, dz):
            assert torch.all(t.as_strided((T, D + pad), (D + pad, 1))[:, D:].float() == 5.0)
