"""GPU parity of fused add + RMSNorm (the decoder-norm path of the zero-centred
RMSNorm PR, RL-Kernel pull request 467: normalise the fp32 sum x + res and
return it) against the float64 oracle, plus batch invariance of its rows.

Tolerances as in test_gpu_parity; the returned bf16 sum is deterministic
(one fp32 add, one bf16 rounding) and must match the oracle bit for bit.
"""
from __future__ import annotations

import pytest
import torch

from invariant_rmsnorm_gb300 import synth
from tests.gpu_common import DEV, check_bwd, check_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def _case(T, D, seed, zc=False, with_gres=True, ld_in=None, ld_out=None, name=""):
    x = synth.normal_bf16((T, D), seed, DEV)
    res = synth.normal_bf16((T, D), seed + 1, DEV, std=4.0)   # residual stream larger than the update
    g = synth.normal_bf16((T, D), seed + 2, DEV)
    gr = synth.normal_bf16((T, D), seed + 3, DEV) if with_gres else None
    w = synth.gamma_f32(D, seed + 4, DEV, mean=0.0 if zc else 1.0, std=0.1)
    if ld_in is not None:
        x, res = synth.strided(x, ld_in), synth.strided(res, ld_in + 8)
        g = synth.strided(g, ld_in + 16)
        gr = synth.strided(gr, ld_in + 24) if gr is not None else None
    fo = run_fwd("fused", x, w, 1e-6, zc, res=res, ld_out=ld_out)
    bo = run_bwd("fused", g, x, w, fo["rstd"], zc, g_res=gr, res=res, ld_out=ld_out)
    torch.cuda.synchronize()
    check_fwd("fused", x, w, 1e-6, zc, fo, res=res, name=name)
    check_bwd("fused", g, x, w, fo["rstd"], zc, bo, g_res=gr, res=res, name=name)
    return fo, bo


@pytest.mark.parametrize("with_gres", [True, False])
@pytest.mark.parametrize("D,T", [(D, T) for D in (8, 128, 256, 264, 2048, 4096, 7168) for T in (1, 70, 333)]
                         + [(14528, 40), (16384, 33)])
def test_fused_add_shapes(D, T, with_gres):
    _case(T, D, seed=D + 3 * T, with_gres=with_gres, name=f"fused T={T} D={D}")


@pytest.mark.parametrize("D", [128, 2048])
def test_fused_add_zero_centred_and_strided(D):
    _case(77, D, seed=5, zc=True, ld_in=D + 64, ld_out=D + 8, name="fused zc strided")


def test_fused_add_decoder_size():
    """Qwen3-Next decoder norm shape: 32768 tokens x hidden 2048, full comparison;
    the weight gradient is bitwise reproducible."""
    fo, bo = _case(32768, 2048, seed=11, name="fused 32768x2048")
    x = synth.normal_bf16((32768, 2048), 11, DEV)
    res = synth.normal_bf16((32768, 2048), 12, DEV, std=4.0)
    g = synth.normal_bf16((32768, 2048), 13, DEV)
    gr = synth.normal_bf16((32768, 2048), 14, DEV)
    w = synth.gamma_f32(2048, 15, DEV, mean=1.0, std=0.1)
    b2 = run_bwd("fused", g, x, w, fo["rstd"], False, g_res=gr, res=res)
    b3 = run_bwd("fused", g, x, w, fo["rstd"], False, g_res=gr, res=res)
    torch.cuda.synchronize()
    assert torch.equal(b2["dgamma"].view(torch.int32), b3["dgamma"].view(torch.int32))


def test_fused_add_zero_residual_is_plain_norm():
    """res = 0: y and rstd equal the plain forward bit for bit; res_out == x."""
    x = synth.normal_bf16((300, 4096), 21, DEV)
    w = synth.gamma_f32(4096, 22, DEV)
    fo = run_fwd("fused", x, w, 1e-6, False, res=torch.zeros_like(x))
    po = run_fwd("plain", x, w, 1e-6, False)
    torch.cuda.synchronize()
    assert torch.equal(fo["y"].view(torch.int16), po["y"].view(torch.int16))
    assert torch.equal(fo["rstd"], po["rstd"]) and torch.equal(fo["res_out"], x)


@pytest.mark.parametrize("D", [2048, 128])
def test_fused_add_anchor_row_batch_invariant(D):
    ax, ar = synth.normal_bf16((D,), 31, DEV), synth.normal_bf16((D,), 32, DEV, std=4.0)
    ag, agr = synth.normal_bf16((D,), 33, DEV), synth.normal_bf16((D,), 34, DEV)
    w = synth.gamma_f32(D, 35, DEV)
    ref = None
    for T in synth.INVARIANCE_T:
        for pos in synth.INVARIANCE_POSITIONS:
            seed = 500 + 10 * T + synth.INVARIANCE_POSITIONS.index(pos)
            x, g, idx = synth.invariance_batch(ax, ag, T, pos, seed)
            res = synth.normal_bf16((T, D), seed + 5, DEV, std=4.0)
            gr = synth.normal_bf16((T, D), seed + 6, DEV)
            res[idx], gr[idx] = ar, agr
            fo = run_fwd("fused", x, w, 1e-6, False, res=res)
            bo = run_bwd("fused", g, x, w, fo["rstd"], False, g_res=gr, res=res)
            got = [fo["y"][idx].view(torch.int16).clone(), fo["res_out"][idx].view(torch.int16).clone(),
                   fo["rstd"][idx].view(torch.int32).clone(), bo["dx"][idx].view(torch.int16).clone()]
            if ref is None:
                ref = got
            for a, b in zip(got, ref):
                assert torch.equal(a, b), f"anchor differs at T={T} pos={pos}"
