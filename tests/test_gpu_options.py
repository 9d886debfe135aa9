"""GPU parity of the activation-format and gate options (the *_ex entry points).

fp16 activations for every variant, and the sigmoid gate of the gated norm in
both formats, against the float64 oracle in the same format: outputs within
one ulp of the oracle's correctly rounded value (or the stated cancellation
bound), rstd within 1e-5 relative, dgamma within 1e-4 relative (or the fixed
tree's forward-error bound). With bf16 and the silu gate the *_ex calls are
bitwise the unsuffixed ones. Batch invariance and run-to-run determinism hold
for the new variants as for the old.

Sources: RL-Kernel pull request 467 "[WS1][CUDA][Qwen3-Next] C1: zero-centred
RMSNorm references and CUDA kernel" (gate activation silu or sigmoid; op
contract tolerances for bf16 and fp16).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from invariant_rmsnorm_gb300 import synth
from tests.gpu_common import DEV, check_bwd, check_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

F16 = torch.float16
BF16 = torch.bfloat16


def _inputs(variant, T, D, seed, dtype, zc, zstd=1.0):
    x = synth.normal16((T, D), seed, DEV, dtype=dtype)
    g = synth.normal16((T, D), seed + 1, DEV, dtype=dtype)
    w = synth.gamma_f32(D, seed + 2, DEV, mean=0.0 if zc else 1.0, std=0.1 if zc else 0.2)
    z = synth.normal16((T, D), seed + 3, DEV, std=zstd, dtype=dtype) if variant == "gated" else None
    gr = synth.normal16((T, D), seed + 4, DEV, dtype=dtype) if variant in ("residual", "fused") else None
    res = synth.normal16((T, D), seed + 5, DEV, std=4.0, dtype=dtype) if variant == "fused" else None
    return dict(x=x, g=g, w=w, z=z, g_res=gr, res=res)


def _run_check(variant, T, D, seed, dtype, zc, gate="silu", name="", eps=1e-6, zstd=1.0):
    a = _inputs(variant, T, D, seed, dtype, zc, zstd)
    fo = run_fwd(variant, a["x"], a["w"], eps, zc, z=a["z"], res=a["res"], ex=True, gate=gate)
    bo = run_bwd(variant, a["g"], a["x"], a["w"], fo["rstd"], zc, z=a["z"], g_res=a["g_res"], res=a["res"],
                 ex=True, gate=gate)
    torch.cuda.synchronize()
    check_fwd(variant, a["x"], a["w"], eps, zc, fo, z=a["z"], res=a["res"], gate=gate, name=name)
    check_bwd(variant, a["g"], a["x"], a["w"], fo["rstd"], zc, bo, z=a["z"], g_res=a["g_res"], res=a["res"],
              gate=gate, name=name)
    return a, fo, bo


# Widths: narrow groups of 8 and 16 lanes (64, 128), a ragged narrow row (200),
# wide rows with one and two vectors per thread (768, 4096) and a non-power-of-two
# width (7168). T spans several stages and chunks with a ragged tail.
DS = [64, 128, 200, 768, 4096, 7168]


@pytest.mark.parametrize("D", DS)
@pytest.mark.parametrize("variant", ["plain", "residual", "gated", "fused"])
def test_f16_parity(variant, D):
    T = 300 if D <= 1024 else 97
    zc = variant == "gated"
    _run_check(variant, T, D, seed=11 + D, dtype=F16, zc=zc, name=f"f16 {variant} D={D}")


@pytest.mark.parametrize("D", [128, 200, 2048, 4096])
@pytest.mark.parametrize("dtype", [BF16, F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("zc", [False, True])
def test_sigmoid_gate_parity(D, dtype, zc):
    T = 300 if D <= 256 else 97
    _run_check("gated", T, D, seed=31 + D, dtype=dtype, zc=zc, gate="sigmoid", name=f"sigmoid {dtype} D={D}",
               zstd=3.0)


@pytest.mark.parametrize("D", [128, 4096])
@pytest.mark.parametrize("dtype", [BF16, F16], ids=["bf16", "f16"])
@pytest.mark.parametrize("gate", ["silu", "sigmoid"])
def test_extreme_gates(D, dtype, gate):
    """Gates across [-100, 100] and exactly zero, in both formats: finite outputs
    within tolerance of the oracle's double-precision gate."""
    T = 96
    a = _inputs("gated", T, D, 21, dtype, True)
    zf = torch.linspace(-100.0, 100.0, T * D, device=DEV).reshape(T, D)
    zf[::7] = 0.0
    z = zf[torch.randperm(T, generator=torch.Generator().manual_seed(3)).to(DEV)].to(dtype)
    fo = run_fwd("gated", a["x"], a["w"], 1e-6, True, z=z, ex=True, gate=gate)
    bo = run_bwd("gated", a["g"], a["x"], a["w"], fo["rstd"], True, z=z, ex=True, gate=gate)
    torch.cuda.synchronize()
    assert torch.isfinite(fo["y"].float()).all() and torch.isfinite(bo["dz"].float()).all()
    check_fwd("gated", a["x"], a["w"], 1e-6, True, fo, z=z, gate=gate, name="extreme gates")
    check_bwd("gated", a["g"], a["x"], a["w"], fo["rstd"], True, bo, z=z, gate=gate, name="extreme gates")


@pytest.mark.parametrize("D", [128, 4096])
@pytest.mark.parametrize("variant", ["plain", "residual", "gated", "fused"])
def test_ex_bf16_is_the_unsuffixed_call(variant, D):
    """dtype bf16 (and gate silu) through *_ex gives the unsuffixed call's bits."""
    T = 200
    zc = variant == "gated"
    a = _inputs(variant, T, D, 5, BF16, zc)
    kw = dict(z=a["z"], res=a["res"])
    f0 = run_fwd(variant, a["x"], a["w"], 1e-6, zc, **kw)
    f1 = run_fwd(variant, a["x"], a["w"], 1e-6, zc, ex=True, **kw)
    b0 = run_bwd(variant, a["g"], a["x"], a["w"], f0["rstd"], zc, g_res=a["g_res"], **kw)
    b1 = run_bwd(variant, a["g"], a["x"], a["w"], f0["rstd"], zc, g_res=a["g_res"], ex=True, **kw)
    torch.cuda.synchronize()
    for k in f0:
        assert torch.equal(_bits(f0[k]), _bits(f1[k])), k
    for k in ("dx", "dgamma") + (("dz",) if variant == "gated" else ()):
        assert torch.equal(_bits(b0[k]), _bits(b1[k])), k


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


@pytest.mark.parametrize("D", [128, 4096])
@pytest.mark.parametrize("case", ["f16-plain", "f16-gated-sigmoid", "bf16-gated-sigmoid"])
def test_batch_invariance_and_determinism(case, D):
    """An anchor row's y, rstd, dx (and dz) bits do not depend on T or its
    position; dgamma is bitwise equal on a repeated call."""
    dt = F16 if case.startswith("f16") else BF16
    variant = "gated" if "gated" in case else "plain"
    gate = "sigmoid" if "sigmoid" in case else "silu"
    zc = variant == "gated"
    anchor = _inputs(variant, 1, D, 77, dt, zc)
    w = anchor["w"]
    ref = None
    for T, pos in ((1, 0), (33, 0), (257, 128), (1000, 999)):
        b = _inputs(variant, T, D, 100 + T, dt, zc)
        b["x"][pos] = anchor["x"][0]
        b["g"][pos] = anchor["g"][0]
        if variant == "gated":
            b["z"][pos] = anchor["z"][0]
        fo = run_fwd(variant, b["x"], w, 1e-6, zc, z=b["z"], ex=True, gate=gate)
        bo = run_bwd(variant, b["g"], b["x"], w, fo["rstd"], zc, z=b["z"], ex=True, gate=gate)
        bo2 = run_bwd(variant, b["g"], b["x"], w, fo["rstd"], zc, z=b["z"], ex=True, gate=gate)
        torch.cuda.synchronize()
        assert torch.equal(bo["dgamma"].view(torch.int32), bo2["dgamma"].view(torch.int32))
        row = [fo["y"][pos].view(torch.int16), fo["rstd"][pos:pos + 1].view(torch.int32),
               bo["dx"][pos].view(torch.int16)]
        if variant == "gated":
            row.append(bo["dz"][pos].view(torch.int16))
        if ref is None:
            ref = [r.clone() for r in row]
        else:
            for r0, r1 in zip(ref, row):
                assert torch.equal(r0, r1), (T, pos)


def test_f16_overflow_and_subnormal_outputs():
    """Outputs beyond the fp16 range become infinite, as the oracle's rounding
    does; outputs in the fp16 subnormal range keep their subnormal bits."""
    D, T = 4096, 4
    x = torch.zeros((T, D), dtype=F16, device=DEV)
    x[:, 0] = 4.0  # r = sqrt(D) / 4, y_0 = sqrt(D) w_0 = 64 w_0
    x[:, 1:] = synth.normal16((T, D - 1), 3, DEV, std=1e-3, dtype=F16)
    w = torch.full((D,), 2000.0, device=DEV)  # y_0 about 128000: overflow
    w[1:] = 1e-3  # y_j about 16e-3 * x_j, x_j about 1e-3: fp16 subnormals
    fo = run_fwd("plain", x, w, 1e-6, False, ex=True)
    torch.cuda.synchronize()
    assert torch.isinf(fo["y"][:, 0].float()).all()
    sub = (fo["y"].float().abs() < 2.0**-14) & (fo["y"].float() != 0)
    assert int(sub.sum()) > 0
    check_fwd("plain", x, w, 1e-6, False, fo, name="f16 range")
    assert np.isfinite(fo["rstd"].cpu().numpy()).all()


@pytest.mark.parametrize("workload", ["residual-f16-32768x4096", "gated-sigmoid-bf16-262144x128",
                                      "gated-f16-262144x128"])
def test_full_size_sampled(workload):
    """The benchmark's and the gated workload's full sizes in the new formats and
    gate: sampled rows against the oracle, sampled weight-gradient columns with
    all rows, and the weight gradient bitwise equal on a repeated call."""
    import oracle
    from tests._helpers import assert_bf16_parity, assert_dgamma_parity, assert_rel, to_f64
    from tests.gpu_common import chunk_rows_hint
    if workload.startswith("residual"):
        variant, T, D, dt, gate, zc = "residual", 32768, 4096, F16, "silu", False
    else:
        variant, T, D, zc = "gated", 262144, 128, True
        dt = F16 if "f16" in workload else BF16
        gate = "sigmoid" if "sigmoid" in workload else "silu"
    fmt = "f16" if dt == F16 else "bf16"
    a = _inputs(variant, T, D, 61, dt, zc, zstd=2.0)
    fo = run_fwd(variant, a["x"], a["w"], 1e-6, zc, z=a["z"], ex=True, gate=gate)
    bo = run_bwd(variant, a["g"], a["x"], a["w"], fo["rstd"], zc, z=a["z"], g_res=a["g_res"], ex=True, gate=gate)
    bo2 = run_bwd(variant, a["g"], a["x"], a["w"], fo["rstd"], zc, z=a["z"], g_res=a["g_res"], ex=True, gate=gate)
    torch.cuda.synchronize()
    assert torch.equal(bo["dgamma"].view(torch.int32), bo2["dgamma"].view(torch.int32)), "dgamma not bitwise"
    gen = torch.Generator().manual_seed(T + D)
    rows = torch.cat([torch.tensor([0, T - 1]), torch.randint(0, T, (510,), generator=gen)]).to(DEV)
    pick = lambda t: None if t is None else to_f64(t.index_select(0, rows))
    x, g, w, r = pick(a["x"]), pick(a["g"]), to_f64(a["w"]), pick(fo["rstd"])
    if variant == "gated":
        z = pick(a["z"])
        y_ref, r_ref = oracle.gated_fwd(x, z, w, 1e-6, zc, gate=gate, fmt=fmt)
        dx_ref, dz_ref, _, diag = oracle.gated_bwd(g, x, z, w, r, zc, diagnostics=True, gate=gate, fmt=fmt)
        assert_bf16_parity("dz", pick(bo["dz"]), dz_ref, diag["dz_pre"], diag["dz_scale"], fmt=fmt)
    else:
        y_ref, r_ref = oracle.rmsnorm_fwd(x, w, 1e-6, zc, fmt=fmt)
        dx_ref, _, diag = oracle.rmsnorm_bwd(g, x, w, r, zc, g_res=pick(a["g_res"]), diagnostics=True, fmt=fmt)
        assert torch.equal(fo["x_copy"].view(torch.int16), a["x"].view(torch.int16))
    assert_rel("rstd", r, r_ref, 1e-5)
    assert_bf16_parity("y", pick(fo["y"]), y_ref, fmt=fmt)
    assert_bf16_parity("dx", pick(bo["dx"]), dx_ref, diag["dx_pre"], diag["dx_scale"], fmt=fmt)
    cols = torch.cat([torch.tensor([0, D - 1]), torch.randint(0, D, (30,), generator=gen)]).to(DEV)
    col = lambda t: to_f64(t.index_select(1, cols))
    dw_ref, dw_abs = oracle.weight_grad(col(a["g"]), col(a["x"]), to_f64(fo["rstd"]),
                                        z=None if a["z"] is None else col(a["z"]), with_abs=True, gate=gate)
    C, n = chunk_rows_hint(T, D)
    assert_dgamma_parity("dgamma", to_f64(bo["dgamma"].index_select(0, cols)), dw_ref, dw_abs, C, n)
