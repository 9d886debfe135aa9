"""GPU parity of every mode on the wide backward's balanced weight-gradient chunks.

For 2048 < D <= 7168, a T whose 32-row chunks fill fewer than 90 % of their
rounds of 152 x 2 CTAs gets shorter chunks (17 rows at T = 9729 and 10000, 20
at T = 12000), taken by the stepping instantiation of the two-vector backward
kernels (256 threads up to D = 4096; up to 512 threads beyond, which these
modes use there; the plain mode's four-vector 224-thread kernel is covered by
the bit-for-bit tests). The bit-for-bit tests
cover the plain, residual and fused-add modes there; this file adds the gated
mode with both gates and the fp16 format, against the float64 oracle with the
usual tolerances (outputs within one ulp or the cancellation bound, rstd 1e-5
relative, dgamma 1e-4 relative or the fixed tree's bound), and checks that the
chunk really is the shortened one.
"""
from __future__ import annotations

import pytest
import torch

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import synth
from tests._helpers import wide_chunk_rows
from tests.gpu_common import DEV, check_bwd, check_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

# (D, T): the 256-thread two-vector kernel (2056, 4096) and the two-vector
# kernel on up to 512 threads (7168), each at a T that shortens the chunk
SHAPES = [(2056, 12000), (4096, 10000), (7168, 9729)]
CASES = [("gated", torch.bfloat16, "silu"), ("gated", torch.bfloat16, "sigmoid"),
         ("gated", torch.float16, "sigmoid"), ("residual", torch.float16, "silu"),
         ("fused", torch.float16, "silu")]


@pytest.mark.parametrize("D,T", SHAPES)
@pytest.mark.parametrize("variant,dtype,gate", CASES, ids=lambda v: str(v).replace("torch.", ""))
def test_balanced_chunk_parity(variant, dtype, gate, D, T):
    C = wide_chunk_rows(T, D)
    assert C < 32 and rn.workspace_bytes(T, D) == -(-T // C) * 4 * D  # the shortened chunk is in use
    seed = D + T + len(variant) + (dtype == torch.float16) + 2 * (gate == "sigmoid")
    zc = variant == "gated"
    x = synth.normal16((T, D), seed, DEV, dtype=dtype)
    g = synth.normal16((T, D), seed + 1, DEV, dtype=dtype)
    w = synth.gamma_f32(D, seed + 2, DEV, mean=0.0 if zc else 1.0, std=0.1 if zc else 0.2)
    z = synth.normal16((T, D), seed + 3, DEV, dtype=dtype) if variant == "gated" else None
    gr = synth.normal16((T, D), seed + 4, DEV, dtype=dtype) if variant in ("residual", "fused") else None
    res = synth.normal16((T, D), seed + 5, DEV, std=4.0, dtype=dtype) if variant == "fused" else None
    fo = run_fwd(variant, x, w, 1e-6, zc, z=z, res=res, ex=True, gate=gate)
    bo = run_bwd(variant, g, x, w, fo["rstd"], zc, z=z, g_res=gr, res=res, ex=True, gate=gate)
    torch.cuda.synchronize()
    name = f"{variant} {dtype} {gate} T={T} D={D} chunk={C}"
    check_fwd(variant, x, w, 1e-6, zc, fo, z=z, res=res, gate=gate, name=name)
    check_bwd(variant, g, x, w, fo["rstd"], zc, bo, z=z, g_res=gr, res=res, gate=gate, name=name)
    assert rn.rmsnorm_device_error() == 0
