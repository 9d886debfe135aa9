"""The weight gradient of the backward, bit for bit against a float32
model of its stated arithmetic.

Per RL-Kernel pull request 414 "[DSv4][P1-5] rmsnorm_residual" (Implementation:
ascending fp32 reductions, every multiply and add rounded on its own, no
atomics), dgamma_j is built from the products ((g_tj * x_tj) * r_t), each
rounded to fp32, added in ascending row order within each chunk (pass 1; wide
path: chunks of wide_chunk_rows(T, D) rows, 32 or, at some T for
2048 < D <= 7168, fewer; the narrow path's order is described below), and the chunk
partials added by the fixed pass-2 tree: 32 contiguous ranges of
ceil(n / 32) chunks, each summed in ascending order, then the 32 range totals
in order. Every operand here is exact in fp32 (bf16 or fp16 activations, the
rstd given as input), so numpy's float32 operations reproduce each rounding,
and any fused multiply-add anywhere in the kernel, or any change of order,
changes bits. The gated mode is left out: its products involve the gate,
which the kernel evaluates with the hardware exponential.

Widths cover every backward launch shape: on the narrow path (D <= 256),
lane groups of 1, 2, 8, 16 and 32 lanes a row, whose chunk order is its own
(lane groups over interleaved rows, then the group totals in order; see
dgamma_model); on the wide path one vector a thread (264, 1000, and 2048
outside the plain mode), two vectors on 128 threads (2048 plain), on 256
(4096) and on up to 512 (8192; 7168 outside the plain mode), four vectors on
224 (7168 plain) and on 512 threads (16384).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import synth
from tests._helpers import dgamma_model
from tests.gpu_common import DEV

pytestmark = pytest.mark.gpu


def _f32(t):
    return t.detach().float().cpu().numpy().astype(np.float32)


WIDE = [(D, T) for D in (264, 1000, 2048, 4096, 7168, 8192, 16384) for T in (100, 1100)]
# T where 32-row chunks fill their rounds poorly and the chunk is shortened
# (4096 x 10000: 17-row chunks; 7168 x 9729: 17; 4096 x 32768: 27)
BALANCED = [(4096, 10000), (7168, 9729), (4096, 32768)]
NARROW = [(D, T) for D in (8, 16, 40, 64, 128, 200, 256) for T in (100, 1100)]  # lane groups of 1 to 32
CASES = NARROW + WIDE + BALANCED


@pytest.mark.parametrize("variant", ["plain", "residual", "fused"])
@pytest.mark.parametrize("D,T", CASES)
def test_dgamma_bits(D, T, variant):
    if D >= 7168 and T == 1100:
        T = 300  # keeps the model quick for the widest rows (10 chunks)
    seed = D + T + len(variant)
    dtype = torch.float16 if (D // 8) % 2 else torch.bfloat16
    x = synth.normal16((T, D), seed, DEV, dtype=dtype)
    g = synth.normal16((T, D), seed + 1, DEV, dtype=dtype)
    w = synth.gamma_f32(D, seed + 2, DEV)
    r = (torch.rand(T, device=DEV, generator=torch.Generator(DEV).manual_seed(seed)) + 0.5).float()
    dx = torch.empty_like(x)
    dg = torch.empty(D, device=DEV)
    ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=DEV)
    h = _f32(x)
    if variant == "plain":
        rn.rmsnorm_bwd_ex(g, x, w, r, dx, dg, ws, False)
    elif variant == "residual":
        gr = synth.normal16((T, D), seed + 3, DEV, dtype=dtype)
        rn.rmsnorm_residual_bwd_ex(g, x, w, r, gr, dx, dg, ws, True)
    else:
        res = synth.normal16((T, D), seed + 4, DEV, std=4.0, dtype=dtype)
        gr = synth.normal16((T, D), seed + 5, DEV, dtype=dtype)
        rn.rmsnorm_fused_add_bwd_ex(g, x, res, w, r, gr, dx, dg, ws, False)
        h = h + _f32(res)                     # the fused mode normalises h = x + res (fp32)
    torch.cuda.synchronize()
    want = dgamma_model(_f32(g), h, _f32(r))
    got = dg.cpu().numpy()
    bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, (f"{variant} D={D} T={T} {dtype}: {bad.size} columns differ, first {bad[:5].tolist()}: "
                           f"got {got[bad[:3]].tolist()} want {want[bad[:3]].tolist()}")
