"""The float32 model of the weight gradient (tests/_helpers.py), which the
GPU test holds the kernels to bit for bit, checked on the CPU: it agrees with
the float64 oracle within the weight gradient's tolerance, and it can tell
separately rounded arithmetic from a fused multiply-add on ordinary inputs, so
a kernel that fused would fail the GPU test."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests._helpers import dgamma_model


def _inputs(T, D, seed):
    rng = np.random.default_rng(seed)
    g = oracle.round_bf16(rng.standard_normal((T, D))).astype(np.float32)
    x = oracle.round_bf16(rng.standard_normal((T, D))).astype(np.float32)
    r = (rng.random(T) + 0.5).astype(np.float32)
    return g, x, r


@pytest.mark.parametrize("D", [64, 264])
def test_model_matches_the_oracle_within_tolerance(D):
    T = 1100
    g, x, r = _inputs(T, D, 5)
    got = dgamma_model(g, x, r).astype(np.float64)
    w = np.ones(D)
    _, want = oracle.rmsnorm_bwd(g.astype(np.float64), x.astype(np.float64), w, r.astype(np.float64), False)
    absum = (np.abs(g.astype(np.float64) * x) * r[:, None]).sum(axis=0)
    assert np.all(np.abs(got - want) <= 1e-4 * np.abs(want) + 1e-6 * absum)


@pytest.mark.parametrize("D", [128, 1000])
def test_model_separates_fused_from_separate_rounding(D):
    T = 300
    g, x, r = _inputs(T, D, 9)
    a = dgamma_model(g, x, r)
    b = dgamma_model(g, x, r, fused=True)
    differ = np.count_nonzero(a.view(np.uint32) != b.view(np.uint32))
    assert differ > D // 10, differ   # most columns tell the two apart


@pytest.mark.parametrize("D", [128, 264, 4096])
def test_dx_model_matches_the_oracle(D):
    """The dx model (fixed row tree, fp32 steps, one rounding) is within the
    contract's bound of the float64 oracle: one ulp, or the cancellation bound."""
    from tests._helpers import assert_bf16_parity, dx_model
    T = 40
    g, x, r = _inputs(T, D, 13)
    w = (1.0 + 0.1 * np.random.default_rng(14).standard_normal(D)).astype(np.float32)
    got = dx_model(g, x, w, r, "plain").astype(np.float64)
    dx, _, diag = oracle.rmsnorm_bwd(g.astype(np.float64), x.astype(np.float64), w.astype(np.float64),
                                     r.astype(np.float64), False, diagnostics=True)
    assert_bf16_parity(f"dx model D={D}", got, dx, diag["dx_pre"], diag["dx_scale"])


def test_row_sum_model_tree_is_not_a_plain_sum():
    """The row tree of the model differs from a left-to-right sum on ordinary
    inputs, so the GPU test pins the kernels' tree, not just the total."""
    from tests._helpers import row_sums_model
    rng = np.random.default_rng(3)
    terms = rng.standard_normal((64, 4096)).astype(np.float32)
    tree = row_sums_model(terms, 4096, "residual")
    seq = np.zeros(64, np.float32)
    for k in range(4096):
        seq = seq + terms[:, k]
    assert np.count_nonzero(tree.view(np.uint32) != seq.view(np.uint32)) > 16
