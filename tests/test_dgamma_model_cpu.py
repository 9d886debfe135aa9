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
