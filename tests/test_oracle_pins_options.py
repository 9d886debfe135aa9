"""Pins of the oracle's activation-format and gate options (no GPU needed).

The gated norm's activation is configurable: silu by default, sigmoid allowed
([ZC-norm], "Not covered here": the gate activation comes from the model
config). The op contract carries tolerances for fp16 activations beside bf16
([ZC-norm], the list of in-tree corrections: contract-derived tolerances,
fp16 cases). These tests tie the oracle's fp16 rounding and its sigmoid gate to
facts outside the oracle: numpy's and torch's conversions, brute force over the
table of every fp16 value, central differences, and closed forms at special
gates.

Sources: [ZC-norm] RL-Kernel pull request 467 "[WS1][CUDA][Qwen3-Next] C1:
zero-centred RMSNorm references and CUDA kernel".
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests._helpers import f16_round_bruteforce, fd_grad

RNG = np.random.default_rng(4321)


def _f16_grid(a):
    """Random values already on the fp16 grid (as float64)."""
    return torch.tensor(np.asarray(a), dtype=torch.float32).to(torch.float16).to(torch.float64).numpy()


def _fd_setup(T, D):
    x = RNG.standard_normal((T, D))
    w = RNG.standard_normal(D)
    g = RNG.standard_normal((T, D))
    return x, w, g


# ==========================================================================
# fp16 rounding
# ==========================================================================

def test_round_f16_matches_torch_on_fp32_inputs():
    """For exact fp32 inputs, one rounding from double equals torch's fp32 -> fp16
    conversion (nearest even), ties, subnormals and overflow included."""
    bits = RNG.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # Values in and around the fp16 range, with explicit ties (low 13 bits 0x1000).
    near = (RNG.standard_normal(8000) * np.exp2(RNG.integers(-28, 17, 8000))).astype(np.float32)
    tie_bits = (near.view(np.uint32) & ~np.uint32(0x1FFF)) | np.uint32(0x1000)
    ties = tie_bits.view(np.float32)
    extra = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, -65520.0, 2.0**-24, 2.0**-25,
                      3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, 1e-45], dtype=np.float32)
    vals = np.concatenate([f, near, ties, extra])
    ref = torch.from_numpy(vals).to(torch.float16).to(torch.float64).numpy()
    got = oracle.round_f16(vals.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_round_f16_is_one_rounding_from_double():
    """Values finer than fp32: the table brute force and numpy's direct double ->
    half conversion. Rounding through fp32 first would get the first case wrong
    (1 + 2^-11 + 2^-40 becomes the tie 1 + 2^-11, which goes to even, 1.0)."""
    cases = [1 + 2**-11 + 2**-40, -(1 + 2**-11 + 2**-40), 1 + 2**-11, 1 + 3 * 2**-11,
             2.0**-25, 2.0**-25 + 2.0**-70, 3 * 2.0**-26, 2.0**-26, 65504 + 16 - 2.0**-30, 65520.0,
             1e-300, -1e-300, 1e300]
    cases += list(RNG.standard_normal(400) * np.exp2(RNG.integers(-30, 17, 400)))
    got = oracle.round_f16(np.array(cases))
    with np.errstate(over="ignore"):
        np.testing.assert_array_equal(got, np.array(cases).astype(np.float16).astype(np.float64))
    for v, g in zip(cases, got):
        assert g == f16_round_bruteforce(Fraction(v)), v
    assert got[0] == 1 + 2**-10 and got[2] == 1.0 and got[3] == 1 + 2**-9
    assert got[4] == 0.0 and got[5] == 2.0**-24 and got[6] == 2.0**-24


# ==========================================================================
# fp16 activations: only the final roundings change
# ==========================================================================

@pytest.mark.parametrize("zc", [False, True])
def test_f16_forward_output_bits_bruteforce(zc):
    """y = RN_f16( x * rstd * w_eff ) exactly (rationals and the fp16 table); the
    inverse RMS does not depend on the activation format."""
    T, D = 4, 16
    x = _f16_grid(RNG.standard_normal((T, D)) * 4)
    w = np.float32(RNG.standard_normal(D) * 0.3).astype(np.float64)
    y, rstd = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=zc, fmt="f16")
    _, rstd_b = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=zc, fmt="bf16")
    np.testing.assert_array_equal(rstd, rstd_b)
    weff = (np.float32(w) + np.float32(1.0)).astype(np.float64) if zc else w
    for t in range(T):
        for j in range(D):
            assert y[t, j] == f16_round_bruteforce(Fraction(x[t, j]) * Fraction(rstd[t]) * Fraction(weff[j]))


def test_f16_backward_rounds_the_same_values():
    """The backward's pre-rounding values and the fp32 weight gradient are the
    same in both formats; dx is their fp16 rounding (checked by brute force)."""
    T, D = 3, 16
    x = _f16_grid(RNG.standard_normal((T, D)))
    g = _f16_grid(RNG.standard_normal((T, D)))
    gr = _f16_grid(RNG.standard_normal((T, D)))
    w = np.float32(RNG.standard_normal(D)).astype(np.float64)
    _, r = oracle.rmsnorm_fwd(x, w, 1e-6, fmt="f16")
    dxh, dwh, dh = oracle.rmsnorm_bwd(g, x, w, r, g_res=gr, diagnostics=True, fmt="f16")
    dxb, dwb, db = oracle.rmsnorm_bwd(g, x, w, r, g_res=gr, diagnostics=True, fmt="bf16")
    np.testing.assert_array_equal(dh["dx_pre"], db["dx_pre"])
    np.testing.assert_array_equal(dwh, dwb)
    for v, got in zip(dh["dx_pre"].ravel(), dxh.ravel()):
        assert got == f16_round_bruteforce(Fraction(v))


def test_f16_gated_and_fused_add_bruteforce():
    """Gated: y = RN_f16(u * q(z)) for both gates; fused add: res_out =
    RN_f16(RN_fp32(x + res)) and y = RN_f16(h32 * rstd * w_eff)."""
    T, D = 2, 16
    x = _f16_grid(RNG.standard_normal((T, D)))
    z = _f16_grid(RNG.standard_normal((T, D)) * 3)
    w = np.float32(RNG.standard_normal(D)).astype(np.float64)
    for gate in ("silu", "sigmoid"):
        y, r = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=False, gate=gate, fmt="f16")
        for t in range(T):
            for j in range(D):
                sg = 1.0 / (1.0 + math.exp(-z[t, j]))
                q = sg if gate == "sigmoid" else z[t, j] * sg
                exact = Fraction(x[t, j]) * Fraction(r[t]) * Fraction(w[j]) * Fraction(q)
                ref = f16_round_bruteforce(exact)
                assert abs(y[t, j] - ref) <= abs(ref) * 2.0**-40, (gate, t, j)  # q rounded to double only
    res = _f16_grid(RNG.standard_normal((T, D)) * 8)
    y, rstd, ro = oracle.fused_add_fwd(x, res, w, 1e-6, fmt="f16")
    for t in range(T):
        for j in range(D):
            h32 = float(np.float32(Fraction(x[t, j]) + Fraction(res[t, j])))
            assert ro[t, j] == f16_round_bruteforce(Fraction(h32))
            assert y[t, j] == f16_round_bruteforce(Fraction(h32) * Fraction(rstd[t]) * Fraction(w[j]))


# ==========================================================================
# Sigmoid gate
# ==========================================================================

@pytest.mark.parametrize("zc", [False, True])
def test_sigmoid_gate_bwd_matches_finite_differences(zc):
    """dx, dz and dweight of y = ((x r) w_eff) sigmoid(z) against central
    differences of the forward; the weight gradient alone agrees on a column
    subset."""
    x, w, g = _fd_setup(T=3, D=8)
    z = RNG.standard_normal(x.shape) * 2

    def loss():
        y, _ = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=zc, rounded=False, gate="sigmoid")
        return float(np.sum(g * y))

    _, r = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=zc, rounded=False, gate="sigmoid")
    dx, dz, dw = oracle.gated_bwd(g, x, z, w, r, zero_centered_gamma=zc, rounded=False, gate="sigmoid")
    assert np.abs(dx - fd_grad(loss, x)).max() < 2e-8
    assert np.abs(dz - fd_grad(loss, z)).max() < 2e-8
    assert np.abs(dw - fd_grad(loss, w)).max() < 2e-8
    cols = [0, 5]
    dwc = oracle.weight_grad(g[:, cols], x[:, cols], r, z=z[:, cols], rounded=False, gate="sigmoid")
    np.testing.assert_array_equal(dwc, dw[cols])


def test_sigmoid_gate_special_values():
    """sigmoid(0) = 1/2 and sigmoid'(0) = 1/4; sigmoid(ln 3) = 3/4 and its slope
    3/16; for large z the gate is 1 (the plain norm) with slope e^-z; and the
    silu gate is z times the sigmoid gate."""
    T, D = 3, 16
    x = RNG.standard_normal((T, D))
    w = RNG.standard_normal(D)
    g = RNG.standard_normal((T, D))
    y_plain, r = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=True, rounded=False)
    _, dw_plain = oracle.rmsnorm_bwd(g, x, w, r, zero_centered_gamma=True, rounded=False)
    kw = dict(zero_centered_gamma=True, rounded=False, gate="sigmoid")
    for zval, q, dq in ((0.0, 0.5, 0.25), (math.log(3.0), 0.75, 3.0 / 16.0)):
        z = np.full((T, D), zval)
        y, rz = oracle.gated_fwd(x, z, w, 1e-6, **kw)
        np.testing.assert_array_equal(rz, r)
        np.testing.assert_allclose(y, q * y_plain, rtol=1e-15, atol=1e-300)
        _, dz, dw = oracle.gated_bwd(g, x, z, w, r, **kw)
        np.testing.assert_allclose(dz, dq * g * y_plain, rtol=1e-14, atol=1e-300)
        np.testing.assert_allclose(dw, q * dw_plain, rtol=1e-13, atol=1e-14)
    zb = np.full((T, D), 60.0)
    y, _ = oracle.gated_fwd(x, zb, w, 1e-6, **kw)
    np.testing.assert_array_equal(y, y_plain)
    _, dz, _ = oracle.gated_bwd(g, x, zb, w, r, **kw)
    np.testing.assert_allclose(dz, g * y_plain * math.exp(-60.0), rtol=1e-13)
    z = RNG.standard_normal((T, D)) * 3
    ys, _ = oracle.gated_fwd(x, z, w, 1e-6, **kw)
    yq, _ = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=True, rounded=False, gate="silu")
    np.testing.assert_allclose(yq, z * ys, rtol=1e-14, atol=1e-300)


def test_sigmoid_gate_slope_has_no_cancellation_in_the_tails():
    """q'(z) = sigmoid(z) sigmoid(-z) keeps full relative precision far out in
    both tails (where 1 - sigmoid(z) would round to 0): compare with the closed
    form e^-|z| / (1 + e^-|z|)^2."""
    x, w, g = _fd_setup(T=1, D=8)
    z = np.array([[-45.0, -30.0, -20.0, 20.0, 30.0, 45.0, 0.5, -0.5]])
    _, r = oracle.gated_fwd(x, z, w, 1e-6, rounded=False, gate="sigmoid")
    _, dz, _ = oracle.gated_bwd(g, x, z, w, r, rounded=False, gate="sigmoid")
    u = x * r[:, None] * (w + 1.0)
    e = np.exp(-np.abs(z))
    np.testing.assert_allclose(dz, g * u * e / (1.0 + e) ** 2, rtol=1e-13)
