"""Pins of the float64 CPU oracle to facts outside itself (no GPU needed).

Each test ties one part of the oracle to something it cannot trivially agree
with: a finite difference of its own forward, a closed form for a special
input, an exact brute-force evaluation, a library routine, or a figure the
pages print. Together they are chosen so that a dropped term, a wrong sign,
a wrong divisor, a misplaced rounding point or a transposed operand in the
oracle fails at least one of them.

Sources: [Megatron] Megatron-LM pull request 6859 "Fix the batch-invariant
RMSNorm forward and its input gradient"; [ZC-norm] RL-Kernel pull request 467
"[WS1][CUDA][Qwen3-Next] C1: zero-centred RMSNorm references and CUDA kernel";
[Residual] RL-Kernel pull request 414 "[DSv4][P1-5] rmsnorm_residual".
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests._helpers import bf16_round_bruteforce, fd_grad, fp32_round_exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_grid(a):
    """Random values already on the bf16 grid (as float64)."""
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


# ==========================================================================
# bf16 rounding (the oracle's only non-library rounding step)
# ==========================================================================

def test_round_bf16_matches_torch_on_fp32_inputs():
    """For values that are exact fp32 numbers, one rounding from double equals
    torch's fp32 -> bf16 conversion (round to nearest even), ties included."""
    bits = RNG.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # Explicit ties (low 16 bits exactly 0x8000), odd and even, and near overflow.
    tie_bits = (RNG.integers(0, 2**16, size=2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties = tie_bits.view(np.float32)
    ties = ties[np.isfinite(ties)]
    extra = np.array([0.0, -0.0, 1e-45, -1e-45, 1.17549435e-38, 3.3895314e38, 3.4028235e38,
                      -3.4028235e38, 3.3961e38], dtype=np.float32)
    vals = np.concatenate([f, ties, extra])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(vals.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_round_bf16_is_one_rounding_from_double():
    """Values between fp32 and bf16 precision: brute force over the bf16 table.
    Rounding via fp32 first would get the first two wrong (double rounding)."""
    cases = [1 + 2**-8 + 2**-40, -(1 + 2**-8 + 2**-40), 1 + 2**-8, 1 + 3 * 2**-8,
             2**-134, 3 * 2**-134, 2**-134 + 2**-200, 2.0**-140, 1.5 * 2**-126 + 2**-150,
             (2 - 2**-8) * 2.0**127, (2 - 2**-8) * 2.0**127 - 2.0**100, 1e-300, -1e-300]
    cases += list(RNG.standard_normal(300) * np.exp2(RNG.integers(-130, 120, 300)))
    got = oracle.round_bf16(np.array(cases))
    for v, g in zip(cases, got):
        assert g == bf16_round_bruteforce(Fraction(v)) or (math.isinf(g) and math.isinf(
            bf16_round_bruteforce(Fraction(v)))), v
    assert got[0] == 1 + 2**-7 and got[2] == 1.0 and got[3] == 1 + 2**-6


# ==========================================================================
# Forward: closed forms and exact brute force
# ==========================================================================

@pytest.mark.parametrize("c", [0.75, -3.0, 1.0, 2.0**-20])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.25])
def test_fwd_constant_row_closed_form(c, eps):
    """x_j = c for all j: mean(x^2) = c^2, so r = (c^2 + eps)^(-1/2), exactly.
    Pins the divisor (D, not D-1), eps inside the root, and the fp32 rounding of r."""
    D = 24
    x = np.full((1, D), c)
    w = _bf16_grid(RNG.standard_normal(D))
    y, rstd = oracle.rmsnorm_fwd(x, w, eps, rounded=True)
    eps32 = Fraction(float(np.float32(eps)))
    getcontext().prec = 60
    ms = Fraction(c) ** 2 + eps32
    r_exact = Decimal(1) / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
    f = np.float32(float(r_exact))
    # nearest fp32 to the 60-digit value (check both neighbours)
    cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(0))]
    best = min(cands, key=lambda v: abs(Decimal(float(v)) - r_exact))
    assert rstd[0] == float(best)
    if eps == 0.0 and c in (1.0, 2.0**-20):
        # r = 1/|c| is a power of two, so y = sign(c) * w exactly
        np.testing.assert_array_equal(y[0], np.sign(c) * w)


def test_rstd_correctly_rounded_bruteforce():
    """rstd is the fp32 value nearest to the exact (mean(x^2) + eps)^(-1/2)."""
    getcontext().prec = 60
    for D in (8, 13, 64):
        x = _bf16_grid(RNG.standard_normal((6, D)) * 3)
        _, rstd = oracle.rmsnorm_fwd(x, np.ones(D), 1e-6, rounded=True)
        eps = Fraction(float(np.float32(1e-6)))
        for t in range(x.shape[0]):
            ms = sum(Fraction(v) ** 2 for v in x[t]) / D + eps
            r = Decimal(1) / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
            f = np.float32(float(r))
            cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(0))]
            best = min(cands, key=lambda c: abs(Decimal(float(c)) - r))
            assert rstd[t] == float(best)


@pytest.mark.parametrize("zc", [False, True])
def test_fwd_output_bits_bruteforce(zc):
    """y = RN_bf16( x * rstd * w_eff ) evaluated exactly with rationals; w_eff is the
    fp32 sum w + 1 when zero-centred ([Megatron], What does this PR do, item 1)."""
    T, D = 4, 16
    x = _bf16_grid(RNG.standard_normal((T, D)))
    w = np.float32(RNG.standard_normal(D) * 0.3).astype(np.float64)
    y, rstd = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=zc, rounded=True)
    weff = (np.float32(w) + np.float32(1.0)).astype(np.float64) if zc else w
    for t in range(T):
        for j in range(D):
            exact = Fraction(x[t, j]) * Fraction(rstd[t]) * Fraction(weff[j])
            assert y[t, j] == bf16_round_bruteforce(exact)


def test_fwd_scale_invariance_eps0():
    """At eps=0 the output does not depend on the row's scale: bitwise for powers of
    two (every step scales exactly), to double precision for a general factor."""
    x = _bf16_grid(RNG.standard_normal((5, 32)))
    w = np.float32(1 + 0.1 * RNG.standard_normal(32)).astype(np.float64)
    y0, r0 = oracle.rmsnorm_fwd(x, w, 0.0, rounded=True)
    for k in (-3, 5):
        y1, r1 = oracle.rmsnorm_fwd(x * 2.0**k, w, 0.0, rounded=True)
        np.testing.assert_array_equal(y1, y0)
        np.testing.assert_array_equal(r1, r0 * 2.0**-k)
    ye, _ = oracle.rmsnorm_fwd(x, w, 0.0, rounded=False)
    yc, _ = oracle.rmsnorm_fwd(x * 1.37, w, 0.0, rounded=False)
    np.testing.assert_allclose(yc, ye, rtol=1e-14, atol=0)
    # and the gradient scales as 1/c
    g = RNG.standard_normal((5, 32))
    _, r_e = oracle.rmsnorm_fwd(x, w, 0.0, rounded=False)
    _, r_c = oracle.rmsnorm_fwd(x * 1.37, w, 0.0, rounded=False)
    dx0, dw0 = oracle.rmsnorm_bwd(g, x, w, r_e, rounded=False)
    dx1, dw1 = oracle.rmsnorm_bwd(g, x * 1.37, w, r_c, rounded=False)
    np.testing.assert_allclose(dx1, dx0 / 1.37, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dw1, dw0, rtol=1e-12, atol=1e-15)


def test_zero_centred_forward_matches_plain_with_offset_weight():
    """zero_centered_gamma=True equals the plain forward run with the fp32 weight w+1,
    and differs from the plain forward with w by O(1) — the defect the Megatron fix
    removed printed a max difference of ~2.3 ([Megatron], Commit 1)."""
    gold = _golden("megatron_zc_forward.json")
    x = _bf16_grid(RNG.standard_normal((64, 256)))
    w = np.float32(0.1 * RNG.standard_normal(256)).astype(np.float64)
    y_zc, r_zc = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=True)
    w1 = (np.float32(w) + np.float32(1)).astype(np.float64)
    y_p1, r_p1 = oracle.rmsnorm_fwd(x, w1, 1e-6, zero_centered_gamma=False)
    np.testing.assert_array_equal(y_zc, y_p1)
    np.testing.assert_array_equal(r_zc, r_p1)
    y_p, _ = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=False)
    diff = np.abs(y_zc - y_p).max()
    assert diff > 0.25 * gold["before_max_abs_diff"]["bf16"]
    assert np.abs(y_zc - y_p1).max() == gold["after_max_abs_diff"]


def test_zero_rows_padding():
    """A zero row: r = eps^(-1/2) (1000 at eps=1e-6, to fp32), y = 0, dx = RN(g w r)."""
    D = 16
    x = np.zeros((2, D))
    w = np.float32(1 + 0.1 * RNG.standard_normal(D)).astype(np.float64)
    g = _bf16_grid(RNG.standard_normal((2, D)))
    y, r = oracle.rmsnorm_fwd(x, w, 1e-6)
    assert np.all(y == 0) and r[0] == float(np.float32(1.0 / math.sqrt(float(np.float32(1e-6)))))
    dx, dw = oracle.rmsnorm_bwd(g, x, w, r)
    np.testing.assert_array_equal(dx, oracle.round_bf16(g * w * r[:, None]))
    assert np.all(dw == 0)


# ==========================================================================
# Backward: finite differences of the oracle's own unrounded forward
# ==========================================================================

def _fd_setup(T=3, D=8, unit_w=False, zero_w=False):
    x = RNG.standard_normal((T, D))
    if zero_w:
        w = np.zeros(D)
    elif unit_w:
        w = np.ones(D)
    else:
        w = RNG.standard_normal(D)
    g = RNG.standard_normal((T, D))
    return x, w, g


@pytest.mark.parametrize("zc", [False, True])
@pytest.mark.parametrize("eps", [1e-6, 0.3])
def test_plain_bwd_matches_finite_differences(zc, eps):
    """dx and dgamma of L = sum(g * y) against central differences of the forward
    ([Megatron], How to reproduce: analytic backward vs a finite difference of the
    function's own forward, with non-unit weights)."""
    gold = _golden("megatron_fd_table.json")
    x, w, g = _fd_setup(T=3, D=8)

    def loss():
        y, _ = oracle.rmsnorm_fwd(x, w, eps, zero_centered_gamma=zc, rounded=False)
        return float(np.sum(g * y))

    _, r = oracle.rmsnorm_fwd(x, w, eps, zero_centered_gamma=zc, rounded=False)
    dx, dw = oracle.rmsnorm_bwd(g, x, w, r, zero_centered_gamma=zc, rounded=False)
    fdx = fd_grad(loss, x)
    fdw = fd_grad(loss, w)
    err = max(np.abs(dx - fdx).max(), np.abs(dw - fdw).max())
    # the pages' fp64 FD harness reached ~2e-9 after the fix
    assert err < 10 * max(gold["fp64"]["after_randn"]), err


def _defective_dx(g, x, w, r):
    """The double-weight defect, planted on the CPU side: the variance term is
    multiplied by w_k a second time ([Megatron], What does this PR do, item 2)."""
    D = x.shape[1]
    s = np.sum(g * x * w, axis=1, keepdims=True)
    return g * w * r[:, None] - w * (r[:, None] ** 3 * x / D) * s


def test_fd_discriminates_the_double_weight_defect():
    """The FD pin rejects the defect with non-unit weights (O(1) error) and cannot
    see it with unit weights, exactly as the pages' table shows; weight=0 gives dx=0."""
    gold = _golden("megatron_fd_table.json")
    for unit in (False, True):
        x, w, g = _fd_setup(T=4, D=16, unit_w=unit)

        def loss():
            y, _ = oracle.rmsnorm_fwd(x, w, 1e-6, rounded=False)
            return float(np.sum(g * y))

        _, r = oracle.rmsnorm_fwd(x, w, 1e-6, rounded=False)
        fdx = fd_grad(loss, x)
        bad = np.abs(_defective_dx(g, x, w, r) - fdx).max()
        good, _ = oracle.rmsnorm_bwd(g, x, w, r, rounded=False)
        good_err = np.abs(good - fdx).max()
        assert good_err < 10 * max(gold["fp64"]["after_randn"])
        if unit:
            assert bad < 10 * max(gold["fp64"]["ones"]), bad
        else:
            assert bad > 0.05 * min(gold["fp64"]["before_randn"]), bad
    x, w, g = _fd_setup(T=3, D=8, zero_w=True)
    _, r = oracle.rmsnorm_fwd(x, w, 1e-6, rounded=False)
    dx, _ = oracle.rmsnorm_bwd(g, x, w, r, rounded=False)
    assert np.all(dx == gold["weight_zeros_dx"])
    dxr, _ = oracle.rmsnorm_bwd(_bf16_grid(g), _bf16_grid(x), w, r, rounded=True)
    assert np.all(dxr == 0.0)


def test_residual_bwd_matches_finite_differences():
    """rmsnorm_residual: L = sum(g*y) + sum(g_res * x_copy), so dx gains g_res
    ([Residual], reviewer's "for dx"); the copy is the input bit for bit."""
    x, w, g = _fd_setup(T=3, D=8)
    gres = RNG.standard_normal(x.shape)

    def loss():
        y, _, xc = oracle.residual_fwd(x, w, 1e-6, rounded=False)
        return float(np.sum(g * y) + np.sum(gres * xc))

    _, r, xc = oracle.residual_fwd(x, w, 1e-6, rounded=False)
    assert np.array_equal(xc, x)
    dx, dw = oracle.residual_bwd(g, x, w, r, gres, rounded=False)
    assert np.abs(dx - fd_grad(loss, x)).max() < 2e-8
    assert np.abs(dw - fd_grad(loss, w)).max() < 2e-8
    xb = _bf16_grid(x)
    yb, rb, xcb = oracle.residual_fwd(xb, w, 1e-6)
    assert np.array_equal(xcb, xb)


@pytest.mark.parametrize("zc,residual", [(False, False), (True, False), (False, True)])
def test_bwd_output_bits_bruteforce(zc, residual):
    """In rounded mode dx is the bf16 value nearest the exact input gradient at
    the saved fp32 rstd: g w_eff r - (r^3 x / D) sum_i g_i x_i w_eff_i [+ g_res]
    ([Megatron], What does this PR do, item 2; [Residual], the reviewer's "for
    dx"), evaluated with rationals and rounded once."""
    T, D = 3, 16
    x = _bf16_grid(RNG.standard_normal((T, D)))
    g = _bf16_grid(RNG.standard_normal((T, D)))
    gres = _bf16_grid(RNG.standard_normal((T, D))) if residual else None
    w = np.float32(RNG.standard_normal(D) * 0.3 + (0.0 if zc else 1.0)).astype(np.float64)
    _, r = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=zc)
    if residual:
        dx, _ = oracle.residual_bwd(g, x, w, r, gres, zero_centered_gamma=zc)
    else:
        dx, _ = oracle.rmsnorm_bwd(g, x, w, r, zero_centered_gamma=zc)
    weff = [Fraction(float(np.float32(v) + np.float32(1.0))) if zc else Fraction(v) for v in w]
    for t in range(T):
        rt = Fraction(r[t])
        s = sum(Fraction(g[t, i]) * Fraction(x[t, i]) * weff[i] for i in range(D))
        for k in range(D):
            v = Fraction(g[t, k]) * weff[k] * rt - rt ** 3 * Fraction(x[t, k]) / D * s
            if residual:
                v += Fraction(gres[t, k])
            assert dx[t, k] == bf16_round_bruteforce(v), (t, k)


@pytest.mark.parametrize("zc", [False, True])
def test_gated_bwd_matches_finite_differences(zc):
    """Gated norm: dx, dz and dweight against central differences of the forward."""
    x, w, g = _fd_setup(T=3, D=8)
    z = RNG.standard_normal(x.shape) * 2

    def loss():
        y, _ = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=zc, rounded=False)
        return float(np.sum(g * y))

    _, r = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=zc, rounded=False)
    dx, dz, dw = oracle.gated_bwd(g, x, z, w, r, zero_centered_gamma=zc, rounded=False)
    assert np.abs(dx - fd_grad(loss, x)).max() < 2e-8
    assert np.abs(dz - fd_grad(loss, z)).max() < 2e-8
    assert np.abs(dw - fd_grad(loss, w)).max() < 2e-8
    # the weight gradient alone, on a column subset, equals the full one's columns
    cols = [1, 6]
    dwc = oracle.weight_grad(g[:, cols], x[:, cols], r, z=z[:, cols], rounded=False)
    np.testing.assert_array_equal(dwc, dw[cols])


def test_gated_special_gates():
    """silu(0) = 0, so y = 0 and dz = g u / 2; for z = ln 3, sigmoid = 3/4 so
    y = (3/4) ln3 times the plain output; for very large z, silu(z) -> z."""
    T, D = 3, 16
    x = RNG.standard_normal((T, D))
    w = RNG.standard_normal(D)
    g = RNG.standard_normal((T, D))
    y_plain, r = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=True, rounded=False)
    z0 = np.zeros((T, D))
    y0, r0 = oracle.gated_fwd(x, z0, w, 1e-6, zero_centered_gamma=True, rounded=False)
    assert np.all(y0 == 0)
    np.testing.assert_array_equal(r0, r)
    _, dz0, dw0 = oracle.gated_bwd(g, x, z0, w, r, zero_centered_gamma=True, rounded=False)
    np.testing.assert_allclose(dz0, 0.5 * g * y_plain, rtol=1e-15, atol=1e-300)
    assert np.all(dw0 == 0)
    zl3 = np.full((T, D), math.log(3.0))
    yl3, _ = oracle.gated_fwd(x, zl3, w, 1e-6, zero_centered_gamma=True, rounded=False)
    np.testing.assert_allclose(yl3, y_plain * 0.75 * math.log(3.0), rtol=1e-14)
    zb = np.full((T, D), 60.0)
    yb, _ = oracle.gated_fwd(x, zb, w, 1e-6, zero_centered_gamma=True, rounded=False)
    np.testing.assert_allclose(yb, y_plain * 60.0, rtol=1e-14)


def test_weight_grad_column_subset_and_rows_order_free_of_layout():
    """The weight gradient is per column: slicing columns commutes with it, and
    the result is an fp32 value ([Residual], Implementation: the weight gradient
    is fp32), the one nearest the exact sum (checked against rationals)."""
    T, D = 5, 8
    x = _bf16_grid(RNG.standard_normal((T, D)))
    g = _bf16_grid(RNG.standard_normal((T, D)))
    r = np.float32(RNG.uniform(0.5, 2, T)).astype(np.float64)
    dw = oracle.weight_grad(g, x, r)
    for j in range(D):
        exact = sum(Fraction(g[t, j]) * Fraction(x[t, j]) * Fraction(r[t]) for t in range(T))
        assert abs(Fraction(dw[j]) - exact) <= abs(exact) * Fraction(1, 2**23) + Fraction(1, 2**140)
        assert dw[j] == fp32_round_exact(exact), j


# ==========================================================================
# Fused add + RMSNorm (the decoder-norm path of the zero-centred RMSNorm PR)
# ==========================================================================

def test_fused_add_bwd_matches_finite_differences():
    """L = sum(g*y) + sum(g_res*res_out): the gradient of x and of res are the same
    dh, and dgamma follows the plain form on h = x + res."""
    x, w, g = _fd_setup(T=3, D=8)
    res = RNG.standard_normal(x.shape)
    gres = RNG.standard_normal(x.shape)

    def loss():
        y, _, ro = oracle.fused_add_fwd(x, res, w, 1e-6, rounded=False)
        return float(np.sum(g * y) + np.sum(gres * ro))

    _, r, _ = oracle.fused_add_fwd(x, res, w, 1e-6, rounded=False)
    dh, dw = oracle.fused_add_bwd(g, x, res, w, r, g_res=gres, rounded=False)
    assert np.abs(dh - fd_grad(loss, x)).max() < 2e-8
    assert np.abs(dh - fd_grad(loss, res)).max() < 2e-8
    assert np.abs(dw - fd_grad(loss, w)).max() < 2e-8


@pytest.mark.parametrize("zc", [False, True])
def test_fused_add_rounding_bruteforce(zc):
    """res_out = RN_bf16(RN_fp32(x + res)) and y = RN_bf16(h32 * rstd * w_eff), with
    rationals; the zero residual reduces to the plain forward bit for bit."""
    T, D = 3, 16
    x = _bf16_grid(RNG.standard_normal((T, D)))
    res = _bf16_grid(RNG.standard_normal((T, D)) * 8)
    w = np.float32(RNG.standard_normal(D) * 0.3).astype(np.float64)
    y, rstd, ro = oracle.fused_add_fwd(x, res, w, 1e-6, zero_centered_gamma=zc)
    weff = (np.float32(w) + np.float32(1.0)).astype(np.float64) if zc else w
    for t in range(T):
        for j in range(D):
            h32 = float(np.float32(Fraction(x[t, j]) + Fraction(res[t, j])))  # x + res is exact in double
            assert ro[t, j] == bf16_round_bruteforce(Fraction(h32))
            assert y[t, j] == bf16_round_bruteforce(Fraction(h32) * Fraction(rstd[t]) * Fraction(weff[j]))
    y0, r0, ro0 = oracle.fused_add_fwd(x, np.zeros_like(x), w, 1e-6, zero_centered_gamma=zc)
    yp, rp = oracle.rmsnorm_fwd(x, w, 1e-6, zero_centered_gamma=zc)
    np.testing.assert_array_equal(y0, yp)
    np.testing.assert_array_equal(r0, rp)
    np.testing.assert_array_equal(ro0, x)


def test_fused_add_sum_is_rounded_to_fp32_before_the_norm():
    """The norm is taken over the fp32 sum h = fl32(x + res), not over the exact
    sum (the reading of [ZC-norm]'s fused add: one fp32 add). Rows whose residual
    dwarfs x (an exponent gap of about 20, so x + res needs more than 24 bits)
    are drawn until some of them have a different correctly rounded rstd for the
    fp32 sum than for the exact one; on every row the oracle's rstd must be the
    one of the fp32 sum, and y follows from it."""
    getcontext().prec = 60
    T, D = 96, 8
    rng = np.random.default_rng(77)
    res = _bf16_grid(rng.standard_normal((T, D)) * 2.0**12)
    x = _bf16_grid(rng.standard_normal((T, D)) * 2.0**-8)
    w = np.float32(rng.standard_normal(D) * 0.3 + 1.0).astype(np.float64)
    eps = Fraction(float(np.float32(1e-6)))
    y, rstd, _ = oracle.fused_add_fwd(x, res, w, 1e-6)

    def rstd_of(h):
        ms = sum(Fraction(v) ** 2 for v in h) / D + eps
        return fp32_round_exact(Fraction(Decimal(1) / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()))

    telling = 0
    for t in range(T):
        exact = [Fraction(x[t, j]) + Fraction(res[t, j]) for j in range(D)]  # exact in double too
        h32 = [float(np.float32(float(v))) for v in exact]
        want = rstd_of(h32)
        telling += want != rstd_of(exact)
        assert rstd[t] == want, t
        for j in range(D):
            assert y[t, j] == bf16_round_bruteforce(Fraction(h32[j]) * Fraction(rstd[t]) * Fraction(w[j]))
    assert telling >= 4, telling  # the case tells the two sums apart


# ==========================================================================
# Gated norm, HF convention (witness of the convention divergence)
# ==========================================================================

def test_gated_hf_convention_divergence_matches_the_pages():
    """bf16, D=128, 512 rows, randn weights: the HF and vLLM conventions agree on
    roughly two thirds of the elements and differ by at most a few bf16 ulps of
    values near 10 (the page: 65 %, max |d| 6.25e-2); with no rounding at all
    (the fp32-input case, where the casts are no-ops) they are identical."""
    gold = _golden("zc_norm_gated_conventions.json")
    g = torch.Generator().manual_seed(0)
    x = torch.randn(gold["rows"], gold["D"], generator=g).to(torch.bfloat16).double().numpy()
    z = torch.randn(gold["rows"], gold["D"], generator=g).to(torch.bfloat16).double().numpy()
    w = np.float32(torch.randn(gold["D"], generator=g).double().numpy()).astype(np.float64)
    yv, rv = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=False)
    yh, rh = oracle.gated_hf_fwd(x, z, w, 1e-6, zero_centered_gamma=False)
    np.testing.assert_array_equal(rv, rh)
    same = float(np.mean(yv == yh))
    mx = float(np.abs(yv - yh).max())
    assert abs(same - gold["same_fraction"]) < 0.15, same
    assert gold["max_abs_diff"] / 2 <= mx <= 2 * gold["max_abs_diff"], mx
    ye, _ = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=False, rounded=False)
    yhe, _ = oracle.gated_hf_fwd(x, z, w, 1e-6, zero_centered_gamma=False, rounded=False)
    np.testing.assert_array_equal(ye, yhe)


def _bf16_rn(v):
    """Nearest bf16 (ties to even) of normal doubles: 8 significant bits."""
    m, e = np.frexp(v)
    return np.ldexp(np.round(m * 256) / 256, e)


def test_gated_hf_reading_is_a_choice_the_page_figure_does_not_make():
    """The page gives no cast points for the HF-convention gated norm, only that
    its weight multiply is not the vLLM one's fp32 multiply, and the 65 % figure.
    Three readings, all with the normalised value cast to bf16, measured on the
    page's setup (seed 0, randn weights): the oracle's (bf16 weight, product
    rounded to bf16) agrees with the vLLM convention on 60.1 %; keeping the
    product in fp32 with a bf16 weight gives 66.7 %; an fp32 weight and product
    74.2 %. The page's band (65 % +- 15) takes all three, so it cannot choose
    between them: these exact fractions make a change of the oracle's reading a
    visible decision rather than a silent one."""
    gold = _golden("zc_norm_gated_conventions.json")
    g = torch.Generator().manual_seed(0)
    x = torch.randn(gold["rows"], gold["D"], generator=g).to(torch.bfloat16).double().numpy()
    z = torch.randn(gold["rows"], gold["D"], generator=g).to(torch.bfloat16).double().numpy()
    w = np.float32(torch.randn(gold["D"], generator=g).double().numpy()).astype(np.float64)
    yv, rv = oracle.gated_fwd(x, z, w, 1e-6, zero_centered_gamma=False)
    yh, _ = oracle.gated_hf_fwd(x, z, w, 1e-6, zero_centered_gamma=False)
    n = _bf16_rn(np.float32(x * rv[:, None]).astype(np.float64))   # the normalised value, cast to bf16
    silu = z / (1.0 + np.exp(-z))
    y_fp32_w = _bf16_rn(np.float32(w[None, :] * n).astype(np.float64) * silu)
    y_bf16_w = _bf16_rn(np.float32(_bf16_rn(w)[None, :] * n).astype(np.float64) * silu)
    fractions = {name: float(np.mean(y == yv)) for name, y in
                 (("oracle", yh), ("bf16 weight, fp32 product", y_bf16_w), ("fp32 weight", y_fp32_w))}
    assert abs(fractions["oracle"] - 0.601) < 0.005, fractions
    assert abs(fractions["bf16 weight, fp32 product"] - 0.667) < 0.005, fractions
    assert abs(fractions["fp32 weight"] - 0.742) < 0.005, fractions
    for f in fractions.values():
        assert abs(f - gold["same_fraction"]) < 0.15, fractions


def test_gated_hf_rounding_points_bruteforce():
    """Each of the HF reading's casts, checked with rationals and the bf16 table."""
    T, D = 2, 16
    x = _bf16_grid(RNG.standard_normal((T, D)))
    z = _bf16_grid(RNG.standard_normal((T, D)))
    w = np.float32(RNG.standard_normal(D)).astype(np.float64)
    y, r = oracle.gated_hf_fwd(x, z, w, 1e-6)
    for t in range(T):
        for j in range(D):
            n = bf16_round_bruteforce(Fraction(float(np.float32(Fraction(x[t, j]) * Fraction(r[t])))))
            wb = bf16_round_bruteforce(Fraction(w[j]))
            tt = bf16_round_bruteforce(Fraction(float(np.float32(Fraction(wb) * Fraction(n)))))
            silu = z[t, j] / (1.0 + math.exp(-z[t, j]))
            assert abs(y[t, j] - bf16_round_bruteforce(Fraction(tt) * Fraction(silu))) <= \
                abs(y[t, j]) * 2.0**-40  # silu rounded to double only


def test_gated_hf_apply_is_the_forward_given_its_rstd():
    x = _bf16_grid(RNG.standard_normal((4, 32)))
    z = _bf16_grid(RNG.standard_normal((4, 32)))
    w = np.float32(RNG.standard_normal(32)).astype(np.float64)
    y, r = oracle.gated_hf_fwd(x, z, w, 1e-6, zero_centered_gamma=True)
    np.testing.assert_array_equal(oracle.gated_hf_apply(x, z, w, r, zero_centered_gamma=True), y)
