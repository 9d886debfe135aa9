"""Shared test helpers: exact conversions, bf16 ulps, tolerances and finite differences.

Nothing here computes the normalisation; it only converts and compares.
"""
from __future__ import annotations

import bisect
import math
from fractions import Fraction

import numpy as np
import torch


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact conversion of a bf16/fp32 tensor (any device) to a float64 numpy array."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (the gap to the next larger magnitude)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, e, -126.0)
    e = np.maximum(e, -126.0)
    return np.exp2(e - 7.0)


# --------------------------------------------------------------------------
# Brute-force bf16 rounding: nearest entry of the table of all bf16 values.
# --------------------------------------------------------------------------
_BF16_POS = None


def _bf16_table():
    global _BF16_POS
    if _BF16_POS is None:
        bits = torch.arange(0, 0x7F80, dtype=torch.int32).to(torch.int16)
        vals = bits.view(torch.bfloat16).to(torch.float64).tolist()
        _BF16_POS = [Fraction(v) for v in vals]  # ascending, 0 .. max finite
    return _BF16_POS


def bf16_round_bruteforce(v) -> float:
    """Nearest bf16 value to the exact rational ``v`` (ties to the even bit pattern)."""
    v = Fraction(v)
    tab = _bf16_table()
    a = abs(v)
    top = tab[-1]
    half_gap_top = (top - tab[-2]) / 2
    if a >= top + half_gap_top:
        return math.copysign(math.inf, v)
    i = bisect.bisect_right(tab, a) - 1  # tab[i] <= a < tab[i+1]
    if tab[i] == a or i == len(tab) - 1:
        r, idx = tab[i], i
    else:
        lo, hi = tab[i], tab[i + 1]
        dl, dh = a - lo, hi - a
        if dl < dh or (dl == dh and i % 2 == 0):
            r, idx = lo, i
        else:
            r, idx = hi, i + 1
    out = float(r)
    return -out if v < 0 else out


# --------------------------------------------------------------------------
# Finite differences (central, float64)
# --------------------------------------------------------------------------
def fd_grad(loss, arr: np.ndarray, h: float = 1e-5) -> np.ndarray:
    """Central-difference gradient of the scalar ``loss()`` with respect to ``arr``
    (perturbed in place and restored)."""
    grad = np.zeros_like(arr)
    flat = arr.reshape(-1)
    gflat = grad.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        step = h * max(1.0, abs(old))
        flat[i] = old + step
        lp = loss()
        flat[i] = old - step
        lm = loss()
        flat[i] = old
        gflat[i] = (lp - lm) / (2 * step)
    return grad


# --------------------------------------------------------------------------
# Parity tolerances
# --------------------------------------------------------------------------
U32 = 2.0 ** -24


def check_bf16_within_1ulp(got: np.ndarray, ref_rounded: np.ndarray):
    """Spec bar for bf16 outputs: |got - RN(ref)| <= 1 bf16 ulp of RN(ref).
    Returns the boolean pass mask."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref_rounded, np.float64)
    same_special = (np.isnan(got) & np.isnan(ref)) | (np.isinf(got) & (got == ref))
    return same_special | (np.abs(got - ref) <= bf16_ulp(ref))
