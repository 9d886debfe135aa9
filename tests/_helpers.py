"""Shared test helpers: exact conversions, bf16 ulps, tolerances and finite differences.

Nothing here computes the normalisation; it only converts and compares.
"""
from __future__ import annotations

import bisect
import glob
import math
import os
import re
from fractions import Fraction

import numpy as np
import torch

ROOT_DIR = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact conversion of a bf16/fp16/fp32 tensor (any device) to a float64 numpy array."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (the gap to the next larger magnitude)."""
    return act_ulp(v, "bf16")


# (fraction bits, smallest normal exponent) of each activation format
_FORMATS = {"bf16": (7, -126), "f16": (10, -14)}


def act_ulp(v: np.ndarray, fmt: str = "bf16") -> np.ndarray:
    """Spacing of ``fmt`` numbers at |v| (the gap to the next larger magnitude;
    the subnormal spacing below the normal range)."""
    mant, emin = _FORMATS[fmt]
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, e, float(emin))
    e = np.maximum(e, float(emin))
    return np.exp2(e - float(mant))


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


_F16_POS = None


def _f16_table():
    global _F16_POS
    if _F16_POS is None:
        bits = torch.arange(0, 0x7C00, dtype=torch.int32).to(torch.int16)
        vals = bits.view(torch.float16).to(torch.float64).tolist()
        _F16_POS = [Fraction(v) for v in vals]  # ascending, 0 .. 65504
    return _F16_POS


def bf16_round_bruteforce(v) -> float:
    """Nearest bf16 value to the exact rational ``v`` (ties to the even bit pattern)."""
    return _round_bruteforce(v, _bf16_table())


def f16_round_bruteforce(v) -> float:
    """Nearest IEEE fp16 value to the exact rational ``v`` (ties to the even bit pattern)."""
    return _round_bruteforce(v, _f16_table())


def fp32_round_exact(v) -> float:
    """Nearest fp32 value to the exact rational ``v`` (ties to the even bit
    pattern), by exact comparison of the candidates' distances. The double
    nearest to v, cast to fp32, is the answer or a neighbour of it (a double
    rounding errs by at most one step), so those three are the candidates."""
    v = Fraction(v)
    f = np.float32(float(v))
    cands = [c for c in (f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf)))
             if np.isfinite(c)]
    return float(min(cands, key=lambda c: (abs(Fraction(float(c)) - v),
                                           int(np.array(c, np.float32).view(np.uint32)) & 1)))


def _round_bruteforce(v, tab) -> float:
    v = Fraction(v)
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


def check_bf16_within_1ulp(got: np.ndarray, ref_rounded: np.ndarray, fmt: str = "bf16"):
    """The bar for 16-bit outputs: |got - RN(ref)| <= 1 ulp of RN(ref) in the
    output format ``fmt`` (bf16, or fp16). Returns the boolean pass mask."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref_rounded, np.float64)
    same_special = (np.isnan(got) & np.isnan(ref)) | (np.isinf(got) & (got == ref))
    with np.errstate(invalid="ignore"):  # inf - inf where both are special: decided above
        return same_special | (np.abs(got - ref) <= act_ulp(ref, fmt))


def _ulp_of_max(a, b, fmt="bf16"):
    return act_ulp(np.maximum(np.abs(a), np.abs(b)), fmt)


def bf16_parity_mask(got, ref_rounded, pre=None, scale=None, K: float = 96.0, fmt: str = "bf16"):
    """Parity of a 16-bit output (format ``fmt``, bf16 by default) with the oracle.

    Clause 1 (the bar): |got - RN(ref)| <= 1 ulp of RN(ref).
    Clause 2 (only with ``pre``/``scale``, for outputs whose terms cancel):
    |got - ref| <= 1/2 ulp + K * 2^-24 * scale, where ``ref`` is the exact
    pre-rounding value and ``scale`` the magnitude of its terms: the error an
    fp32 evaluation with at most K separately rounded steps can make, plus the
    final rounding to the output format. Returns (mask, n_clause2).
    """
    got = np.asarray(got, np.float64)
    m1 = check_bf16_within_1ulp(got, ref_rounded, fmt)
    if pre is None:
        return m1, 0
    m2 = np.abs(got - pre) <= 0.5 * _ulp_of_max(got, pre, fmt) + K * U32 * scale
    return m1 | m2, int(np.count_nonzero(m2 & ~m1))


def assert_bf16_parity(name, got, ref_rounded, pre=None, scale=None, K: float = 96.0, fmt: str = "bf16"):
    mask, n2 = bf16_parity_mask(got, ref_rounded, pre, scale, K, fmt)
    bad = np.argwhere(~mask)
    if bad.size:
        i = tuple(bad[0])
        msg = f"{name}: {len(bad)} of {mask.size} outside tolerance; first at {i}: got {got[i]!r} " \
              f"ref {ref_rounded[i]!r}"
        if pre is not None:
            msg += f" pre {pre[i]!r} scale {scale[i]!r}"
        raise AssertionError(msg)
    return n2


def assert_rel(name, got, ref, rtol):
    got = np.asarray(got, np.float64)
    ok = np.abs(got - ref) <= rtol * np.abs(ref)
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError(f"{name}: {np.count_nonzero(~ok)} outside rtol {rtol}; first at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r}")


def dgamma_bound_gamma(chunk_rows: int, nchunks: int, reduce_warps: int = 32) -> float:
    """Rounding-error factor of the library's fixed weight-gradient tree: products
    (2-3 roundings, +8 for a gate), C sequential adds per chunk, ceil(n/32)
    sequential adds per warp in pass 2, 32 warp totals."""
    return (chunk_rows + -(-nchunks // reduce_warps) + reduce_warps + 8) * U32


def assert_dgamma_parity(name, got, ref, abs_sum, chunk_rows: int, nchunks: int):
    """|got - ref| <= 1e-4 |ref| (the bar), or within the fixed tree's forward-error
    bound gamma * sum|terms| for columns whose sum cancels. Returns n_clause2."""
    got = np.asarray(got, np.float64)
    m1 = np.abs(got - ref) <= 1e-4 * np.abs(ref)
    m2 = np.abs(got - ref) <= dgamma_bound_gamma(chunk_rows, nchunks) * abs_sum
    ok = m1 | m2
    if not ok.all():
        i = int(np.argwhere(~ok)[0][0])
        raise AssertionError(f"{name}: {np.count_nonzero(~ok)} columns outside tolerance; first {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} sum|t| {abs_sum[i]!r}")
    return int(np.count_nonzero(m2 & ~m1))


WIDE_CHUNK_ROWS = 32    # longest weight-gradient chunk of the wide path (D > 256)
PASS2_RANGES = 32       # pass-2 ranges of contiguous chunks
BALANCE_SMS = 152       # the constant the wide chunk rule balances for


def wide_chunk_rows(T: int, D: int) -> int:
    """The wide backward's chunk rule: 32 rows, except for 2048 < D <= 7168
    when 32-row chunks fill less than 90 % of their rounds of 152 x 2 CTAs;
    then 32 rows shortened just enough that the chunks come in whole rounds."""
    c0 = WIDE_CHUNK_ROWS
    if D <= 2048 or D > 7168 or T <= 0:
        return c0
    ctas = BALANCE_SMS * 2
    n0 = -(-T // c0)
    if n0 <= ctas:
        return c0
    rounds = -(-n0 // ctas)
    if 10 * n0 >= 9 * rounds * ctas:
        return c0
    return -(-T // (rounds * ctas))


def _pass2(partials):
    """The fixed pass-2 tree over chunk partials [n, D] (float32)."""
    nch, D = partials.shape
    per = -(-nch // PASS2_RANGES)
    totals = []
    for w in range(PASS2_RANGES):
        s = np.zeros(D, np.float32)
        for c in range(w * per, min(nch, (w + 1) * per)):
            s = s + partials[c]
        totals.append(s)
    out = totals[0]
    for w in range(1, PASS2_RANGES):
        out = out + totals[w]
    return out


def _accumulate(acc, gx, rt, fused):
    if fused:
        return (gx.astype(np.float64) * np.float64(rt) + acc.astype(np.float64)).astype(np.float32)
    return acc + gx * rt


def dgamma_model(g, h, r, fused: bool = False):
    """float32 model of the weight gradient: ((g*h)*r) per element, each
    multiply and add rounded to fp32, summed per chunk in the order the path
    fixes, then the chunk partials through the pass-2 tree (32 contiguous
    ranges of ceil(n/32) chunks in ascending order, the range totals in order).
    g, h [T, D] and r [T] are float32 and exact. D > 256 (wide path): chunks of
    wide_chunk_rows(T, D) rows, rows in ascending order. D <= 256 (narrow path): G = next power of
    two of D/8 lanes per row, P = 256/G rows per pass, stages of RS = 32 rows
    (P if larger; 32 when G = 32), chunks of max(RS, 128) rows; lane group q
    adds the rows chunk + s*RS + p*P + q, stage by stage and pass by pass, and
    the chunk partial is the group totals added in group order. With
    fused=True the per-row update is a fused multiply-add instead (acc + gx*r
    rounded once), the rounding the kernels must not do."""
    T, D = g.shape
    if D > 256:
        C = wide_chunk_rows(T, D)
        nch = -(-T // C)
        partials = np.zeros((nch, D), np.float32)
        for c in range(nch):
            acc = np.zeros(D, np.float32)
            for t in range(c * C, min(T, (c + 1) * C)):
                acc = _accumulate(acc, g[t] * h[t], r[t], fused)
            partials[c] = acc
        return _pass2(partials)
    G = 1
    while G < D // 8:
        G *= 2
    P = 256 // G
    RS = 32 if G == 32 else max(P, 32)
    CN = max(RS, 128)
    nch = -(-T // CN)
    partials = np.zeros((nch, D), np.float32)
    for c in range(nch):
        groups = []
        for q in range(P):
            acc = np.zeros(D, np.float32)
            for st in range(CN // RS):
                for p in range(RS // P):
                    t = c * CN + st * RS + p * P + q
                    if t < T:
                        acc = _accumulate(acc, g[t] * h[t], r[t], fused)
            groups.append(acc)
        tot = groups[0]
        for q in range(1, P):
            tot = tot + groups[q]
        partials[c] = tot
    return _pass2(partials)


def f32_round_act(v, fmt: str = "bf16") -> np.ndarray:
    """float32 values rounded to bf16 or fp16, nearest even, returned as float32."""
    v = np.asarray(v, np.float32)
    if fmt == "f16":
        return v.astype(np.float16).astype(np.float32)
    bits = v.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32)


def _wide_shape(NV: int, ntmax: int):
    """Threads (a multiple of 32) and vectors a thread for NV vectors on at most
    ntmax threads (512 beyond 4*ntmax vectors); 1, 2 or 4 vectors each."""
    if NV > 4 * ntmax:
        ntmax = 512
    need = -(-NV // ntmax)
    vpt = 1 if need <= 1 else (2 if need <= 2 else 4)
    return -(-(-(-NV // vpt)) // 32) * 32, vpt


def bwd_row_shape(D: int, mode: str):
    """Consumer threads and 16-byte vectors a thread of the wide backward's row
    reduction, a function of D and the mode: up to 256 threads, 1, 2 or 4
    vectors each; plain rows of at most 256 vectors on at most 128 threads; rows
    of 897..1024 vectors on 512 threads, and in every mode but the plain one
    already rows of 513..896 vectors. Rows of more than 1024 vectors are split
    between two CTAs (bwd_is_pair): the shape is then each half's, for
    ceil(NV/2) vectors on up to 512 threads."""
    NV = D // 8
    if bwd_is_pair(D, mode):
        return _wide_shape((NV + 1) // 2, 512)
    nt, vpt = _wide_shape(NV, 256)
    if mode == "plain" and NV <= 256:
        nt, vpt = _wide_shape(NV, 128)
    if 897 <= NV <= 1024 or (mode != "plain" and 513 <= NV <= 896):
        nt, vpt = _wide_shape(NV, 512)
    return nt, vpt


def bwd_is_pair(D: int, mode: str) -> bool:
    """Rows of more than 1024 vectors (D > 8192; in the plain mode only up to
    1152 vectors, D <= 9216): the two CTAs of a cluster take the first
    ceil(NV/2) vectors and the rest, and add their halves in that order."""
    NV = D // 8
    return NV > 1024 and (mode != "plain" or NV <= 1152)


def _thread_tree(vec, nt: int, vpt: int):
    """One CTA's part of the tree over vec [T, NVc, 8]: thread t adds its
    vectors v = j*nt + t (j ascending, the 8 elements of each in order) from 0,
    an xor butterfly over each warp (offsets 16..1), the warp totals in order."""
    T, NVc = vec.shape[0], vec.shape[1]
    th = np.zeros((T, nt), np.float32)
    for j in range(vpt):
        for t0 in range(nt):
            v = j * nt + t0
            if v < NVc:
                for e in range(8):
                    th[:, t0] = th[:, t0] + vec[:, v, e]
    nw = nt // 32
    warps = th.reshape(T, nw, 32)
    o = 16
    while o > 0:
        warps = warps + warps[:, :, np.arange(32) ^ o]
        o //= 2
    s = warps[:, 0, 0]
    for i in range(1, nw):
        s = s + warps[:, i, 0]
    return s


def row_sums_model(terms, D: int, mode: str):
    """The fixed row reduction of [T, D] float32 terms: on the wide path each
    consumer thread t adds its elements (vectors v = j*NT + t, j ascending, the 8
    elements of each in order) from 0, an xor butterfly over each warp (offsets
    16..1) gives every lane the warp total, and the warp totals are added in
    warp order; rows of more than 1024 vectors do that over each half (the first
    ceil(NV/2) vectors, the rest) and add the two totals, first half first; on
    the narrow path (D <= 256) each lane of a row's group of G = next_pow2(D/8)
    lanes adds its 8 elements and a butterfly over the group (offsets G/2..1)
    gives the total."""
    T = terms.shape[0]
    NV = D // 8
    vec = terms.reshape(T, NV, 8)
    if D <= 256:
        G = 1
        while G < NV:
            G *= 2
        lanes = np.zeros((T, G), np.float32)
        for e in range(8):
            lanes[:, :NV] = lanes[:, :NV] + vec[:, :, e]
        o = G // 2
        while o > 0:
            lanes = lanes + lanes[:, np.arange(G) ^ o]
            o //= 2
        return lanes[:, 0]
    nt, vpt = bwd_row_shape(D, mode)
    if bwd_is_pair(D, mode):
        NVh = (NV + 1) // 2
        return _thread_tree(vec[:, :NVh], nt, vpt) + _thread_tree(vec[:, NVh:], nt, vpt)
    return _thread_tree(vec, nt, vpt)


def dx_model(g, h, w_eff, r, mode: str, g_res=None, fmt: str = "bf16"):
    """The backward's input gradient, modelled in float32 and rounded once:
    s = fixed row sum of ((g*w_eff)*h); coef = (((r*r)*r) / D) * s (a power-of-two D
    scales by its exact reciprocal); dx = ((g*w_eff)*r) - (h*coef) [+ g_res]."""
    T, D = g.shape
    gw = g * w_eff[None, :]
    s = row_sums_model(gw * h, D, mode)
    r3 = (r * r) * r
    q = r3 * np.float32(1.0 / D) if (D & (D - 1)) == 0 else r3 / np.float32(D)
    coef = q * s
    d = gw * r[:, None] - h * coef[:, None]
    if g_res is not None:
        d = d + g_res
    return f32_round_act(d, fmt)


def header_declarations(root: str = ROOT_DIR):
    """(return type, name, [parameter types]) of every entry point in include/*.h."""
    out = []
    for h in glob.glob(os.path.join(root, "include", "*.h")):
        txt = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        txt = "\n".join(l for l in txt.split("\n") if not l.strip().startswith("#"))
        for ret, name, params in re.findall(r"([A-Za-z_][\w\s\*]*?)\b(rmsnorm_\w+)\s*\(([^)]*)\)\s*;", txt):
            types = [re.sub(r"\b\w+$", "", q.strip()).strip() for q in params.split(",") if q.strip()]
            out.append((" ".join(ret.split()).replace(" *", "*"), name, types))
    return out
