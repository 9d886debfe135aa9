"""Every pin of the oracle can fail: plausible mistakes planted in the oracle
are each caught by at least one pin.

Each entry below alters one spot of ``oracle/rmsnorm_oracle.c`` the way a
slip in writing it could have: a wrong divisor or exponent, a dropped term or
rounding, a flipped sign, an operand used twice or left out, the wrong gate.
The altered source is compiled on the CPU into ``oracle/_build/mutants/`` and
the pin suites (``tests/test_oracle_pins.py``, ``tests/test_oracle_pins_options.py``)
run against it in a child process (the oracle package loads the library that
``RMSN_ORACLE_LIB`` names). The test requires every such run to fail. A
mistake no pin notices would mean the oracle could carry it unseen into every
parity comparison.

Sources the mistakes refer to: [Megatron] Megatron-LM pull request 6859 "Fix
the batch-invariant RMSNorm forward and its input gradient" (item 1: the
zero-centred offset; item 2: the input gradient, whose defect was a second
weight factor); [ZC-norm] RL-Kernel pull request 467 "[WS1][CUDA][Qwen3-Next]
C1: zero-centred RMSNorm references and CUDA kernel" (gates, conventions, fused
add); [Residual] RL-Kernel pull request 414 "[DSv4][P1-5] rmsnorm_residual"
(Implementation: fp32 saved inverse RMS and weight gradient, bf16 outputs).
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import oracle.build as oracle_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(oracle_build.OUT_DIR, "mutants")
PINS = ["tests/test_oracle_pins.py", "tests/test_oracle_pins_options.py"]

# (name, text in the oracle source, what a slip would have written instead)
MUTANTS = [
    # rounding to the activation formats
    ("bf16_one_bit_short", "int q = (e < -126) ? -133 : e - 7;", "int q = (e < -126) ? -133 : e - 8;"),
    ("bf16_ties_away", "double nr = nearbyint(n);", "double nr = floor(n + 0.5);"),
    ("bf16_no_overflow", "if (r >= ldexp(1.0, 128)) r = INFINITY;", "if (r > ldexp(1.0, 128)) r = INFINITY;"),
    ("bf16_subnormal_quantum", "int q = (e < -126) ? -133 : e - 7;", "int q = (e < -126) ? -134 : e - 7;"),
    ("f16_one_bit_short", "int q = (e < -14) ? -24 : e - 10;", "int q = (e < -14) ? -24 : e - 11;"),
    ("f16_subnormal_quantum", "int q = (e < -14) ? -24 : e - 10;", "int q = (e < -14) ? -25 : e - 10;"),
    ("f16_ties_away", "double r = ldexp(nearbyint(ldexp(a, -q)), q);", "double r = ldexp(floor(ldexp(a, -q) + 0.5), q);"),
    ("f16_truncates", "double r = ldexp(nearbyint(ldexp(a, -q)), q);", "double r = ldexp(trunc(ldexp(a, -q)), q);"),
    ("bf16_truncates", "double nr = nearbyint(n);", "double nr = trunc(n);"),
    ("f16_overflow_late", "if (r >= ldexp(1.0, 16)) r = INFINITY;", "if (r > ldexp(1.0, 16)) r = INFINITY;"),
    ("act_format_bf16_as_f16", "if (rounded == 1) return orc_round_bf16(v);", "if (rounded == 1) return orc_round_f16(v);"),
    ("act_format_f16_as_bf16", "if (rounded == 2) return orc_round_f16(v);", "if (rounded == 2) return orc_round_bf16(v);"),
    # inverse RMS
    ("sum_of_abs", "ss += x[j] * x[j];", "ss += fabs(x[j]);"),
    ("sum_skips_first", "for (int64_t j = 0; j < D; ++j) ss += x[j] * x[j];",
     "for (int64_t j = 1; j < D; ++j) ss += x[j] * x[j];"),
    ("mean_over_d_minus_1", "double mean = ss / (double)D;", "double mean = ss / (double)(D - 1);"),
    ("eps_outside_root", "return 1.0 / sqrt(mean + eps);", "return 1.0 / (sqrt(mean) + eps);"),
    ("rstd_not_fp32",
     "double r = maybe_fl32(row_inv_rms(xr, D, eps), rounded);\n        rstd[t] = r;\n        for (int64_t j = 0; j < D; ++j)\n",
     "double r = row_inv_rms(xr, D, eps);\n        rstd[t] = r;\n        for (int64_t j = 0; j < D; ++j)\n"),
    ("gated_rstd_not_fp32",
     "double r = maybe_fl32(row_inv_rms(xr, D, eps), rounded);\n        rstd[t] = r;\n        for (int64_t j = 0; j < D; ++j) {\n",
     "double r = row_inv_rms(xr, D, eps);\n        rstd[t] = r;\n        for (int64_t j = 0; j < D; ++j) {\n"),
    ("fused_rstd_not_fp32", "double r = maybe_fl32(row_inv_rms(h, D, eps), rounded);", "double r = row_inv_rms(h, D, eps);"),
    ("hf_rstd_not_fp32", "rstd[t] = maybe_fl32(row_inv_rms(x + t * D, D, eps), rounded);",
     "rstd[t] = row_inv_rms(x + t * D, D, eps);"),
    # effective weight
    ("zc_offset_dropped", "return maybe_fl32(w + 1.0, rounded);", "return maybe_fl32(w, rounded);"),
    ("zc_offset_not_fp32", "return maybe_fl32(w + 1.0, rounded);", "return w + 1.0;"),
    # forward
    ("fwd_drops_r", "maybe_act(xr[j] * r * w_eff(w[j], zero_centered, rounded), rounded);",
     "maybe_act(xr[j] * w_eff(w[j], zero_centered, rounded), rounded);"),
    ("fwd_drops_weight", "maybe_act(xr[j] * r * w_eff(w[j], zero_centered, rounded), rounded);",
     "maybe_act(xr[j] * r, rounded);"),
    # input gradient
    ("dx_double_weight", "double b = (r * r * r * xr[k] / (double)D) * s;",
     "double b = w_eff(w[k], zero_centered, rounded) * (r * r * r * xr[k] / (double)D) * s;"),
    ("dx_sign", "double v = a - b;", "double v = a + b;"),
    ("dx_r_not_cubed", "double b = (r * r * r * xr[k] / (double)D) * s;", "double b = (r * xr[k] / (double)D) * s;"),
    ("dx_no_divisor", "double b = (r * r * r * xr[k] / (double)D) * s;", "double b = (r * r * r * xr[k]) * s;"),
    ("dx_first_term_no_r", "double a = gr[k] * w_eff(w[k], zero_centered, rounded) * r;",
     "double a = gr[k] * w_eff(w[k], zero_centered, rounded);"),
    ("dot_without_weight", "double term = gr[i] * xr[i] * w_eff(w[i], zero_centered, rounded);",
     "double term = gr[i] * xr[i];"),
    ("g_res_dropped", "if (g_res) { v += g_res[t * D + k];", "if (g_res) { v += 0.0 * g_res[t * D + k];"),
    ("g_res_subtracted", "if (g_res) { v += g_res[t * D + k];", "if (g_res) { v -= g_res[t * D + k];"),
    # weight gradient
    ("dw_drops_r", "double term = gt * x[t * D + j] * r[t];", "double term = gt * x[t * D + j];"),
    ("dw_not_fp32", "dw[j] = maybe_fl32(acc, rounded);", "dw[j] = acc;"),
    ("dw_keeps_last_term", "acc += term;", "acc = term;"),
    ("dw_transposed_x", "double term = gt * x[t * D + j] * r[t];", "double term = gt * x[j * T + t] * r[t];"),
    ("dw_ignores_gate", "if (z) gt *= gate_q(z[t * D + j], gate);", "if (z) gt *= 1.0;"),
    # gates
    ("sigmoid_sign", "static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }",
     "static double sigmoid(double z) { return 1.0 / (1.0 + exp(z)); }"),
    ("silu_is_sigmoid", "static double silu(double z) { return z * sigmoid(z); }",
     "static double silu(double z) { return sigmoid(z); }"),
    ("dsilu_wrong", "sg * (1.0 + z * (1.0 - sg));", "sg * (1.0 + z * sg);"),
    ("dsigmoid_wrong", "return gate ? sg * sigmoid(-z) : sg * (1.0 + z", "return gate ? sg * sigmoid(z) : sg * (1.0 + z"),
    ("gate_option_ignored", "static double gate_q(double z, int gate) { return gate ? sigmoid(z) : silu(z); }",
     "static double gate_q(double z, int gate) { return silu(z); }"),
    ("gated_dx_without_gate", "double a = gr[k] * gate_q(zr[k], gate) * we * r;", "double a = gr[k] * we * r;"),
    ("gated_dot_without_gate", "double term = gr[i] * gate_q(zr[i], gate) * xr[i] * w_eff(w[i], zero_centered, rounded);",
     "double term = gr[i] * xr[i] * w_eff(w[i], zero_centered, rounded);"),
    ("gated_dz_drops_r", "double u = xr[k] * r * we;", "double u = xr[k] * we;"),
    ("gated_bwd_ignores_zc", "double we = w_eff(w[k], zero_centered, rounded);", "double we = w[k];"),
    ("gated_fwd_ignores_zc", "double u = xr[j] * r * w_eff(w[j], zero_centered, rounded);", "double u = xr[j] * r * w[j];"),
    ("gated_fwd_drops_gate", "y[t * D + j] = maybe_act(u * gate_q(z[t * D + j], gate), rounded);",
     "y[t * D + j] = maybe_act(u, rounded);"),
    # fused add + norm
    ("fused_sum_not_fp32", "for (int64_t j = 0; j < D; ++j) h[j] = maybe_fl32(x[t * D + j] + res[t * D + j], rounded);",
     "for (int64_t j = 0; j < D; ++j) h[j] = x[t * D + j] + res[t * D + j];"),
    ("fused_norm_of_rounded_sum",
     "for (int64_t j = 0; j < D; ++j) h[j] = maybe_fl32(x[t * D + j] + res[t * D + j], rounded);",
     "for (int64_t j = 0; j < D; ++j) h[j] = maybe_act(x[t * D + j] + res[t * D + j], rounded);"),
    ("fused_res_out_unrounded", "h[j] = maybe_act(h[j], rounded);", "h[j] = h[j];"),
    ("fused_bwd_at_x", "orc_rmsnorm_bwd(T, D, g, h_scratch, w,", "orc_rmsnorm_bwd(T, D, g, x, w,"),
    ("fused_bwd_drops_res", "h_scratch[t * D + j] = maybe_fl32(x[t * D + j] + res[t * D + j], rounded);",
     "h_scratch[t * D + j] = maybe_fl32(x[t * D + j], rounded);"),
    # HF-convention gated forward
    ("hf_no_cast_of_normalised", "double n = maybe_act(maybe_fl32(x[t * D + j] * r, rounded), rounded);",
     "double n = maybe_fl32(x[t * D + j] * r, rounded);"),
    ("hf_no_cast_of_weight", "double wb = maybe_act(w_eff(w[j], zero_centered, rounded), rounded);",
     "double wb = w_eff(w[j], zero_centered, rounded);"),
    ("hf_product_not_cast", "double tt = maybe_act(maybe_fl32(wb * n, rounded), rounded);",
     "double tt = maybe_fl32(wb * n, rounded);"),
    ("hf_sigmoid_for_silu", "y[t * D + j] = maybe_act(tt * silu(z[t * D + j]), rounded);",
     "y[t * D + j] = maybe_act(tt * sigmoid(z[t * D + j]), rounded);"),
]


def _build(name: str, src: str) -> str:
    """Compile one altered copy with the oracle's own flags (single-threaded)."""
    os.makedirs(OUT, exist_ok=True)
    c_path = os.path.join(OUT, name + ".c")
    so_path = os.path.join(OUT, name + ".so")
    with open(c_path, "w") as f:
        f.write(src)
    res = subprocess.run(["gcc", *oracle_build._BASE_FLAGS, c_path, "-o", so_path, "-lm"],
                         capture_output=True, text=True)
    assert res.returncode == 0, f"{name}: altered oracle does not compile:\n{res.stderr}"
    return so_path


def _pins_against(so_path: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, RMSN_ORACLE_LIB=so_path, OMP_NUM_THREADS="1")
    return subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_mutant_table_is_well_formed():
    """Every altered text occurs exactly once in the oracle source, and every
    entry changes it (so each mutant is the one slip it names)."""
    src = open(oracle_build.SRC).read()
    names = [m[0] for m in MUTANTS]
    assert len(set(names)) == len(names)
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, (name, src.count(old))
        assert old != new, name


def test_every_planted_mistake_fails_a_pin():
    src = open(oracle_build.SRC).read()
    libs = {name: _build(name, src.replace(old, new, 1)) for name, old, new in MUTANTS}
    with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as pool:
        runs = dict(zip(libs, pool.map(_pins_against, libs.values())))
    survived = [n for n, r in runs.items() if r.returncode == 0]
    broken = {n: r.returncode for n, r in runs.items() if r.returncode not in (0, 1)}
    assert not survived, f"mistakes no pin catches: {survived}"
    assert not broken, f"pin runs that errored instead of failing: {broken}"
    # and the unaltered source passes the same runs
    ok = _pins_against(_build("unaltered", src))
    assert ok.returncode == 0, ok.stdout[-2000:]
