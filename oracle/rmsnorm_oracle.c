/*
 * Float64 CPU oracle for batch-invariant RMSNorm (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or
 * call this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline use it. It shares no code, header or constant with the CUDA library.
 *
 * Sources (cited by the short key in brackets):
 *   [Megatron]  Megatron-LM pull request 6859, "Fix the batch-invariant RMSNorm
 *               forward and its input gradient"
 *   [ZC-norm]   RL-Kernel pull request 467, "[WS1][CUDA][Qwen3-Next] C1: zero-centred
 *               RMSNorm references and CUDA kernel"
 *   [Residual]  RL-Kernel pull request 414, "[DSv4][P1-5] rmsnorm_residual"
 *
 * Everything is evaluated in IEEE double. Rounding happens only at the points
 * the method states, and only when `rounded` is non-zero. Its value names the
 * activation format: 1 = bf16, 2 = fp16 ([ZC-norm]: the op contract carries
 * tolerances for both; the arithmetic between load and store is the same).
 *   - the saved inverse RMS is an fp32 value                  ([Residual], Implementation)
 *   - the zero-centred offset is an fp32 add after the fp32 cast
 *                                     ([Megatron], What does this PR do, item 1;
 *                                      [ZC-norm], the GemmaRMSNorm forward_native note)
 *   - activations and activation gradients are bf16 (or fp16), rounded to
 *     nearest even                                            ([Residual], Implementation)
 *   - the weight gradient is an fp32 value                    ([Residual], Implementation)
 * With `rounded == 0` nothing is rounded: that mode is the plain mathematical
 * function, used by the finite-difference checks.
 *
 * Arrays are dense row-major: activations [T][D], weights [D], inverse RMS [T].
 * Sums run over the index in ascending order with one double accumulator.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Round a double to the nearest bf16 value (8 significant bits, fp32 exponent
 * range), ties to even, in ONE rounding step from the double. Returns the
 * rounded value as a double (exactly representable). */
double orc_round_bf16(double v) {
    if (isnan(v)) return v;
    if (isinf(v)) return v;
    double a = fabs(v);
    if (a == 0.0) return v;
    int E;
    (void)frexp(a, &E);               /* a = m * 2^E, m in [0.5, 1) */
    int e = E - 1;                    /* a in [2^e, 2^(e+1)) */
    int q = (e < -126) ? -133 : e - 7; /* quantum exponent: normal 2^(e-7), subnormal 2^-133 */
    double n = ldexp(a, -q);          /* exact scaling by a power of two */
    double nr = nearbyint(n);         /* default mode: round half to even */
    double r = ldexp(nr, q);
    /* Overflow: anything that rounds to 2^128 or beyond is infinite in bf16. */
    if (r >= ldexp(1.0, 128)) r = INFINITY;
    return signbit(v) ? -r : r;
}

/* Round a double to the nearest IEEE binary16 value (11 significant bits,
 * normal exponents -14..15, subnormal quantum 2^-24), ties to even, in ONE
 * rounding step from the double; overflow (a result of 2^16 or beyond) is
 * infinite. Returns the rounded value as a double. */
double orc_round_f16(double v) {
    if (isnan(v)) return v;
    if (isinf(v)) return v;
    double a = fabs(v);
    if (a == 0.0) return v;
    int E;
    (void)frexp(a, &E);
    int e = E - 1;                     /* a in [2^e, 2^(e+1)) */
    int q = (e < -14) ? -24 : e - 10;  /* quantum exponent */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r >= ldexp(1.0, 16)) r = INFINITY;
    return signbit(v) ? -r : r;
}

/* Round a double to fp32 (C conversion, round to nearest even). */
static double fl32(double v) { return (double)(float)v; }

/* An activation output in the format `rounded` names (0: unrounded). */
static double maybe_act(double v, int rounded) {
    if (rounded == 1) return orc_round_bf16(v);
    if (rounded == 2) return orc_round_f16(v);
    return v;
}
static double maybe_fl32(double v, int rounded) { return rounded ? fl32(v) : v; }

/* Effective weight: w, or w + 1 applied in fp32 after the fp32 cast when the
 * gamma is zero-centred ([Megatron], What does this PR do, item 1). */
static double w_eff(double w, int zero_centered, int rounded) {
    if (!zero_centered) return w;
    return maybe_fl32(w + 1.0, rounded);
}

/* Inverse RMS of one row: r = (mean_j x_j^2 + eps)^(-1/2), mean = (sum x^2) / D
 * ([Megatron], What does this PR do, item 2, definition of r; [Residual], the
 * reviewer's "Forward" summary). */
static double row_inv_rms(const double* x, int64_t D, double eps) {
    double ss = 0.0;
    for (int64_t j = 0; j < D; ++j) ss += x[j] * x[j];
    double mean = ss / (double)D;
    return 1.0 / sqrt(mean + eps);
}

/* silu(z) = z * sigmoid(z), sigmoid(z) = 1 / (1 + exp(-z)). */
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }
static double silu(double z) { return z * sigmoid(z); }

/* The gated norm's gate q(z): silu (gate 0, the default) or sigmoid (gate 1)
 * ([ZC-norm]: the activation is read from the model config, silu by default,
 * sigmoid also allowed), and its derivative q'(z):
 *   silu:    q' = sigmoid(z) (1 + z (1 - sigmoid(z)))
 *   sigmoid: q' = sigmoid(z) (1 - sigmoid(z)) = sigmoid(z) sigmoid(-z)
 * gate_dq_scale is q' with the cancelling term taken in absolute value: the
 * magnitude of the terms q' is made of (for the tolerance of a finite-precision
 * evaluation of q'). */
static double gate_q(double z, int gate) { return gate ? sigmoid(z) : silu(z); }
static double gate_dq(double z, int gate) {
    double sg = sigmoid(z);
    return gate ? sg * sigmoid(-z) : sg * (1.0 + z * (1.0 - sg));
}
static double gate_dq_scale(double z, int gate) {
    double sg = sigmoid(z);
    return gate ? sg * sigmoid(-z) : sg * (1.0 + fabs(z) * (1.0 - sg));
}

/* ------------------------------------------------------------------------ */
/* Plain / zero-centred forward:  y = (x * r) * w_eff,  rstd = r              */
/* ([Megatron], item 1; [Residual], reviewer's "Forward" summary)            */
/* ------------------------------------------------------------------------ */
void orc_rmsnorm_fwd(int64_t T, int64_t D, const double* x, const double* w, double eps,
                     int zero_centered, int rounded, double* y, double* rstd) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* xr = x + t * D;
        double r = maybe_fl32(row_inv_rms(xr, D, eps), rounded);
        rstd[t] = r;
        for (int64_t j = 0; j < D; ++j)
            y[t * D + j] = maybe_act(xr[j] * r * w_eff(w[j], zero_centered, rounded), rounded);
    }
}

/* ------------------------------------------------------------------------ */
/* Weight gradient: dgamma_j = sum_t g_tj * x_tj * r_t  (ascending t)         */
/* ([Megatron], item 2, g_w unchanged; [Residual], reviewer's "for dgamma")  */
/* Gated variant (z != NULL): g is replaced by g * q(z) (gate as in gate_q),  */
/* the gradient that reaches the normalised-and-scaled value.                 */
/* Columns are independent: any column subset may be passed with all T rows.  */
/* dw_abs (may be NULL) receives sum_t |term|, the scale of the rounding     */
/* error any finite-precision evaluation of the sum can make.                */
/* ------------------------------------------------------------------------ */
void orc_weight_grad(int64_t T, int64_t D, const double* g, const double* z, int gate,
                     const double* x, const double* r, int rounded, double* dw, double* dw_abs) {
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < D; ++j) {
        double acc = 0.0, mag = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            double gt = g[t * D + j];
            if (z) gt *= gate_q(z[t * D + j], gate);
            double term = gt * x[t * D + j] * r[t];
            acc += term;
            mag += fabs(term);
        }
        dw[j] = maybe_fl32(acc, rounded);
        if (dw_abs) dw_abs[j] = mag;
    }
}

/* ------------------------------------------------------------------------ */
/* Plain / zero-centred / residual backward.                                  */
/*   s    = sum_i g_i x_i w_eff_i                                             */
/*   dx_k = g_k w_eff_k r - (r^3 x_k / D) * s  [+ g_res_k]                    */
/* ([Megatron], item 2, the dL/dx_k formula; [Residual], reviewer's "for dx", */
/* which adds d_residual)                                                     */
/* `rstd` is the forward's saved value; `g_res` may be NULL (zero).           */
/* Optional diagnostics (each may be NULL): dx_pre = dx before its bf16       */
/* rounding; dx_scale = |g_k w_k r| + (r^3 |x_k| / D) sum_i |g_i x_i w_i|     */
/* [+ |g_res_k|], the magnitude the terms of dx_k had before they cancelled;  */
/* dw_abs as in orc_weight_grad.                                              */
/* ------------------------------------------------------------------------ */
void orc_rmsnorm_bwd(int64_t T, int64_t D, const double* g, const double* x, const double* w,
                     const double* rstd, const double* g_res, int zero_centered, int rounded,
                     double* dx, double* dw, double* dx_pre, double* dx_scale, double* dw_abs) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* gr = g + t * D;
        const double* xr = x + t * D;
        double r = rstd[t];
        double s = 0.0, s_abs = 0.0;
        for (int64_t i = 0; i < D; ++i) {
            double term = gr[i] * xr[i] * w_eff(w[i], zero_centered, rounded);
            s += term;
            s_abs += fabs(term);
        }
        for (int64_t k = 0; k < D; ++k) {
            double a = gr[k] * w_eff(w[k], zero_centered, rounded) * r;
            double b = (r * r * r * xr[k] / (double)D) * s;
            double v = a - b;
            double mag = fabs(a) + (r * r * r * fabs(xr[k]) / (double)D) * s_abs;
            if (g_res) { v += g_res[t * D + k]; mag += fabs(g_res[t * D + k]); }
            dx[t * D + k] = maybe_act(v, rounded);
            if (dx_pre) dx_pre[t * D + k] = v;
            if (dx_scale) dx_scale[t * D + k] = mag;
        }
    }
    orc_weight_grad(T, D, g, NULL, 0, x, rstd, rounded, dw, dw_abs);
}

/* ------------------------------------------------------------------------ */
/* Gated forward (Qwen3-Next, vLLM convention: weight multiply in fp32):      */
/*   u = (x * r) * w_eff,  y = u * q(z),  q = silu (gate 0) or sigmoid (1)    */
/* ([ZC-norm], the two gated-norm conventions: Qwen3NextRMSNormGatedOp)      */
/* ------------------------------------------------------------------------ */
void orc_gated_fwd(int64_t T, int64_t D, const double* x, const double* z, const double* w,
                   double eps, int zero_centered, int gate, int rounded, double* y, double* rstd) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* xr = x + t * D;
        double r = maybe_fl32(row_inv_rms(xr, D, eps), rounded);
        rstd[t] = r;
        for (int64_t j = 0; j < D; ++j) {
            double u = xr[j] * r * w_eff(w[j], zero_centered, rounded);
            y[t * D + j] = maybe_act(u * gate_q(z[t * D + j], gate), rounded);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Gated backward. With q = q(z) and u = x r w_eff (so y = u q):             */
/*   dL/du = g q, which enters the plain backward in place of g:              */
/*     s    = sum_i (g_i q_i) x_i w_eff_i                                     */
/*     dx_k = (g_k q_k) w_eff_k r - (r^3 x_k / D) * s                         */
/*   dz_k = g_k u_k q'(z_k)                                                   */
/*   dw_j = sum_t g_tj q_tj x_tj r_t                                          */
/* ------------------------------------------------------------------------ */
void orc_gated_bwd(int64_t T, int64_t D, const double* g, const double* x, const double* z,
                   const double* w, const double* rstd, int zero_centered, int gate, int rounded,
                   double* dx, double* dz, double* dw,
                   double* dx_pre, double* dx_scale, double* dz_pre, double* dz_scale, double* dw_abs) {
    /* Diagnostics as in orc_rmsnorm_bwd; dz_scale = |g u| gate_dq_scale(z). */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* gr = g + t * D;
        const double* xr = x + t * D;
        const double* zr = z + t * D;
        double r = rstd[t];
        double s = 0.0, s_abs = 0.0;
        for (int64_t i = 0; i < D; ++i) {
            double term = gr[i] * gate_q(zr[i], gate) * xr[i] * w_eff(w[i], zero_centered, rounded);
            s += term;
            s_abs += fabs(term);
        }
        for (int64_t k = 0; k < D; ++k) {
            double we = w_eff(w[k], zero_centered, rounded);
            double a = gr[k] * gate_q(zr[k], gate) * we * r;
            double v = a - (r * r * r * xr[k] / (double)D) * s;
            dx[t * D + k] = maybe_act(v, rounded);
            if (dx_pre) dx_pre[t * D + k] = v;
            if (dx_scale) dx_scale[t * D + k] = fabs(a) + (r * r * r * fabs(xr[k]) / (double)D) * s_abs;
            double u = xr[k] * r * we;
            double d = gr[k] * u * gate_dq(zr[k], gate);
            dz[t * D + k] = maybe_act(d, rounded);
            if (dz_pre) dz_pre[t * D + k] = d;
            if (dz_scale) dz_scale[t * D + k] = fabs(gr[k] * u) * gate_dq_scale(zr[k], gate);
        }
    }
    orc_weight_grad(T, D, g, z, gate, x, rstd, rounded, dw, dw_abs);
}

/* ------------------------------------------------------------------------ */
/* Fused add + RMSNorm (vLLM fused_add_rms_norm, which [ZC-norm] names as    */
/* the path of every decoder norm except layer 0's input norm): the          */
/* norm is applied to the fp32 sum h = x + res, which is also returned       */
/* rounded to the activation format as the new residual stream.             */
/*   h = fl32(x + res);  res_out = act(h);  rstd, y as the plain forward on h  */
/* Reading (the pages give no rounding order): the sum is one fp32 add; the  */
/* normalisation uses that fp32 h, not its rounding to the activation format. */
/* ------------------------------------------------------------------------ */
void orc_fused_add_fwd(int64_t T, int64_t D, const double* x, const double* res, const double* w,
                       double eps, int zero_centered, int rounded,
                       double* y, double* rstd, double* res_out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double* h = res_out + t * D;  /* holds the unrounded sum until the end of the row */
        for (int64_t j = 0; j < D; ++j) h[j] = maybe_fl32(x[t * D + j] + res[t * D + j], rounded);
        double r = maybe_fl32(row_inv_rms(h, D, eps), rounded);
        rstd[t] = r;
        for (int64_t j = 0; j < D; ++j) {
            y[t * D + j] = maybe_act(h[j] * r * w_eff(w[j], zero_centered, rounded), rounded);
            h[j] = maybe_act(h[j], rounded);
        }
    }
}

/* Backward of the fused add + norm. The gradient reaching h is the plain     */
/* backward at h plus the gradient of res_out (g_res, may be NULL = 0); it is */
/* the gradient of both x and res (dh/dx = dh/dres = 1). The weight gradient  */
/* is sum_t g_tj h_tj r_t. h is recomputed from x and res exactly as forward. */
void orc_fused_add_bwd(int64_t T, int64_t D, const double* g, const double* x, const double* res,
                       const double* w, const double* rstd, const double* g_res, int zero_centered,
                       int rounded, double* dh, double* dw, double* h_scratch,
                       double* dh_pre, double* dh_scale, double* dw_abs) {
    /* h_scratch: caller-provided [T][D] buffer that receives h. */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < D; ++j)
            h_scratch[t * D + j] = maybe_fl32(x[t * D + j] + res[t * D + j], rounded);
    orc_rmsnorm_bwd(T, D, g, h_scratch, w, rstd, g_res, zero_centered, rounded, dh, dw, dh_pre, dh_scale,
                    dw_abs);
}

/* ------------------------------------------------------------------------ */
/* Gated norm, HF/transformers convention, forward only ([ZC-norm]: the two  */
/* upstreams round the gated norm differently; the vLLM one multiplies by    */
/* the weight in fp32, and with fp32 inputs the two agree bitwise, since the */
/* cast then changes nothing). Reading: the normalised value is cast to the  */
/* activation dtype (bf16) and the weight multiply happens in that dtype:    */
/*   n = bf16(fl32(x r));  t = bf16(fl32(bf16(w_eff) n));  y = bf16(t silu(z)) */
/* In unrounded mode every cast is the identity, so the function equals the  */
/* vLLM convention's.                                                        */
/* ------------------------------------------------------------------------ */
/* The HF convention's output for given fp32 inverse RMS values. */
void orc_gated_hf_apply(int64_t T, int64_t D, const double* x, const double* z, const double* w,
                        const double* rstd, int zero_centered, int rounded, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double r = rstd[t];
        for (int64_t j = 0; j < D; ++j) {
            double n = maybe_act(maybe_fl32(x[t * D + j] * r, rounded), rounded);
            double wb = maybe_act(w_eff(w[j], zero_centered, rounded), rounded);
            double tt = maybe_act(maybe_fl32(wb * n, rounded), rounded);
            y[t * D + j] = maybe_act(tt * silu(z[t * D + j]), rounded);
        }
    }
}

void orc_gated_hf_fwd(int64_t T, int64_t D, const double* x, const double* z, const double* w,
                      double eps, int zero_centered, int rounded, double* y, double* rstd) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) rstd[t] = maybe_fl32(row_inv_rms(x + t * D, D, eps), rounded);
    orc_gated_hf_apply(T, D, x, z, w, rstd, zero_centered, rounded, y);
}
