/*
 * rmsnorm.h — C ABI of the GB300 (sm_103a) batch-invariant RMSNorm library.
 *
 * Operations (sources, cited by page title and section):
 *   [Megatron]  Megatron-LM pull request 6859, "Fix the batch-invariant RMSNorm
 *               forward and its input gradient" — "What does this PR do", items 1-2.
 *   [ZC-norm]   RL-Kernel pull request 467, "[WS1][CUDA][Qwen3-Next] C1: zero-centred
 *               RMSNorm references and CUDA kernel" — the GemmaRMSNorm forward_native
 *               note (+1 in fp32) and the two gated-norm conventions.
 *   [Residual]  RL-Kernel pull request 414, "[DSv4][P1-5] rmsnorm_residual" —
 *               Summary, Implementation, and the reviewer's Forward/Backward notes.
 *
 * Forward, per row t of x [T][D]:
 *   r_t   = rsqrt( (sum_j x_tj^2) / D + eps )          saved as fp32 rstd[t]
 *   w_eff = w, or (fp32) w + 1.0f when zero_centered_gamma is set
 *   y_tj  = bf16( (x_tj * r_t) * w_eff_j )             two separately rounded fp32 multiplies
 * Backward, per row (g = dL/dy, saved r):
 *   s     = sum_i g_i x_i w_eff_i
 *   dx_k  = bf16( g_k w_eff_k r  -  (r^3 x_k / D) * s  [+ g_res_k] )
 *   dgamma_j = sum_t g_tj x_tj r_t                     fp32
 *
 * Batch invariance: every row is reduced by a fixed tree whose shape depends on
 * D alone (in the backward, on D and the variant called), so y[t], rstd[t] and
 * dx[t] are bitwise independent of T, of the row's position, of the other rows
 * and of the GPU's SM count. In the backward of rows wider than 8192 (in the
 * plain variant, of 8193..9216 only) the tree has one more level: the row's two
 * column halves are reduced by the two CTAs of a thread-block cluster and their
 * sums added, first half first. dgamma is a sum over
 * rows; it is computed with no atomics, in row chunks whose size depends on T
 * and D alone (pass 1), whose partial sums are added in a fixed order (pass 2),
 * so it is bitwise identical from run to run and across GPUs with different
 * SM counts.
 *
 * The weight-gradient chunk: every chunk of one call has the same number of
 * rows (only the last may be shorter), a function of T and D only ("fixed-size
 * row chunks" read as fixed for a given problem shape).
 *
 * Common conventions for every entry point:
 *   - Activations (x, z, g, g_res, y, dx, dz, x_copy) are bf16 (fp16 as an
 *     option of the *_ex calls), row-major [T][D] with a row stride `ld*` in
 *     ELEMENTS (ld >= D). They are passed as raw 16-bit patterns (rmsn_bf16,
 *     rmsn_act16). w / dgamma are fp32 [D]; rstd is fp32 [T].
 *   - All pointers are DEVICE pointers, 16-byte aligned; every ld* is a multiple
 *     of 8 (so each row starts on a 16-byte boundary). D is a multiple of 8 with
 *     8 <= D <= 16384. eps is finite and >= 0. 0 <= T < 2^31; T == 0 returns
 *     RMSN_OK without launching anything.
 *   - Outputs must not overlap inputs or each other.
 *   - The library allocates no device memory. Scratch for the weight gradient is
 *     the caller's workspace `ws` of at least rmsnorm_bwd_workspace_bytes(T, D)
 *     bytes (16-byte aligned). The caller owns every buffer. (The host-buffer step
 *     creates two copy streams and a few events per device on its first call.)
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default stream);
 *     calls on one stream execute in order. A call that returns an error has
 *     enqueued nothing.
 *   - Validation runs on the host before any launch; invalid arguments are
 *     rejected with a status code. There is no fallback path of any kind.
 *   - Launch failures are reported as RMSN_ECUDA (from cudaGetLastError). Faults
 *     during execution surface on the stream as CUDA errors, as usual.
 *   - Each kernel bounds every wait on its asynchronous copies; if a wait ever
 *     exceeds its limit the kernel stops, records a flag readable with
 *     rmsnorm_device_error(), and returns.
 */
#ifndef RMSNORM_GB300_H_
#define RMSNORM_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t rmsn_bf16;               /* raw bf16 bit pattern                      */
typedef uint16_t rmsn_act16;              /* raw 16-bit activation, bf16 or fp16 by `dtype` */
typedef struct CUstream_st* rmsn_stream;  /* identical to cudaStream_t; NULL = default */

enum rmsn_status {
    RMSN_OK = 0,
    RMSN_EINVAL = -1,        /* null pointer, bad size, ld < D, negative/non-finite eps */
    RMSN_EALIGN = -2,        /* a pointer or row stride is not 16-byte aligned          */
    RMSN_EUNSUPPORTED = -3,  /* D outside [8, 16384] or not a multiple of 8             */
    RMSN_ECUDA = -4,         /* a CUDA runtime or driver call failed                    */
    RMSN_EWORKSPACE = -5     /* workspace missing or smaller than the query's answer    */
};

/* Activation storage formats of the *_ex entry points. */
enum rmsn_dtype {
    RMSN_DTYPE_BF16 = 0,     /* bfloat16 (what every entry point without _ex takes)     */
    RMSN_DTYPE_F16 = 1       /* IEEE binary16                                           */
};

/* Gate activation of the gated norm (*_ex entry points). */
enum rmsn_gate {
    RMSN_GATE_SILU = 0,      /* q(z) = z * sigmoid(z) (what rmsnorm_gated_fwd/bwd use)  */
    RMSN_GATE_SIGMOID = 1    /* q(z) = sigmoid(z)                                       */
};

/* Human-readable name of a status code (static string). */
const char* rmsnorm_status_string(int status);

/* Forward, plain or zero-centred ([Megatron] item 1; [Residual] Forward).
 *   x [T][ldx] in, w [D] in, y [T][ldy] out, rstd [T] out (fp32 inverse RMS). */
int rmsnorm_fwd(const rmsn_bf16* x, int64_t ldx, const float* w,
                rmsn_bf16* y, int64_t ldy, float* rstd,
                int64_t T, int64_t D, float eps, int zero_centered_gamma, rmsn_stream stream);

/* Bytes of workspace the backward entry points need for T rows of width D
 * (0 for T == 0; also 0 for an unsupported D). Not monotone in T: at some
 * widths the weight-gradient chunk is shortened so that chunks fill whole
 * rounds of the grid, and a larger T can then need fewer bytes than a smaller
 * one (D = 4096: T = 20000 needs more than T = 27360). To size one buffer for
 * every T up to a maximum, use rmsnorm_bwd_workspace_bytes_max. */
size_t rmsnorm_bwd_workspace_bytes(int64_t T, int64_t D);

/* The largest rmsnorm_bwd_workspace_bytes(T, D) over 0 <= T <= T_max: one
 * buffer of this many bytes serves every such T (0 for T_max <= 0 or an
 * unsupported D). Computed in closed form, in constant time for any T_max. */
size_t rmsnorm_bwd_workspace_bytes_max(int64_t T_max, int64_t D);

/* Backward, plain or zero-centred ([Megatron] item 2; [Residual] Backward).
 *   g [T][ldg] (dL/dy) in, x [T][ldx] in, w [D] in, rstd [T] in (the forward's),
 *   dx [T][lddx] out, dgamma [D] out (fp32), ws workspace.
 *   If dgamma is NULL, only pass 1 runs: the per-chunk partial sums are left in
 *   ws and rmsnorm_dgamma_reduce() finishes them later. */
int rmsnorm_bwd(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                const float* w, const float* rstd,
                rmsn_bf16* dx, int64_t lddx, float* dgamma,
                void* ws, size_t ws_bytes,
                int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream);

/* rmsnorm_residual forward ([Residual] Summary): the plain forward, plus a
 * bitwise copy of x into x_copy [T][ldxc]. It is not RMSNorm(x + residual). */
int rmsnorm_residual_fwd(const rmsn_bf16* x, int64_t ldx, const float* w,
                         rmsn_bf16* y, int64_t ldy, float* rstd,
                         rmsn_bf16* x_copy, int64_t ldxc,
                         int64_t T, int64_t D, float eps, int zero_centered_gamma,
                         rmsn_stream stream);

/* rmsnorm_residual backward ([Residual] Backward: dx gains d_residual).
 *   g_res [T][ldgr] is the gradient arriving at x_copy, added in fp32 before dx's
 *   single bf16 rounding; NULL means zero. Other arguments as rmsnorm_bwd. */
int rmsnorm_residual_bwd(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                         const float* w, const float* rstd,
                         const rmsn_bf16* g_res, int64_t ldgr,
                         rmsn_bf16* dx, int64_t lddx, float* dgamma,
                         void* ws, size_t ws_bytes,
                         int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream);

/* Gated forward, Qwen3-Next / vLLM convention ([ZC-norm], gated-norm conventions):
 *   y = bf16( ((x * r) * w_eff) * silu(z) ), weight multiply and gate in fp32,
 *   silu(z) = z * sigmoid(z), sigmoid evaluated in fp32 in a two-sided form
 *   from the PTX approximate instructions ex2 and rcp (relative error a few
 *   fp32 ulp plus about |z| * 2^-24, far inside one bf16 ulp).
 *   z [T][ldz] in (the gate). */
int rmsnorm_gated_fwd(const rmsn_bf16* x, int64_t ldx, const rmsn_bf16* z, int64_t ldz,
                      const float* w, rmsn_bf16* y, int64_t ldy, float* rstd,
                      int64_t T, int64_t D, float eps, int zero_centered_gamma,
                      rmsn_stream stream);

/* Gated forward in the HF/transformers convention, kept as a witness of the
 * convention divergence ([ZC-norm]: the two upstreams round the gated norm
 * differently; they agree bitwise with fp32 inputs). Forward only:
 *   n = bf16((x * r)),  t = bf16(bf16(w_eff) * n),  y = bf16(t * silu(z)).
 * The pages give no cast points, only that this convention's weight multiply is
 * not an fp32 one: these are the library's reading of them.
 * Arguments as rmsnorm_gated_fwd. */
int rmsnorm_gated_hf_fwd(const rmsn_bf16* x, int64_t ldx, const rmsn_bf16* z, int64_t ldz,
                         const float* w, rmsn_bf16* y, int64_t ldy, float* rstd,
                         int64_t T, int64_t D, float eps, int zero_centered_gamma,
                         rmsn_stream stream);

/* Gated backward: with q = silu(z) and u = (x r) w_eff,
 *   dx = plain backward with g*q in place of g;  dz = bf16( g u silu'(z) );
 *   dw_j = sum_t g q x r. dw NULL: as rmsnorm_bwd with dgamma NULL. */
int rmsnorm_gated_bwd(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                      const rmsn_bf16* z, int64_t ldz, const float* w, const float* rstd,
                      rmsn_bf16* dx, int64_t lddx, rmsn_bf16* dz, int64_t lddz, float* dw,
                      void* ws, size_t ws_bytes,
                      int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream);

/* Fused add + RMSNorm, the decoder-norm path of Qwen3-Next ([ZC-norm]: all
 * decoder norms but layer 0's input norm add the residual stream first and
 * normalise the fp32 sum). Forward, per element and row:
 *   h = x + res (one fp32 add);  res_out = bf16(h)  (the new residual stream);
 *   rstd, y as rmsnorm_fwd applied to the fp32 h (not to its bf16 rounding).
 *   x, res [T][ld*] in; y, res_out [T][ld*] out; rstd [T] out. */
int rmsnorm_fused_add_fwd(const rmsn_bf16* x, int64_t ldx, const rmsn_bf16* res, int64_t ldres,
                          const float* w, rmsn_bf16* y, int64_t ldy, float* rstd,
                          rmsn_bf16* res_out, int64_t ldro,
                          int64_t T, int64_t D, float eps, int zero_centered_gamma,
                          rmsn_stream stream);

/* Fused add + RMSNorm backward. h is recomputed from x and res exactly as in
 * the forward; with g = dL/dy and g_res = dL/d res_out (NULL = zero), the
 * gradient of h (and so of both x and res) is
 *   dh = bf16( rmsnorm backward at h  +  g_res ),   dgamma_j = sum_t g_tj h_tj r_t.
 * Workspace and dgamma == NULL as in rmsnorm_bwd. */
int rmsnorm_fused_add_bwd(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                          const rmsn_bf16* res, int64_t ldres, const float* w, const float* rstd,
                          const rmsn_bf16* g_res, int64_t ldgr,
                          rmsn_bf16* dh, int64_t lddh, float* dgamma,
                          void* ws, size_t ws_bytes,
                          int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream);

/* Backward with recomputation of the forward output (activation recompute):
 * exactly rmsnorm_residual_bwd (g_res NULL = the plain / zero-centred
 * backward) that also writes y [T][ldy] = bf16((x * rstd) * w_eff) from the
 * saved rstd — the same operations as the forward, so the same bits as the
 * forward's y — in the same pass over x, for one extra row write instead of a
 * second forward launch. */
int rmsnorm_bwd_recompute(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                          const float* w, const float* rstd,
                          const rmsn_bf16* g_res, int64_t ldgr,
                          rmsn_bf16* dx, int64_t lddx, float* dgamma,
                          rmsn_bf16* y, int64_t ldy,
                          void* ws, size_t ws_bytes,
                          int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream);

/* Gated backward with recomputation of the gated forward output y (same bits
 * as rmsnorm_gated_fwd's y); otherwise exactly rmsnorm_gated_bwd. */
int rmsnorm_gated_bwd_recompute(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                                const rmsn_bf16* z, int64_t ldz, const float* w, const float* rstd,
                                rmsn_bf16* dx, int64_t lddx, rmsn_bf16* dz, int64_t lddz, float* dw,
                                rmsn_bf16* y, int64_t ldy,
                                void* ws, size_t ws_bytes,
                                int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream);

/* ------------------------------------------------------------------------
 * Activation dtype and gate options ([ZC-norm]: the gated norm's activation
 * is configurable, silu by default with sigmoid allowed; the op contract's
 * tolerances cover fp16 activations beside bf16).
 *
 * Each *_ex entry point is the entry point of the same name without the
 * suffix, with two changes:
 *   - `dtype` (enum rmsn_dtype) names the storage format of EVERY activation
 *     argument (inputs and outputs alike): RMSN_DTYPE_BF16 gives exactly the
 *     unsuffixed call's results; with RMSN_DTYPE_F16 every activation is an
 *     IEEE binary16 bit pattern, widened exactly to fp32 on load, and every
 *     activation output is rounded from the same fp32 value to the nearest
 *     fp16 (ties to even; subnormals kept; overflow gives infinity). w, rstd
 *     and dgamma stay fp32, and the fp32 arithmetic, its reduction trees and
 *     the batch-invariance and determinism guarantees are unchanged.
 *   - the gated calls take `gate` (enum rmsn_gate). With RMSN_GATE_SIGMOID:
 *       y  = round( ((x * r) * w_eff) * sigmoid(z) ),
 *       backward: dx as rmsnorm_bwd with g * sigmoid(z) in place of g;
 *       dz = round( g * u * sigmoid(z) * sigmoid(-z) ),  u = (x * r) * w_eff;
 *       dw_j = sum_t g sigmoid(z) x r.
 * An unknown dtype or gate is RMSN_EINVAL. Alignment, ownership, workspace
 * and error behaviour as the unsuffixed call.
 * ------------------------------------------------------------------------ */
int rmsnorm_fwd_ex(const rmsn_act16* x, int64_t ldx, const float* w,
                   rmsn_act16* y, int64_t ldy, float* rstd,
                   int64_t T, int64_t D, float eps, int zero_centered_gamma,
                   int dtype, rmsn_stream stream);

int rmsnorm_bwd_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                   const float* w, const float* rstd,
                   rmsn_act16* dx, int64_t lddx, float* dgamma,
                   void* ws, size_t ws_bytes,
                   int64_t T, int64_t D, int zero_centered_gamma, int dtype, rmsn_stream stream);

int rmsnorm_residual_fwd_ex(const rmsn_act16* x, int64_t ldx, const float* w,
                            rmsn_act16* y, int64_t ldy, float* rstd,
                            rmsn_act16* x_copy, int64_t ldxc,
                            int64_t T, int64_t D, float eps, int zero_centered_gamma,
                            int dtype, rmsn_stream stream);

int rmsnorm_residual_bwd_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                            const float* w, const float* rstd,
                            const rmsn_act16* g_res, int64_t ldgr,
                            rmsn_act16* dx, int64_t lddx, float* dgamma,
                            void* ws, size_t ws_bytes,
                            int64_t T, int64_t D, int zero_centered_gamma, int dtype,
                            rmsn_stream stream);

int rmsnorm_gated_fwd_ex(const rmsn_act16* x, int64_t ldx, const rmsn_act16* z, int64_t ldz,
                         const float* w, rmsn_act16* y, int64_t ldy, float* rstd,
                         int64_t T, int64_t D, float eps, int zero_centered_gamma,
                         int gate, int dtype, rmsn_stream stream);

int rmsnorm_gated_bwd_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                         const rmsn_act16* z, int64_t ldz, const float* w, const float* rstd,
                         rmsn_act16* dx, int64_t lddx, rmsn_act16* dz, int64_t lddz, float* dw,
                         void* ws, size_t ws_bytes,
                         int64_t T, int64_t D, int zero_centered_gamma, int gate, int dtype,
                         rmsn_stream stream);

int rmsnorm_fused_add_fwd_ex(const rmsn_act16* x, int64_t ldx, const rmsn_act16* res, int64_t ldres,
                             const float* w, rmsn_act16* y, int64_t ldy, float* rstd,
                             rmsn_act16* res_out, int64_t ldro,
                             int64_t T, int64_t D, float eps, int zero_centered_gamma,
                             int dtype, rmsn_stream stream);

int rmsnorm_fused_add_bwd_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                             const rmsn_act16* res, int64_t ldres, const float* w, const float* rstd,
                             const rmsn_act16* g_res, int64_t ldgr,
                             rmsn_act16* dh, int64_t lddh, float* dgamma,
                             void* ws, size_t ws_bytes,
                             int64_t T, int64_t D, int zero_centered_gamma, int dtype,
                             rmsn_stream stream);

/* The backward with recomputation of the forward output, with the activation
 * dtype (and, for the gated call, the gate) as in the *_ex calls above; y is
 * written in the activation format, bit for bit the *_ex forward's y. */
int rmsnorm_bwd_recompute_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                             const float* w, const float* rstd,
                             const rmsn_act16* g_res, int64_t ldgr,
                             rmsn_act16* dx, int64_t lddx, float* dgamma,
                             rmsn_act16* y, int64_t ldy,
                             void* ws, size_t ws_bytes,
                             int64_t T, int64_t D, int zero_centered_gamma, int dtype, rmsn_stream stream);

int rmsnorm_gated_bwd_recompute_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                                   const rmsn_act16* z, int64_t ldz, const float* w, const float* rstd,
                                   rmsn_act16* dx, int64_t lddx, rmsn_act16* dz, int64_t lddz, float* dw,
                                   rmsn_act16* y, int64_t ldy,
                                   void* ws, size_t ws_bytes,
                                   int64_t T, int64_t D, int zero_centered_gamma, int gate, int dtype,
                                   rmsn_stream stream);

/* Weight-gradient pass 2 on its own: sums the per-chunk partials that a backward
 * call with a NULL dgamma/dw left in ws (same T, D and workspace), in the fixed
 * order, into dgamma [D]. ws must be unchanged since that call. */
int rmsnorm_dgamma_reduce(const void* ws, size_t ws_bytes, int64_t T, int64_t D,
                          float* dgamma, rmsn_stream stream);

/* Backward without a caller workspace (no counterpart in the pages: this is a
 * library convenience). For callers that cannot allocate device memory — code
 * that may only use the tensors it is handed, or a runtime that must not grow
 * its device footprint after start-up — the weight-gradient scratch lives in a
 * fixed array inside the library's device image: RMSN_NOALLOC_SCRATCH_BYTES on
 * every GPU that loads the library, held until the process exits. The call
 * allocates nothing; inputs and outputs are the caller's, as in rmsnorm_bwd
 * (same arguments minus the workspace; dgamma must not be NULL).
 *   - Arguments are checked as rmsnorm_bwd checks them, and fail with its
 *     statuses; then a NULL dgamma is RMSN_EINVAL, and a problem needing more
 *     scratch than the array holds, i.e. with
 *     rmsnorm_bwd_workspace_bytes(T, D) > RMSN_NOALLOC_SCRATCH_BYTES, is
 *     rejected with RMSN_EWORKSPACE. Every T up to T_max fits exactly when
 *     rmsnorm_bwd_workspace_bytes_max(T_max, D) <= RMSN_NOALLOC_SCRATCH_BYTES:
 *     every T <= 32768 at D <= 6896 and at 7176 <= D <= 8192 (D = 8192,
 *     T = 32768 fills the array exactly), every T <= 29250 at
 *     6904 <= D <= 7168 (shortened chunks), every T <= 16384 at D = 16384.
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *     A cudaDeviceReset destroys the context and can move the array; the
 *     next call in the new context looks the address up again.
 *   - Every call shares the one array: calls whose work overlaps on the GPU
 *     (other streams or threads, unordered) race and corrupt dgamma. Calls on
 *     one stream are safe. Leftover contents are never read.
 *   - Results are bitwise those of rmsnorm_bwd on the same inputs. */
#define RMSN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int rmsnorm_bwd_noalloc(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                        const float* w, const float* rstd,
                        rmsn_bf16* dx, int64_t lddx, float* dgamma,
                        int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream);

/* rmsnorm_residual forward + backward on HOST buffers (no counterpart in the
 * pages: a library convenience around [Residual]'s forward and backward). One
 * call copies the inputs in, runs rmsnorm_residual_fwd_ex and
 * rmsnorm_residual_bwd_ex, and copies every output back, with the copies
 * overlapped against the kernels: the rows go in slabs, and while slab k's
 * kernels run, slab k+1's inputs come in and slab k-1's outputs go out.
 *   Host buffers, dense row-major (row stride D), in the activation format
 *   `dtype` (RMSN_DTYPE_BF16 / RMSN_DTYPE_F16) unless marked fp32:
 *     in:  x [T][D], g [T][D] (dL/dy), g_res [T][D] (dL/dx_copy; NULL = zero),
 *          w [D] fp32
 *     out: y [T][D], x_copy [T][D], rstd [T] fp32, dx [T][D], dgamma [D] fp32
 *   Results are bitwise those of rmsnorm_residual_fwd_ex followed by
 *   rmsnorm_residual_bwd_ex on device copies of the same inputs.
 *   - The host buffers are read and written asynchronously: the caller must
 *     not touch them until the work on `stream` has completed. Page-locked
 *     (pinned) host memory gives the overlap; pageable memory is accepted but
 *     the copies then run in step with the calling thread.
 *   - work: a DEVICE buffer, 256-byte aligned, of at least
 *     rmsnorm_residual_step_host_work_bytes(T, D, slab_rows) bytes, owned by the
 *     caller. It holds three slab slots (six [slab][D] activation buffers and
 *     a [slab] fp32 buffer each), w, dgamma and the weight-gradient partials of
 *     all T rows. Too small or NULL: RMSN_EWORKSPACE; misaligned: RMSN_EALIGN.
 *     Calls that overlap on the GPU must not share one work buffer.
 *   - slab_rows: rows per slab, rounded up to a multiple of the weight-gradient
 *     chunk of the whole problem (for D > 256: 32 rows, or fewer at some T for
 *     2048 < D <= 7168; for D <= 256: 128 rows or more) and capped at T; 0
 *     takes the default, 4096.
 *   - The kernels run on `stream`; the copies run on two copy streams per
 *     device that the library creates on the first call made with that device
 *     current (make that first call outside any stream capture) and keeps
 *     until the process exits. The call starts after the earlier work on
 *     `stream`, and `stream` waits for the last copy, so it is ordered like any
 *     other work on `stream`. Calls from several host threads are serialised
 *     while they enqueue.
 *   - Every argument is validated before anything is enqueued. A CUDA failure
 *     while enqueueing (RMSN_ECUDA) may leave part of the step enqueued. */
size_t rmsnorm_residual_step_host_work_bytes(int64_t T, int64_t D, int64_t slab_rows);
int rmsnorm_residual_step_host(const rmsn_act16* x, const rmsn_act16* g, const rmsn_act16* g_res,
                               const float* w,
                               rmsn_act16* y, rmsn_act16* x_copy, float* rstd,
                               rmsn_act16* dx, float* dgamma,
                               int64_t T, int64_t D, float eps, int zero_centered_gamma, int dtype,
                               int64_t slab_rows, void* work, size_t work_bytes, rmsn_stream stream);

/* Reads the device-side error flags of the current device (OR of all kernels'
 * flags since the last clear) into *flags; clears them if `clear` is non-zero.
 * Synchronises with the device. 0 means no kernel ever gave up on a wait;
 * RMSN_DEVICE_ERR_WAIT_TIMEOUT is set when a wait ran out of time. */
#define RMSN_DEVICE_ERR_WAIT_TIMEOUT 1u
int rmsnorm_device_error(unsigned int* flags, int clear);

/* Self-test of the error path above (no counterpart in the pages). Launches one
 * thread on `stream` that waits, with the kernels' own bounded wait and the limit
 * `limit_ns` (1 ns .. 1 s), on a fresh mbarrier that nothing ever completes: the
 * wait runs out, the thread raises RMSN_DEVICE_ERR_WAIT_TIMEOUT, and the kernel
 * returns normally, leaving the context usable. If `waited_ns` (a DEVICE pointer
 * to one 8-byte-aligned uint64, or NULL) is given, the time the wait took is
 * written there. A limit of 0 or above 1 s is RMSN_EINVAL. */
int rmsnorm_selftest_wait_timeout(unsigned long long limit_ns, unsigned long long* waited_ns,
                                  rmsn_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_GB300_H_ */
