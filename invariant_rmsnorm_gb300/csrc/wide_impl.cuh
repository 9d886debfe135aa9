// Wide-row kernels (D > 256): a CTA reduces R whole rows per iteration.
// Kernel and launcher templates, included by the translation units that
// instantiate them (wide.cu: bf16 activations; wide_f16.cu: fp16).
//
// Design (GB300, HBM-bound):
//   * Persistent grid: at most (SM count x resident CTAs) CTAs, each walking a
//     fixed sequence of rows (forward) or of whole row chunks (backward).
//   * Warp-specialised pipeline. The last warp of the CTA is a producer: one
//     lane keeps S stages of R rows in flight with 1-D bulk TMA copies
//     (cp.async.bulk global->shared, completion counted on a per-stage "full"
//     mbarrier). The consumer warps read a stage into registers and release it
//     on its "empty" mbarrier (one arrive per warp) before they reduce, so the
//     producer refills it while the arithmetic runs and no consumer ever
//     waits for a copy to be issued.
//   * Consumer thread t owns VPT 16-byte vectors of each row at slots
//     v = k*NT + t (coalesced, conflict-free shared reads).
//   * Fixed reduction tree (a function of D and, in the backward, of the
//     variant only): per-thread ascending sum over its slots and the 8
//     elements of each vector, an xor-butterfly over the warp (offsets 16..1),
//     then the per-warp totals added in warp order. The R rows of an iteration
//     share one named barrier but each keeps its own tree, so a row's bits
//     depend on nothing but the row, D and the variant: not on T, its
//     position, the other rows, the grid or the GPU.
//   * fp32 arithmetic with every multiply and add rounded separately (no FMA
//     contraction; in some kernels the products of neighbouring elements go
//     through the packed mul.rn.f32x2, with the same bits), rsqrtf for the
//     inverse RMS, round-to-nearest-even bf16 (or fp16) outputs written with
//     128-bit streaming stores.
//   * Backward weight gradient: a CTA owns whole chunks of kWideChunkRows rows,
//     accumulates g*x*r per column in ascending row order in registers and
//     writes one fp32 partial row per chunk; no atomics anywhere.
//   * Every mbarrier wait is bounded; a consumer that gives up votes through the
//     reduction barrier, the CTA stops, the device error flag is raised, and no
//     thread leaves while a copy it issued can still land.
//
// Sources: Megatron-LM pull request 6859 "Fix the batch-invariant RMSNorm
// forward and its input gradient" (What does this PR do, items 1-2);
// RL-Kernel pull request 414 "[DSv4][P1-5] rmsnorm_residual" (Implementation:
// rsqrt, (x*r)*gamma, ascending fp32 reductions, separate rounding, no atomics;
// Summary: the residual variant returns a copy of x); RL-Kernel pull request
// 467 "...zero-centred RMSNorm references and CUDA kernel" (+1 in fp32, gated
// norm with the weight multiply in fp32).
#pragma once

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

// Launch shapes, chosen by measurement on GB300 (T=32768, D=4096): the
// forward gets a 96 KB ring budget and as many CTAs per SM as fit (up to 3;
// 2 at D=4096); the backward 2 CTAs of 64 KB rings (per-width exceptions at
// bwd_min_blocks below).
#ifndef RMSN_WIDE_FWD_SMEM
#define RMSN_WIDE_FWD_SMEM (96 * 1024)   // target ring bytes per CTA (forward)
#endif
#ifndef RMSN_WIDE_FWD_CTAS_PER_SM
#define RMSN_WIDE_FWD_CTAS_PER_SM 3
#endif
#ifndef RMSN_WIDE_BWD_SMEM
#define RMSN_WIDE_BWD_SMEM (64 * 1024)   // target ring bytes per CTA (backward)
#endif
#ifndef RMSN_WIDE_BWD_CTAS_PER_SM
#define RMSN_WIDE_BWD_CTAS_PER_SM 2
#endif
#ifndef RMSN_WIDE_BWD_SMEM_512
#define RMSN_WIDE_BWD_SMEM_512 (96 * 1024)  // ring budget of the 512-thread backward (one CTA per SM)
#endif
#ifndef RMSN_MAX_STAGES
#define RMSN_MAX_STAGES 16
#endif
#ifndef RMSN_FWD_ROWS
#define RMSN_FWD_ROWS 4   // rows per forward iteration
#endif
#ifndef RMSN_BWD_ROWS
#define RMSN_BWD_ROWS 2   // rows per backward iteration (divides the chunk)
#endif
#ifndef RMSN_BWD_LEAN
#define RMSN_BWD_LEAN 1   // backward recomputes products after the reduction (fewer registers)
#endif
#ifndef RMSN_BWD_MINB
#define RMSN_BWD_MINB 2   // backward CTAs that must fit on one SM (register budget), VPT 2
#endif
#ifndef RMSN_BWD_MINB_V1
#define RMSN_BWD_MINB_V1 3  // the same for VPT 1 (3 CTAs of 72 registers)
#endif
#ifndef RMSN_BWD_SGS
#define RMSN_BWD_SGS 1  // gated (silu) backward at one or two vectors a thread: sigmoid(z) parked in shared memory
#endif
#ifndef RMSN_BWD_HOLD_WIDE
#define RMSN_BWD_HOLD_WIDE 1  // VPT 4 at 512 threads: re-read staged operands after the reduction
#endif
#ifndef RMSN_BWD_WL1_WIDE
#define RMSN_BWD_WL1_WIDE 1  // VPT 4 at 512 threads: weights from L1 where used
#endif
#ifndef RMSN_WIDE_BWD_CTAS_PER_SM_V1
#define RMSN_WIDE_BWD_CTAS_PER_SM_V1 3
#endif


namespace rmsn {

// Rows per iteration: 4 (forward) or 2 (backward at VPT 1) for narrow wide
// rows; at VPT 4 the forward takes 2 rows when it streams one operand
// (plain, residual; 32768 x 16384: 498 -> 338 us) and 1 otherwise, since a
// second row of two operands overflows registers (a 9-warp CTA puts 3 warps
// on one scheduler: <= 168 registers per thread) or shared memory.
#ifndef RMSN_FWD_ROWS_V4
#define RMSN_FWD_ROWS_V4 2  // VPT 4 rows on 512 threads (D > 8192), one streamed operand: 2 rows per iteration
#endif
#ifndef RMSN_FWD_ROWS_V4_256
#define RMSN_FWD_ROWS_V4_256 2  // VPT 4 rows on up to 256 threads, one streamed operand
#endif
template <int VPT, int MAXT, int MODE> __host__ __device__ constexpr int fwd_rows() {
    return VPT < 4 ? RMSN_FWD_ROWS
                   : (fwd_inputs(MODE) > 1 ? 1 : (MAXT > 256 ? RMSN_FWD_ROWS_V4 : RMSN_FWD_ROWS_V4_256));
}
// Backward CTAs per SM that the register budget must allow: 3 at VPT 1 (72
// registers) for the modes that fit there without spilling (not the gated or
// the fused-add backward), 2 at VPT 1 otherwise and at VPT 2 (96), 2 for VPT 4
// rows of at most 224 threads (128 registers: 4096 < D <= 7168), 1 beyond.
// The cap on resident CTAs is 3 at VPT 1 in every mode: the gated and
// fused-add kernels reach it on up to 160 threads at 96 registers (gated,
// 32768 rows, backward with pass 2: D=512 80.6 -> 62.0 us, 1024 86.7 -> 72.1).
template <int VPT, int MAXT, int MODE> __host__ __device__ constexpr int bwd_min_blocks() {
    return MAXT == 128 ? 4 : MAXT == 224 ? 2
           : (MAXT > 256 || VPT > 2) ? 1
           : (VPT == 1 && !is_gated(MODE) && base_mode(MODE) != kFusedAdd) ? RMSN_BWD_MINB_V1
                                                                           : RMSN_BWD_MINB;
}
template <int VPT, int MAXT, int MODE> __host__ __device__ constexpr int bwd_ctas_per_sm() {
    return MAXT == 128 ? 4 : MAXT == 224 ? 2 : VPT == 1 ? RMSN_WIDE_BWD_CTAS_PER_SM_V1 : RMSN_WIDE_BWD_CTAS_PER_SM;
}
// Rows per backward iteration: RMSN_BWD_ROWS at one vector a thread; two in
// the plain mode's two-vector kernel on 512 threads (7168 < D <= 8192), which
// fits them in its 96 registers without spilling (131072 x 8192, backward with
// pass 2: 1063 -> 996 us); one elsewhere (a second row of three or four
// operands spills there, and the 256-thread kernels measured mixed). An
// iteration never straddles a chunk, so the rows per iteration divide the
// 32-row chunk; the stepping kernels, whose shortened chunk can be odd, run
// at one row (the dispatch gives them no other shape).
template <int VPT, int MAXT, int MODE, bool PAIR = false> __host__ __device__ constexpr int bwd_rows() {
    return (VPT == 1 && MAXT <= 256)                                       ? RMSN_BWD_ROWS
           : (VPT == 2 && MAXT > 256 && !PAIR && base_mode(MODE) == kPlain) ? 2
                                                                            : 1;
}

constexpr int kConsumerBarrier = 1;  // named barrier id of the consumer warps

namespace {

// Device error word of the including translation unit.
__device__ unsigned int g_wide_error;

cudaError_t read_wide_error_word(unsigned* flags, bool clear) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_wide_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *flags |= v;
    if (clear && v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_wide_error, &zero, sizeof(zero));
    }
    return e;
}

// Load this thread's effective weights: w, or w + 1 in fp32 (zero-centred gamma).
template <int VPT>
__device__ __forceinline__ void load_weights(const float* w, int zc, int NV, int nt, int tid,
                                             float (&we)[VPT][8]) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = k * nt + tid;
        if (v < NV) {
            const float4 lo = __ldg(reinterpret_cast<const float4*>(w) + 2 * v);
            const float4 hi = __ldg(reinterpret_cast<const float4*>(w) + 2 * v + 1);
            we[k][0] = lo.x; we[k][1] = lo.y; we[k][2] = lo.z; we[k][3] = lo.w;
            we[k][4] = hi.x; we[k][5] = hi.y; we[k][6] = hi.z; we[k][7] = hi.w;
            if (zc) {
#pragma unroll
                for (int e = 0; e < 8; ++e) we[k][e] = fadd(we[k][e], 1.0f);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) we[k][e] = 0.0f;
        }
    }
}

// Effective weights of vector v (8 values), read through the non-coherent
// cache path where they are used (volatile: not hoisted into registers).
__device__ __forceinline__ void weights8(const float* w, int zc, int v, float (&o)[8]) {
    const float* p = w + 8 * v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(o[0]), "=f"(o[1]), "=f"(o[2]), "=f"(o[3]) : "l"(p));
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(o[4]), "=f"(o[5]), "=f"(o[6]), "=f"(o[7]) : "l"(p + 4));
    if (zc) {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = fadd(o[e], 1.0f);
    }
}

// The values a row is normalised over: x, or the fp32 sum x + res (fused add).
template <int MODE>
__device__ __forceinline__ void norm_input(const uint4 xv, const uint4 sv, float (&f)[8]) {
    unpack_act<is_f16(MODE)>(xv, f);
    if (is_fused(MODE)) {
        float rv[8];
        unpack_act<is_f16(MODE)>(sv, rv);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = fadd(f[e], rv[e]);
    }
}

// First half of the block-wide fixed tree, for R rows at once: butterfly
// within each consumer warp (the R chains interleave), lane 0 parks each warp
// total in red[r*32 + warp]. The consumers' named barrier doubles as the error
// vote: returns the AND of every consumer's `ok`.
template <int R>
__device__ __forceinline__ int block_partial(float (&v)[R], float* red, int lane, int warp, int nt, bool ok) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = fadd(v[r], __shfl_xor_sync(0xffffffffu, v[r], o));
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) red[r * 32 + warp] = v[r];
    }
    return named_bar_and(kConsumerBarrier, nt, ok ? 1 : 0);
}

// Second half: the warp totals added in warp order (same bits in every thread).
// All loads are issued before the dependent adds.
template <int NWMAX>
__device__ __forceinline__ float block_total(const float* red, int nw) {
    float w[NWMAX];
#pragma unroll
    for (int i = 0; i < NWMAX; ++i) w[i] = (i < nw) ? red[i] : 0.0f;
    float t = w[0];
#pragma unroll
    for (int i = 1; i < NWMAX; ++i)
        if (i < nw) t = fadd(t, w[i]);
    return t;
}

// Producer loop (one lane): fill stage i % S with iteration i once the
// consumers have released the iteration S earlier. `issue(i)` posts the copies.
// If the consumers stop releasing (a consumer gave up), wait (bounded) for the
// copies still in flight, raise the flag and stop.
// Stage index and phase parity advance together (no divisions on the hot path).
template <typename Issue>
__device__ __forceinline__ void produce(uint64_t* full, uint64_t* empty, int S, int n_it, Issue&& issue) {
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < n_it; ++i) {
        if (i >= S && !mbar_wait(&empty[s], ph ^ 1u)) {
            for (int j = i - S; j < i; ++j) (void)mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1));
            atomicOr(&g_wide_error, kErrWaitTimeout);
            return;
        }
        fence_proxy_async_smem();
        issue(i, s);
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// A consumer gave up at iteration i: one thread waits (bounded) for the stages
// the producer may still be filling, then raises the flag.
__device__ void consumer_abort(uint64_t* full, int S, int i, int n_it) {
    for (int j = i; j < n_it && j < i + S; ++j) (void)mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1));
    atomicOr(&g_wide_error, kErrWaitTimeout);
}

// ---------------------------------------------------------------------------
// Forward: plain / zero-centred, residual (adds the copy), gated (reads z).
// Stage layout [row][x | z][D]. blockDim = NT consumers + 32 (producer warp).
// ---------------------------------------------------------------------------
template <int VPT, int MODE, int MAXT>
__global__ void __launch_bounds__(MAXT + 32) wide_fwd_kernel(const FwdArgs a, const int S) {
    constexpr int M = base_mode(MODE);
    constexpr bool F16 = is_f16(MODE);
    constexpr bool SIG = is_sigmoid_gate(MODE);
    static_assert(!(M == kGatedHF && F16), "the HF-convention witness is a bf16 forward");
    // Element pairs through the packed fp32 instructions (same bits as the
    // scalar loops) in the one-vector kernel outside the gated mode (D <= 2048;
    // 131072 x 2048 plain 175.7 -> 171.1 us, residual 272.6 -> 271.0, fused
    // add 376.4 -> 374.6; gated measured 303.1 -> 309.4). With two or four
    // vectors a thread they measured slower (D = 4096: 347 -> 362 us).
    constexpr bool FX2P = RMSN_F32X2 && VPT == 1 && M != kGated;  // the squares of the sum of squares
    constexpr bool FX2O = FX2P;                                   // the output products
    constexpr int NIN = fwd_inputs(MODE);
    constexpr int R = fwd_rows<VPT, MAXT, MODE>();
    constexpr int NWMAX = MAXT / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    const int D = a.D;
    const int NV = D >> 3;
    const int nt = blockDim.x - 32;  // consumer threads
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int64_t T = a.T;
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const uint32_t row_bytes = static_cast<uint32_t>(D) * 2u;
    const uint32_t stage_bytes = R * NIN * row_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t* empty = full + S;
    float* red = reinterpret_cast<float*>(empty + S);  // [2][R][32]

    const int n_my = (cta < T) ? static_cast<int>((T - 1 - cta) / G + 1) : 0;  // rows cta, cta+G, ...
    const int n_it = (n_my + R - 1) / R;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nw);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();  // first global memory access below

    if (warp == nw) {  // producer warp
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            produce(full, empty, S, n_it, [&](int i, int s) {
                unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
                const int nvalid = min(n_my - i * R, R);
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nvalid) * NIN * row_bytes);
                for (int r = 0; r < nvalid; ++r) {
                    const int64_t row = cta + static_cast<int64_t>(i * R + r) * G;
                    unsigned char* dst = st + static_cast<size_t>(r) * NIN * row_bytes;
                    bulk_g2s(dst, a.x + row * a.ldx, row_bytes, &full[s], pol);
                    if (is_gated(MODE)) bulk_g2s(dst + row_bytes, a.z + row * a.ldz, row_bytes, &full[s], pol);
                    if (is_fused(MODE)) bulk_g2s(dst + row_bytes, a.res + row * a.ldres, row_bytes, &full[s], pol);
                }
            });
        }
        return;
    }

    float we[VPT][8];
    load_weights<VPT>(a.w, a.zc, NV, nt, tid, we);

    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < n_it; ++i) {
        const bool ok = mbar_wait(&full[s], ph);
        const unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
        const int nvalid = min(n_my - i * R, R);

        uint4 xv[R][VPT];
        uint4 zv[R][VPT];  // gated: z; fused add: res
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < nvalid) {
                const unsigned char* src = st + static_cast<size_t>(r) * NIN * row_bytes;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int v = j * nt + tid;
                    if (v < NV) {
                        xv[r][j] = ld_shared_v4(src + 16 * v);
                        if (NIN == 2) zv[r][j] = ld_shared_v4(src + row_bytes + 16 * v);
                    }
                }
            }
        }
        // The stage is in registers: hand it back to the producer.
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }

        float ss[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            ss[r] = 0.0f;
            if (r < nvalid) {
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (j * nt + tid < NV) {
                        float f[8];
                        norm_input<MODE>(xv[r][j], zv[r][j], f);
                        if constexpr (FX2P) {
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {  // squares packed, the sum in element order
                                const float2 q2 = fmul2(pair(f, e), pair(f, e));
                                ss[r] = fadd(fadd(ss[r], q2.x), q2.y);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) ss[r] = fadd(ss[r], fmul(f[e], f[e]));
                        }
                    }
                }
            }
        }
        float* rb = red + (i & 1) * (R * 32);
        if (!block_partial<R>(ss, rb, lane, warp, nt, ok)) {
            if (tid == 0) consumer_abort(full, S, i, n_it);
            return;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < nvalid) {
                const float tot = block_total<NWMAX>(rb + r * 32, nw);
                const float rr = rsqrtf(fadd(div_by_d(tot, D, a.inv_d_pow2), a.eps));
                const int64_t row = cta + static_cast<int64_t>(i * R + r) * G;
                if (tid == 0) a.rstd[row] = rr;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int v = j * nt + tid;
                    if (v < NV) {
                        float f[8], o[8];
                        norm_input<MODE>(xv[r][j], zv[r][j], f);
                        if (M == kGated) {
                            float zf[8];
                            unpack_act<F16>(zv[r][j], zf);
                            if constexpr (FX2O) {
                                float q[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) q[e] = gate_value<SIG>(zf[e]);
#pragma unroll
                                for (int e = 0; e < 8; e += 2) {
                                    const float2 o2 = fmul2(fmul2(fmul2(pair(f, e), both(rr)), pair(we[j], e)), pair(q, e));
                                    o[e] = o2.x;
                                    o[e + 1] = o2.y;
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float q = gate_value<SIG>(zf[e]);
                                    o[e] = fmul(fmul(fmul(f[e], rr), we[j][e]), q);
                                }
                            }
                        } else if (M == kGatedHF) {
                            // HF convention: normalised value and weight multiply in bf16.
                            float zf[8];
                            unpack8(zv[r][j], zf);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float n = round_bf16f(fmul(f[e], rr));
                                const float t = round_bf16f(fmul(round_bf16f(we[j][e]), n));
                                o[e] = fmul(t, fmul(zf[e], sigmoidf_rn(zf[e])));
                            }
                        } else if constexpr (FX2O) {
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const float2 o2 = fmul2(fmul2(pair(f, e), both(rr)), pair(we[j], e));
                                o[e] = o2.x;
                                o[e + 1] = o2.y;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) o[e] = fmul(fmul(f[e], rr), we[j][e]);
                        }
                        st_global_cs(a.y + row * a.ldy + 8 * v, pack_act<F16>(o));
                        if (M == kResidual) st_global_cs(a.xc + row * a.ldxc + 8 * v, xv[r][j]);
                        if (is_fused(MODE)) st_global_cs(a.xc + row * a.ldxc + 8 * v, pack_act<F16>(f));  // x + res
                    }
                }
            }
        }
    }
    pdl_release();
}

// ---------------------------------------------------------------------------
// Backward pass 1: dx (and dz), plus one weight-gradient partial per chunk.
// Each iteration handles R consecutive rows of one chunk (R divides the chunk
// size, so an iteration never straddles two chunks). Stage layout
// [row][g | x | g_res or z][D]; each row's rstd arrives in the same stage
// through a 4-byte cp.async, and one no-increment arrive after them makes the
// stage's full barrier (expected count 2) wait for those copies too.
// The products needed after the row reduction (g*w_eff, x, g*x; gated: with
// g*silu(z) for g) are recomputed after it from the packed row, which stays in
// registers (RMSN_BWD_LEAN, the default: the same bits for fewer registers);
// with RMSN_BWD_LEAN = 0 they are computed once before it and kept.
// ---------------------------------------------------------------------------
template <int VPT, int MODE, int MAXT, bool VC = false, bool PAIR = false>
__global__ void __launch_bounds__(MAXT + 32, bwd_min_blocks<VPT, MAXT, MODE>())
wide_bwd_kernel(const BwdArgs a, const int S) {
    constexpr int M = base_mode(MODE);
    constexpr bool F16 = is_f16(MODE);
    constexpr bool SIG = is_sigmoid_gate(MODE);
    constexpr int NIN = bwd_inputs(MODE);
    constexpr int R = bwd_rows<VPT, MAXT, MODE, PAIR>();
    constexpr int NWMAX = MAXT / 32;
    constexpr bool RY = is_recompute(MODE);  // also write y (a.y is then not null)
    // Rows per weight-gradient chunk: kWideChunkRows, or with VC the chunk the
    // host chose for T (a.chunk, which R divides); VC kernels step through
    // their rows without dividing by it.
    constexpr int C0 = kWideChunkRows;
    static_assert(C0 % R == 0, "rows per iteration must divide the chunk");
    const int C = VC ? a.chunk : C0;
    // Register diet of the widest rows (VPT 4 on 512 threads, D > 8192, where
    // the launch allows about 96 registers): HOLD re-reads the staged operands
    // after the row reduction instead of keeping them packed in registers (the
    // stage is released at the end of the iteration); WL1 reads the weights
    // from L1 where they are used instead of keeping them in registers.
    // Measured at D=16384: 783 -> 667 us per 32768 rows; at 256 threads
    // (D <= 8192) both cost more than they save.
    constexpr bool HOLD = VPT == 4 && MAXT > 256 && RMSN_BWD_HOLD_WIDE;
    // SGS (silu gate, one or two vectors a thread): sigmoid(z), computed once
    // before the row reduction, is parked in this thread's own shared-memory
    // slots and read back after it, so the gate's exponential and reciprocal
    // run once per element instead of twice (q = z sigmoid(z) again has the
    // same bits; q' = sigmoid(z) + q (1 - sigmoid(z)), accurate to a few fp32
    // ulps of its terms). 32768 rows, backward with pass 2: D=2048 139 -> 125
    // us, 4096 257 -> 232, 7168 529 -> 479, 8192 552 -> 488. Parking q and q'
    // for both gates instead needed more registers and gained less.
    constexpr bool SGS = M == kGated && !SIG && VPT <= 2 && RMSN_BWD_LEAN && RMSN_BWD_SGS;
    constexpr bool WL1 = VPT == 4 && MAXT > 256 && RMSN_BWD_WL1_WIDE;
    // Element pairs through the packed fp32 instructions (same bits as the
    // scalar loops), where they measured faster: every site of the two-vector
    // kernels on 128 and on 512 threads (131072 x 2048: 282 -> 259 us;
    // 131072 x 8192: 1101 -> 1060 us) and of the one-vector kernel in the
    // gated and fused-add modes (131072 x 2048: 605 -> 585 us, 407 -> 402 us),
    // and the outputs after the reduction in the 256-thread two-vector kernel
    // (D = 4096 plain: 132.7 -> 129.9 us; residual equal). Pairs elsewhere in
    // that kernel, in the one-vector residual backward (336 -> 341 us) and in
    // the four-vector kernels measured slower.
    constexpr bool V1X2 = VPT == 1 && (M == kGated || M == kFusedAdd);
    constexpr bool X2 = ((VPT == 2 && (MAXT == 128 || MAXT > 256)) || V1X2) && RMSN_F32X2;
    constexpr bool X2P1 = X2, X2RC = X2;                      // before the reduction; its recompute
    constexpr bool X2OUT = (VPT == 2 || V1X2) && RMSN_F32X2;  // dx, the weight-gradient term, dz and y
    extern __shared__ __align__(128) unsigned char smem[];
    const int D = a.D;
    // PAIR (rows of more than 1024 vectors): the two CTAs of a cluster split
    // every row's columns, rank 0 the first ceil(NV/2) 16-byte vectors and rank
    // 1 the rest. The pair runs the cluster's chunks; each CTA reduces its half
    // of the row sum with the tree below, and both add the two halves in rank
    // order (the same bits in both).
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    const int NVh = ((D >> 3) + 1) >> 1;
    const int NV = PAIR ? (rank ? (D >> 3) - NVh : NVh) : (D >> 3);  // this CTA's vectors
    const int64_t cb = PAIR ? static_cast<int64_t>(rank) * NVh * 8 : 0;  // its first column
    const int nt = blockDim.x - 32;  // consumer threads
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int64_t T = a.T;
    const int64_t G = PAIR ? static_cast<int64_t>(cluster_count_x()) : static_cast<int64_t>(gridDim.x);
    const int64_t cta = PAIR ? static_cast<int64_t>(cluster_id_x()) : static_cast<int64_t>(blockIdx.x);
    const int64_t nchunks = (T + C - 1) / C;
    // This CTA's bytes of an operand row.
    const uint32_t row_bytes = PAIR ? static_cast<uint32_t>(NV) * 16u : static_cast<uint32_t>(D) * 2u;
    // Their stride in a stage: the same in both CTAs of a pair (ceil(NV/2)
    // vectors), so that the exchange slots after the ring sit at the same
    // offset in both.
    const uint32_t row_stride = PAIR ? static_cast<uint32_t>(NVh) * 16u : row_bytes;
    const uint32_t stage_bytes = R * NIN * row_stride;
    // SGS: [R][VPT][2][nt][4] sigmoid(z) at the start of shared memory (a
    // multiple of 1024 bytes, so the ring after it keeps its alignment), read
    // and written as float4.
    float* sgs = reinterpret_cast<float*>(smem);
    unsigned char* ring = smem + (SGS ? static_cast<size_t>(R) * VPT * 2 * nt * 16 : 0);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(S) * stage_bytes);
    uint64_t* empty = full + S;
    uint64_t* xbar = empty + S;                                        // PAIR: [2], the peer's half
    float* xslot = reinterpret_cast<float*>(xbar + (PAIR ? 2 : 0));    // PAIR: [2]
    float* rs = xslot + (PAIR ? 2 : 0);               // [S][R]
    float* red = rs + S * R;                          // [2][R][32]

    // This CTA's chunks: cta, cta+G, ...; only the globally last chunk can be
    // short, and if this CTA owns it, it is its last one.
    int n_my = 0;
    if (cta < nchunks) {
        const int64_t cnt = (nchunks - 1 - cta) / G + 1;
        const int64_t last = cta + (cnt - 1) * G;
        const int64_t last_rows = (T - last * C) < C ? (T - last * C) : C;
        n_my = static_cast<int>((cnt - 1) * C + last_rows);
    }
    const int n_it = (n_my + R - 1) / R;
    // k-th row of this CTA with the fixed chunk (C0 is a power of two: shifts).
    auto row_of = [&](int k) -> int64_t { return (cta + static_cast<int64_t>(k / C0) * G) * C0 + (k % C0); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 2);
            mbar_init(&empty[s], nw);
        }
        if (PAIR) {
            mbar_init(&xbar[0], 1);
            mbar_init(&xbar[1], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if constexpr (PAIR) cluster_sync_all();  // the peer's barriers exist before any exchange
    pdl_wait();  // first global memory access below

    if (warp == nw) {  // producer warp
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // Operands after g and x: residual g_res; gated z; fused add res, then g_res.
            const uint16_t* third = (M == kResidual) ? a.gres : (M == kGated ? a.z : a.res);
            const int64_t ld_third = (M == kResidual) ? a.ldgr : (M == kGated ? a.ldz : a.ldres);
            // Iteration i's first row, stepped like the consumers' (no division):
            // iterations come in order, R rows each, never straddling a chunk.
            int64_t row0 = cta * C;
            int po = 0;
            produce(full, empty, S, n_it, [&](int i, int s) {
                unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
                const int nvalid = min(n_my - i * R, R);
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nvalid) * NIN * row_bytes);
                for (int r = 0; r < nvalid; ++r)
                    cp_async4(&rs[s * R + r], a.rstd + (VC ? row0 + r : row_of(i * R + r)));
                cp_async_arrive_noinc(&full[s]);
                for (int r = 0; r < nvalid; ++r) {
                    const int64_t row = VC ? row0 + r : row_of(i * R + r);
                    unsigned char* dst = st + static_cast<size_t>(r) * NIN * row_stride;
                    bulk_g2s(dst, a.g + row * a.ldg + cb, row_bytes, &full[s], pol);
                    bulk_g2s(dst + row_stride, a.x + row * a.ldx + cb, row_bytes, &full[s], pol);
                    if (NIN >= 3)
                        bulk_g2s(dst + 2 * row_stride, third + row * ld_third + cb, row_bytes, &full[s], pol);
                    if (NIN == 4)
                        bulk_g2s(dst + 3 * row_stride, a.gres + row * a.ldgr + cb, row_bytes, &full[s], pol);
                }
                row0 += R;
                po += R;
                if (po == C) {  // next chunk of this CTA: G chunks further on
                    po = 0;
                    row0 += (G - 1) * C;
                }
            });
        }
        if constexpr (PAIR) {  // the pair's closing barrier (see the consumers' end)
            __syncwarp();
            cluster_sync_all();
        }
        return;
    }

    const float* wv = a.w + cb;  // this CTA's weights
    float we[VPT][8];
    if (!WL1) load_weights<VPT>(wv, a.zc, NV, nt, tid, we);
    float acc[VPT][8];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;

    int s = 0;
    uint32_t ph = 0;
    int kc = 0, ko = 0;  // this iteration's first row: chunk ordinal kc, offset ko within it
    bool xok = true;     // PAIR: every exchange so far arrived in time
    // PAIR: the peer's slots and barriers, as this CTA addresses them.
    const uint32_t peer_xslot = PAIR ? cluster_map(xslot, static_cast<uint32_t>(rank ^ 1)) : 0u;
    const uint32_t peer_xbar = PAIR ? cluster_map(xbar, static_cast<uint32_t>(rank ^ 1)) : 0u;
    for (int i = 0; i < n_it; ++i) {
        const bool ok = mbar_wait(&full[s], ph) && xok;
        const unsigned char* st = ring + static_cast<size_t>(s) * stage_bytes;
        const int nvalid = min(n_my - i * R, R);

        float gw[R][VPT][8];  // g*w_eff   (gated: g*q(z)*w_eff)
        float xs[R][VPT][8];  // x
        float gx[R][VPT][8];  // g*x       (gated: g*q(z)*x)
        float tz[R][VPT][8];  // residual: g_res; gated: z, then q(z); fused add: res
        float g0[R][VPT][8];  // gated: g q'(z)
        float rr[R];
        float sp[R];          // this thread's part of s = sum g x w_eff (gated: g q x w_eff)
        uint4 gv[R][VPT], xv[R][VPT], tv[R][VPT], fv[R][VPT];  // fv: fused add's g_res
#pragma unroll
        for (int r = 0; r < R; ++r) {
            rr[r] = 0.0f;
            if (r < nvalid) {
                rr[r] = rs[s * R + r];
                const unsigned char* src = st + static_cast<size_t>(r) * NIN * row_stride;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int v = j * nt + tid;
                    if (v < NV) {
                        gv[r][j] = ld_shared_v4(src + 16 * v);
                        xv[r][j] = ld_shared_v4(src + row_stride + 16 * v);
                        if (NIN >= 3) tv[r][j] = ld_shared_v4(src + 2 * row_stride + 16 * v);
                        if (NIN == 4) fv[r][j] = ld_shared_v4(src + 3 * row_stride + 16 * v);
                    }
                }
            }
        }
        // The stage is in registers: hand it back to the producer (HOLD: after
        // the row is done, since the operands are read again).
        const int s_used = s;
        if (!HOLD) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }

#pragma unroll
        for (int r = 0; r < R; ++r) {
            sp[r] = 0.0f;
            if (r < nvalid) {
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    if (j * nt + tid < NV) {
                        float gf[8], wj[8];
                        if (WL1) weights8(wv, a.zc, j * nt + tid, wj);
                        else
#pragma unroll
                            for (int e = 0; e < 8; ++e) wj[e] = we[j][e];
                        unpack_act<F16>(gv[r][j], gf);
                        norm_input<MODE>(xv[r][j], tv[r][j], xs[r][j]);  // x, or h = x + res
                        if (M == kResidual || M == kGated) unpack_act<F16>(tv[r][j], tz[r][j]);
                        if (M == kGated) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                if (SGS) {
                                    g0[r][j][e] = sigmoidf_rn(tz[r][j][e]);  // sigmoid(z), parked below
                                    gf[e] = fmul(gf[e], fmul(tz[r][j][e], g0[r][j][e]));  // g*q(z)
                                } else if (RMSN_BWD_LEAN) {
                                    gf[e] = fmul(gf[e], gate_value<SIG>(tz[r][j][e]));  // g*q(z)
                                } else {  // kept: g*q'(z) in g0, q(z) in tz
                                    float q, dq;
                                    gate_eval<SIG>(tz[r][j][e], q, dq);
                                    g0[r][j][e] = fmul(gf[e], dq);
                                    tz[r][j][e] = q;
                                    gf[e] = fmul(gf[e], q);
                                }
                            }
                            if constexpr (SGS) {
                                float4* slot = reinterpret_cast<float4*>(sgs) + ((r * VPT + j) * 2) * nt + tid;
                                slot[0] = make_float4(g0[r][j][0], g0[r][j][1], g0[r][j][2], g0[r][j][3]);
                                slot[nt] = make_float4(g0[r][j][4], g0[r][j][5], g0[r][j][6], g0[r][j][7]);
                            }
                        }
                        if constexpr (X2P1) {
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {  // element pairs; s in ascending element order
                                const float2 gw2 = fmul2(pair(gf, e), pair(wj, e));
                                gw[r][j][e] = gw2.x;
                                gw[r][j][e + 1] = gw2.y;
                                if (!RMSN_BWD_LEAN) {
                                    const float2 gx2 = fmul2(pair(gf, e), pair(xs[r][j], e));
                                    gx[r][j][e] = gx2.x;
                                    gx[r][j][e + 1] = gx2.y;
                                }
                                const float2 t2 = fmul2(gw2, pair(xs[r][j], e));
                                sp[r] = fadd(fadd(sp[r], t2.x), t2.y);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                gw[r][j][e] = fmul(gf[e], wj[e]);
                                if (!RMSN_BWD_LEAN) gx[r][j][e] = fmul(gf[e], xs[r][j][e]);
                                sp[r] = fadd(sp[r], fmul(gw[r][j][e], xs[r][j][e]));
                            }
                        }
                    }
                }
            }
        }
        float* rb = red + (i & 1) * (R * 32);
        if (!block_partial<R>(sp, rb, lane, warp, nt, ok)) {
            if (tid == 0) consumer_abort(full, S, i, n_it);
            if (PAIR) break;  // to the closing barrier: the peer may still store into this CTA
            return;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < nvalid) {
                const float r1 = rr[r];
                float s_tot = block_total<NWMAX>(rb + r * 32, nw);
                if constexpr (PAIR) {
                    // Exchange the halves (R is 1): thread 0 stores this CTA's half in
                    // the peer's slot b, whose barrier counts the 4 bytes; every thread
                    // waits for the peer's half in its own slot and adds the two in
                    // rank order (the same bits in both CTAs). Slot and barrier b serve
                    // every other row; a failed wait is voted at the next row.
                    const int b = i & 1;
                    if (tid == 0) {
                        mbar_arrive_expect_tx(&xbar[b], 4u);
                        st_async_f32(peer_xslot + 4u * b, s_tot, peer_xbar + 8u * b);
                    }
                    xok = mbar_wait_cluster(&xbar[b], static_cast<uint32_t>((i >> 1) & 1)) && xok;
                    const float s_peer = *reinterpret_cast<volatile float*>(&xslot[b]);
                    s_tot = rank == 0 ? fadd(s_tot, s_peer) : fadd(s_peer, s_tot);
                }
                const float coef = fmul(div_by_d(fmul(fmul(r1, r1), r1), D, a.inv_d_pow2), s_tot);
                const int64_t row = VC ? (cta + static_cast<int64_t>(kc) * G) * C + ko + r : row_of(i * R + r);
                uint16_t* dxrow = a.dx + row * a.lddx + cb;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int v = j * nt + tid;
                    if (v < NV) {
                        float wj[8];
                        if (WL1) weights8(wv, a.zc, v, wj);
                        else
#pragma unroll
                            for (int e = 0; e < 8; ++e) wj[e] = we[j][e];
                        if (HOLD) {  // the operands again, from the stage still held
                            const unsigned char* src = st + static_cast<size_t>(r) * NIN * row_stride;
                            gv[r][j] = ld_shared_v4(src + 16 * v);
                            xv[r][j] = ld_shared_v4(src + row_stride + 16 * v);
                            if (NIN >= 3) tv[r][j] = ld_shared_v4(src + 2 * row_stride + 16 * v);
                            if (NIN == 4) fv[r][j] = ld_shared_v4(src + 3 * row_stride + 16 * v);
                        }
                        if (RMSN_BWD_LEAN) {
                            // Recompute the phase-1 products from the packed row (same bits).
                            float gf[8];
                            unpack_act<F16>(gv[r][j], gf);
                            norm_input<MODE>(xv[r][j], tv[r][j], xs[r][j]);
                            if (M == kResidual || M == kGated) unpack_act<F16>(tv[r][j], tz[r][j]);
                            if constexpr (SGS) {
                                // sigmoid(z) from the slots; q = z sigmoid(z) (the same bits as
                                // before the reduction), q' = sigmoid(z) + q (1 - sigmoid(z)).
                                const float4* slot = reinterpret_cast<const float4*>(sgs) + ((r * VPT + j) * 2) * nt + tid;
                                const float4 lo = slot[0], hi = slot[nt];
                                const float sg[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float q = fmul(tz[r][j][e], sg[e]);
                                    const float dq = fadd(sg[e], fmul(q, fsub(1.0f, sg[e])));
                                    g0[r][j][e] = fmul(gf[e], dq);
                                    tz[r][j][e] = q;
                                    gf[e] = fmul(gf[e], q);
                                }
                            } else if (M == kGated) {
                                // The gate and its derivative, once: g*q'(z) in g0, q(z) in tz.
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    float q, dq;
                                    gate_eval<SIG>(tz[r][j][e], q, dq);
                                    g0[r][j][e] = fmul(gf[e], dq);
                                    tz[r][j][e] = q;
                                    gf[e] = fmul(gf[e], q);
                                }
                            }
                            if constexpr (X2RC) {
#pragma unroll
                                for (int e = 0; e < 8; e += 2) {
                                    const float2 gw2 = fmul2(pair(gf, e), pair(wj, e));
                                    const float2 gx2 = fmul2(pair(gf, e), pair(xs[r][j], e));
                                    gw[r][j][e] = gw2.x;
                                    gw[r][j][e + 1] = gw2.y;
                                    gx[r][j][e] = gx2.x;
                                    gx[r][j][e + 1] = gx2.y;
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    gw[r][j][e] = fmul(gf[e], wj[e]);
                                    gx[r][j][e] = fmul(gf[e], xs[r][j][e]);
                                }
                            }
                        }
                        float o[8], fg[8];
                        if (M == kFusedAdd) unpack_act<F16>(fv[r][j], fg);
                        if constexpr (X2OUT) {
                            const float2 r2 = both(r1), c2 = both(coef);
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {  // element pairs (products packed, their sums scalar)
                                const float2 p2 = fmul2(pair(gw[r][j], e), r2), q2 = fmul2(pair(xs[r][j], e), c2);
                                float2 d = make_float2(fsub(p2.x, q2.x), fsub(p2.y, q2.y));
                                if (M == kResidual) d = fadd2(d, pair(tz[r][j], e));
                                if (M == kFusedAdd) d = fadd2(d, pair(fg, e));
                                o[e] = d.x;
                                o[e + 1] = d.y;
                                const float2 t2 = fmul2(pair(gx[r][j], e), r2);
                                acc[j][e] = fadd(acc[j][e], t2.x);
                                acc[j][e + 1] = fadd(acc[j][e + 1], t2.y);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                float d = fsub(fmul(gw[r][j][e], r1), fmul(xs[r][j][e], coef));
                                if (M == kResidual) d = fadd(d, tz[r][j][e]);
                                if (M == kFusedAdd) d = fadd(d, fg[e]);
                                o[e] = d;
                                acc[j][e] = fadd(acc[j][e], fmul(gx[r][j][e], r1));
                            }
                        }
                        st_global_cs(dxrow + 8 * v, pack_act<F16>(o));
                        if (M == kGated) {
                            float dzv[8], yv[8];
                            // dz = (g q'(z)) u and y = u q(z), u = (x r) w_eff.
                            if constexpr (X2OUT) {
#pragma unroll
                                for (int e = 0; e < 8; e += 2) {
                                    const float2 u = fmul2(fmul2(pair(xs[r][j], e), both(r1)), pair(wj, e));
                                    const float2 dz2 = fmul2(pair(g0[r][j], e), u);
                                    const float2 y2 = fmul2(u, pair(tz[r][j], e));
                                    dzv[e] = dz2.x;
                                    dzv[e + 1] = dz2.y;
                                    yv[e] = y2.x;
                                    yv[e + 1] = y2.y;
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float u = fmul(fmul(xs[r][j][e], r1), wj[e]);
                                    dzv[e] = fmul(g0[r][j][e], u);
                                    yv[e] = fmul(u, tz[r][j][e]);
                                }
                            }
                            st_global_cs(a.dz + row * a.lddz + cb + 8 * v, pack_act<F16>(dzv));
                            if constexpr (RY) st_global_cs(a.y + row * a.ldy + cb + 8 * v, pack_act<F16>(yv));
                        } else if constexpr (RY) {
                            // The forward output again, from the saved rstd: same operations,
                            // same bits as the forward's y.
                            float yv[8];
                            if constexpr (X2OUT) {
#pragma unroll
                                for (int e = 0; e < 8; e += 2) {
                                    const float2 y2 = fmul2(fmul2(pair(xs[r][j], e), both(r1)), pair(wj, e));
                                    yv[e] = y2.x;
                                    yv[e + 1] = y2.y;
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e) yv[e] = fmul(fmul(xs[r][j][e], r1), wj[e]);
                            }
                            st_global_cs(a.y + row * a.ldy + cb + 8 * v, pack_act<F16>(yv));
                        }
                    }
                }
            }
        }
        if (HOLD) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s_used]);
        }
        // End of a chunk: write its partial row and restart the accumulators.
        const int k_last = i * R + nvalid - 1;
        if ((VC ? ko + nvalid == C : (k_last % C0) == C0 - 1) || k_last == n_my - 1) {
            const int64_t chunk = cta + static_cast<int64_t>(VC ? kc : k_last / C0) * G;
            float* prow = a.partials + chunk * D + cb;
            // Partials are re-read by pass 2 right away: keep them in L2.
            const uint64_t keep = policy_evict_last();
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = j * nt + tid;
                if (v < NV) {
                    st_global_f4_hint(prow + 8 * v, acc[j][0], acc[j][1], acc[j][2], acc[j][3], keep);
                    st_global_f4_hint(prow + 8 * v + 4, acc[j][4], acc[j][5], acc[j][6], acc[j][7], keep);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;
            }
        }
        ko += R;
        if (ko == C) {
            ko = 0;
            ++kc;
        }
    }
    if constexpr (PAIR) {
        // The last row's exchange has no next vote: take it here. Then every
        // thread of both CTAs meets once more, so that neither CTA exits while
        // the other may still store into its shared memory (after an abort
        // too: the peer's waits are bounded, so it gets here as well).
        if (!named_bar_and(kConsumerBarrier, nt, xok ? 1 : 0) && tid == 0) atomicOr(&g_wide_error, kErrWaitTimeout);
        pdl_release();
        cluster_sync_all();
        return;
    }
    pdl_release();
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

constexpr int kMaxSmemPerCta = 227 * 1024;

// Ring stages for a budget: at least 2, fewer than the budget allows only if
// the shared memory of a CTA cannot hold them, and 1 when even two stages do
// not fit (the four operands of a fused-add backward row beyond D = 14520).
// With one stage the consumers still hand it back as soon as it is in
// registers, so the next row's copy overlaps the row's arithmetic.
inline int stages_for(size_t budget, size_t stage_bytes, size_t per_stage_extra, size_t fixed) {
    size_t s = budget / stage_bytes;
    if (s > RMSN_MAX_STAGES) s = RMSN_MAX_STAGES;
    if (s < 2) s = 2;
    while (s > 1 && s * (stage_bytes + per_stage_extra) + fixed > static_cast<size_t>(kMaxSmemPerCta)) --s;
    return static_cast<int>(s);
}

template <int VPT, int MODE, int MAXT>
cudaError_t fwd_t(const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    constexpr int NIN = fwd_inputs(MODE);
    constexpr int R = fwd_rows<VPT, MAXT, MODE>();
    const size_t stage = static_cast<size_t>(R) * NIN * a.D * 2;
    const size_t fixed = 2 * R * 32 * 4;
    const int S = stages_for(RMSN_WIDE_FWD_SMEM, stage, 16, fixed);
    const size_t smem = S * (stage + 16) + fixed;
    if (smem > static_cast<size_t>(kMaxSmemPerCta)) return cudaErrorInvalidConfiguration;
    const int threads = c.threads + 32;
    const void* kern = reinterpret_cast<const void*>(wide_fwd_kernel<VPT, MODE, MAXT>);
    cudaError_t e = ensure_smem_attr(kern, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int occ = std::min(ctas_per_sm(kern, threads, static_cast<int>(smem)), RMSN_WIDE_FWD_CTAS_PER_SM);
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int64_t grid = std::min<int64_t>(a.T, static_cast<int64_t>(sm_count()) * occ);
    return launch_kernel(wide_fwd_kernel<VPT, MODE, MAXT>, static_cast<unsigned>(grid), threads, smem, st, a, S);
}

template <int VPT, int MODE, int MAXT, bool VC = false, bool PAIR = false>
cudaError_t bwd_t(const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    constexpr int NIN = bwd_inputs(MODE);
    constexpr int R = bwd_rows<VPT, MAXT, MODE, PAIR>();
    static_assert(!PAIR || (R == 1 && !VC), "a CTA pair runs one row per iteration in fixed chunks");
    constexpr bool SGS = base_mode(MODE) == kGated && !is_sigmoid_gate(MODE) && VPT <= 2 && RMSN_BWD_LEAN &&
                         RMSN_BWD_SGS;
    // A pair's CTA stages its half of the row: ceil(NV/2) vectors at most.
    const size_t row_bytes = PAIR ? static_cast<size_t>((a.D / 8 + 1) / 2) * 16 : static_cast<size_t>(a.D) * 2;
    const size_t stage = static_cast<size_t>(R) * NIN * row_bytes;
    const size_t fixed = 2 * R * 32 * 4 + (SGS ? static_cast<size_t>(R) * VPT * 8 * c.bwd_threads * 4 : 0) +
                         (PAIR ? 24 : 0);
    const int S = stages_for(MAXT > 256 ? RMSN_WIDE_BWD_SMEM_512 : RMSN_WIDE_BWD_SMEM, stage, 16 + 4 * R, fixed);
    const size_t smem = S * (stage + 16 + 4 * R) + fixed;
    if (smem > static_cast<size_t>(kMaxSmemPerCta)) return cudaErrorInvalidConfiguration;
    const int threads = c.bwd_threads + 32;
    const void* kern = reinterpret_cast<const void*>(wide_bwd_kernel<VPT, MODE, MAXT, VC, PAIR>);
    cudaError_t e = ensure_smem_attr(kern, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t nchunks = (a.T + a.chunk - 1) / a.chunk;
    if constexpr (PAIR) {
        // One pair per chunk, up to the pairs that can be resident at once.
        const int np = pair_clusters(kern, threads, static_cast<int>(smem));
        if (np < 1) return cudaErrorInvalidConfiguration;
        const int64_t pairs = std::min<int64_t>(nchunks, np);
        return launch_kernel_clustered(wide_bwd_kernel<VPT, MODE, MAXT, VC, PAIR>, 2u,
                                       static_cast<unsigned>(2 * pairs), threads, smem, st, a, S);
    } else {
        const int occ =
            std::min(ctas_per_sm(kern, threads, static_cast<int>(smem)), bwd_ctas_per_sm<VPT, MAXT, MODE>());
        if (occ < 1) return cudaErrorInvalidConfiguration;
        const int64_t grid = std::min<int64_t>(nchunks, static_cast<int64_t>(sm_count()) * occ);
        return launch_kernel(wide_bwd_kernel<VPT, MODE, MAXT, VC>, static_cast<unsigned>(grid), threads, smem, st,
                             a, S);
    }
}

template <int MODE>
cudaError_t fwd_dispatch(const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    // The shapes row_cfg gives: one and two vectors a thread on up to 256
    // threads (D <= 4096), four on up to 256 (D <= 8192) or 512 (beyond).
    const bool big = c.threads > 256;
    switch (c.vpt) {
        case 1: return big ? cudaErrorInvalidValue : fwd_t<1, MODE, 256>(a, c, st);
        case 2: return big ? cudaErrorInvalidValue : fwd_t<2, MODE, 256>(a, c, st);
        case 4: return big ? fwd_t<4, MODE, 512>(a, c, st) : fwd_t<4, MODE, 256>(a, c, st);
        default: return cudaErrorInvalidValue;
    }
}

template <int MODE>
cudaError_t bwd_dispatch(const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    const bool big = c.bwd_threads > 256;
    // A chunk other than kWideChunkRows (2048 < D <= 7168 only) runs the
    // stepping instantiation of the two kernels those widths use.
    const bool vc = a.chunk != kWideChunkRows;
    // Only the shapes run_bwd gives are instantiated; any other returns an error.
    switch (c.bwd_vpt) {
        case 1:  // D <= 2048: up to 256 threads
            if (vc || big) return cudaErrorInvalidValue;
            return bwd_t<1, MODE, 256>(a, c, st);
        case 2:
            // Rows of more than 1024 vectors: a CTA pair per row, two vectors a
            // thread on up to 512 threads in each CTA.
            if (c.bwd_pair) return vc ? cudaErrorInvalidValue : bwd_t<2, MODE, 512, false, true>(a, c, st);
            if (big) {
                if (!vc) return bwd_t<2, MODE, 512>(a, c, st);
                // Shortened chunks on 512 threads: the modes with three or four
                // operands at 4096 < D <= 7168 (the plain mode runs those on 224).
                if constexpr (base_mode(MODE) != kPlain) return bwd_t<2, MODE, 512, true>(a, c, st);
                return cudaErrorInvalidValue;
            }
            if (c.bwd_threads <= 128) {  // the plain mode's rows of 2 vectors a thread on <= 128 threads
                if constexpr (base_mode(MODE) == kPlain) return vc ? cudaErrorInvalidValue : bwd_t<2, MODE, 128>(a, c, st);
                return cudaErrorInvalidValue;
            }
            return vc ? bwd_t<2, MODE, 256, true>(a, c, st) : bwd_t<2, MODE, 256>(a, c, st);
        case 4:  // the plain mode only (the others run these rows on two vectors, or on CTA pairs)
            if constexpr (base_mode(MODE) == kPlain) {
                // Rows of more than 1152 vectors on 512 threads; 4096 < D <= 7168 on <= 224.
                if (big) return vc ? cudaErrorInvalidValue : bwd_t<4, MODE, 512>(a, c, st);
                if (c.bwd_threads <= 224)
                    return vc ? bwd_t<4, MODE, 224, true>(a, c, st) : bwd_t<4, MODE, 224>(a, c, st);
            }
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

}  // namespace rmsn
