// Narrow-row kernels (D <= 256): many rows per CTA, one lane group per row.
// Kernel and launcher templates, included by the translation units that
// instantiate them (narrow.cu: bf16 activations; narrow_f16.cu: fp16).
//
// Design (GB300, HBM-bound):
//   * A row of D <= 256 16-bit values is at most 32 16-byte vectors, so G lanes
//     (G = D/8 rounded up to a power of two) own one row: the row sum is an
//     xor-butterfly inside the group (offsets G/2..1), with no barrier at all.
//     256 consumer threads therefore reduce P = 256/G rows at a time.
//   * Warp-specialised pipeline as on the wide path: a producer warp keeps S
//     stages of RS rows in flight with 2-D tiled tensor copies
//     (cp.async.bulk.tensor.2d, one per operand per stage; the tensor map
//     carries the row stride, and rows past T arrive as zeros), consumers
//     release a stage through its "empty" mbarrier once they have read it.
//     The backward's rstd tile rides in the same stage through a 1-D tensor map.
//   * The tree of a row depends only on D (its G lanes, ascending sum over the
//     8 values of each lane's vector, then the butterfly), so every row's bits
//     are independent of T, its position, the other rows and the GPU.
//   * Weight gradient: each CTA owns whole chunks of CN rows. Lane group gr of
//     the CTA accumulates, per column, the rows gr, gr+P, gr+2P, ... of the
//     chunk in ascending order; at the end of the chunk the P group totals are
//     added in group order through shared memory and written as the chunk's
//     partial row. No atomics.
//
// Sources: as wide.cu (Megatron-LM pull request 6859; RL-Kernel pull requests
// 414 and 467 — the gated norm of the latter is the D=128 workload here).
#pragma once

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

// Launch shapes, chosen by measurement on GB300 (262144 x 128 gated): 4
// forward CTAs of 48 KB rings per SM, 3 backward CTAs of 48 KB rings (plus the
// chunk combine buffer) with at most 72 registers per thread.
#ifndef RMSN_NARROW_FWD_SMEM
#define RMSN_NARROW_FWD_SMEM (48 * 1024)
#endif
#ifndef RMSN_NARROW_FWD_CTAS_PER_SM
#define RMSN_NARROW_FWD_CTAS_PER_SM 4
#endif
#ifndef RMSN_NARROW_BWD_SMEM
#define RMSN_NARROW_BWD_SMEM (48 * 1024)
#endif
#ifndef RMSN_NARROW_BWD_CTAS_PER_SM
#define RMSN_NARROW_BWD_CTAS_PER_SM 3
#endif
#ifndef RMSN_NARROW_BWD_MINB
#define RMSN_NARROW_BWD_MINB 3  // backward CTAs that must fit on one SM (register budget)
#endif

namespace rmsn {

namespace {

// The narrow kernels' 16-byte output stores (y, the copy, dx, dz) at the L2's
// ordinary write-back policy rather than as streaming (evict-first) stores:
// Qwen3-Next gated step, 262144 x 128, 91.2 -> 90.7 us.
__device__ __forceinline__ void st_store_out(void* p, uint4 v) { __stwb(reinterpret_cast<uint4*>(p), v); }

// Device error word of the including translation unit.
__device__ unsigned int g_narrow_error;

cudaError_t read_narrow_error_word(unsigned* flags, bool clear) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_narrow_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *flags |= v;
    if (clear && v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_narrow_error, &zero, sizeof(zero));
    }
    return e;
}

// The operands' tensor maps, passed by value as one grid-constant parameter.
struct NarrowMaps {
    CUtensorMap a;     // x (forward) / g (backward)
    CUtensorMap b;     // z or res (forward) / x (backward)
    CUtensorMap c;     // g_res, z or res (backward)
    CUtensorMap d;     // g_res (fused-add backward)
    CUtensorMap rstd;  // backward
};

// The values a row is normalised over: x, or the fp32 sum x + res (fused add).
template <int MODE>
__device__ __forceinline__ void narrow_norm_input(const uint4 xv, const uint4 sv, float (&f)[8]) {
    unpack_act<is_f16(MODE)>(xv, f);
    if (is_fused(MODE)) {
        float rv[8];
        unpack_act<is_f16(MODE)>(sv, rv);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = fadd(f[e], rv[e]);
    }
}

constexpr int kNarrowConsumerBarrier = 1;

// Rows of one pass (P), of one stage (RS) and of one weight-gradient chunk (CN).
template <int G> __host__ __device__ constexpr int narrow_pass_rows() { return kNarrowThreads / G; }
// Rows of 256 B < 2D <= 512 B use 32-row stages so that two stages of four
// operands still fit in shared memory; narrower rows use RMSN_NARROW_STAGE_ROWS
// (or P). The stage size does not enter any reduction tree.
#ifndef RMSN_NARROW_STAGE_ROWS
#define RMSN_NARROW_STAGE_ROWS 32
#endif
template <int G> __host__ __device__ constexpr int narrow_stage_rows() {
    return G == 32 ? 32
                   : (narrow_pass_rows<G>() > RMSN_NARROW_STAGE_ROWS ? narrow_pass_rows<G>() : RMSN_NARROW_STAGE_ROWS);
}
// The forward streams at most two operands, so its stages can be longer: each
// lane then handles more rows per stage wait and release (262144 x 128 gated:
// 33.2 -> 31.5 us with 64-row stages).
#ifndef RMSN_NARROW_FWD_STAGE_ROWS
#define RMSN_NARROW_FWD_STAGE_ROWS 64
#endif
template <int G> __host__ __device__ constexpr int narrow_fwd_stage_rows() {
    return narrow_pass_rows<G>() > RMSN_NARROW_FWD_STAGE_ROWS ? narrow_pass_rows<G>() : RMSN_NARROW_FWD_STAGE_ROWS;
}
template <int G> __host__ __device__ constexpr int narrow_chunk_rows() {
    return narrow_stage_rows<G>() > kNarrowChunkRowsMin ? narrow_stage_rows<G>() : kNarrowChunkRowsMin;
}

// Producer loop shared by both kernels (one lane). Stage index and phase
// advance together; on a consumer stall, drain (bounded) and flag.
template <typename Issue>
__device__ __forceinline__ void narrow_produce(uint64_t* full, uint64_t* empty, int S, int n_it, Issue&& issue) {
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < n_it; ++i) {
        if (i >= S && !mbar_wait(&empty[s], ph ^ 1u)) {
            for (int j = i - S; j < i; ++j) (void)mbar_wait(&full[j % S], static_cast<uint32_t>((j / S) & 1));
            atomicOr(&g_narrow_error, kErrWaitTimeout);
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

__device__ __forceinline__ void load_weights8(const float* w, int zc, bool valid, int l, float (&we)[8]) {
    if (valid) {
        const float4 lo = __ldg(reinterpret_cast<const float4*>(w) + 2 * l);
        const float4 hi = __ldg(reinterpret_cast<const float4*>(w) + 2 * l + 1);
        we[0] = lo.x; we[1] = lo.y; we[2] = lo.z; we[3] = lo.w;
        we[4] = hi.x; we[5] = hi.y; we[6] = hi.z; we[7] = hi.w;
        if (zc) {
#pragma unroll
            for (int e = 0; e < 8; ++e) we[e] = fadd(we[e], 1.0f);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) we[e] = 0.0f;
    }
}

// ---------------------------------------------------------------------------
// Forward. CTA = 256 consumers + 1 producer warp; stage = RS rows of x (and z).
// Consumer warps never synchronise with each other.
// ---------------------------------------------------------------------------
template <int MODE, int G>
__global__ void __launch_bounds__(kNarrowThreads + 32)
narrow_fwd_kernel(const FwdArgs a, const __grid_constant__ NarrowMaps m, const int S) {
    constexpr int M = base_mode(MODE);
    constexpr bool F16 = is_f16(MODE);
    constexpr bool SIG = is_sigmoid_gate(MODE);
    static_assert(!(M == kGatedHF && F16), "the HF-convention witness is a bf16 forward");
    constexpr int NIN = fwd_inputs(MODE);
    constexpr int P = narrow_pass_rows<G>();
    constexpr int RS = narrow_fwd_stage_rows<G>();
    constexpr int NP = RS / P;
    extern __shared__ __align__(128) unsigned char smem[];
    const int D = a.D;
    const int NV = D >> 3;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int gr = tid / G, l = tid % G;
    const bool lane_valid = l < NV;
    const int64_t T = a.T;
    const int nblocks = static_cast<int>((T + RS - 1) / RS);
    const int Gd = gridDim.x;
    const int cta = blockIdx.x;
    const uint32_t tile_bytes = static_cast<uint32_t>(RS) * D * 2u;
    const uint32_t stage_bytes = NIN * tile_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t* empty = full + S;
    const int n_it = cta < nblocks ? (nblocks - 1 - cta) / Gd + 1 : 0;  // blocks cta, cta+Gd, ...

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kNarrowThreads / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();  // first global memory access below

    if (warp == kNarrowThreads / 32) {  // producer warp
        if (lane == 0) {
            prefetch_tensormap(&m.a);
            if (NIN == 2) prefetch_tensormap(&m.b);
            // Ordinary L2 priority for the streamed tiles: at evict_first they
            // could never displace the lines of higher priority that other
            // kernels leave in L2 (ordinary stores, evict_last partial rows),
            // and kept only what those leave free (Qwen3-Next gated step,
            // 262144 x 128, after such kernels: 95.9 -> 90.5 us; 90.2 us in a
            // clean L2 either way).
            const uint64_t pol = policy_evict_normal();
            narrow_produce(full, empty, S, n_it, [&](int i, int s) {
                unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
                const int row0 = (cta + i * Gd) * RS;
                mbar_arrive_expect_tx(&full[s], stage_bytes);
                tensor2d_g2s(st, &m.a, 0, row0, &full[s], pol);
                if (NIN == 2) tensor2d_g2s(st + tile_bytes, &m.b, 0, row0, &full[s], pol);
            });
        }
        return;
    }

    float we[8];
    load_weights8(a.w, a.zc, lane_valid, l, we);

    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < n_it; ++i) {
        if (!mbar_wait(&full[s], ph)) {
            // This warp stops; the producer notices the missing release and drains.
            if (lane == 0) atomicOr(&g_narrow_error, kErrWaitTimeout);
            return;
        }
        const unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
        const int64_t row0 = static_cast<int64_t>(cta + i * Gd) * RS;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int rs_ = p * P + gr;
            uint4 xv = make_uint4(0, 0, 0, 0), zv = make_uint4(0, 0, 0, 0);
            if (lane_valid) {
                xv = ld_shared_v4(st + (static_cast<size_t>(rs_) * D + 8 * l) * 2);
                if (NIN == 2) zv = ld_shared_v4(st + tile_bytes + (static_cast<size_t>(rs_) * D + 8 * l) * 2);
            }
            if (p == NP - 1) {  // whole stage read: release it
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            float f[8];
            narrow_norm_input<MODE>(xv, zv, f);  // x, or h = x + res
            // The gate does not depend on the row's statistic: evaluated here, it
            // overlaps the row reduction instead of following it.
            float q[8];
            if (is_gated(MODE)) {
                float zf[8];
                unpack_act<F16>(zv, zf);
#pragma unroll
                for (int e = 0; e < 8; ++e) q[e] = M == kGatedHF ? fmul(zf[e], sigmoidf_rn(zf[e])) : gate_value<SIG>(zf[e]);
            }
            float ss = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fadd(ss, fmul(f[e], f[e]));
            ss = group_sum<G>(ss);
            const float r = rsqrtf(fadd(div_by_d(ss, D, a.inv_d_pow2), a.eps));
            const int64_t row = row0 + rs_;
            if (row < T) {
                if (l == 0) a.rstd[row] = r;
                if (lane_valid) {
                    float o[8];
                    if (M == kGated) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = fmul(fmul(fmul(f[e], r), we[e]), q[e]);
                    } else if (M == kGatedHF) {
                        // HF convention: normalised value and weight multiply in bf16.
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float n = round_bf16f(fmul(f[e], r));
                            const float t = round_bf16f(fmul(round_bf16f(we[e]), n));
                            o[e] = fmul(t, q[e]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = fmul(fmul(f[e], r), we[e]);
                    }
                    st_store_out(a.y + row * a.ldy + 8 * l, pack_act<F16>(o));
                    if (M == kResidual) st_store_out(a.xc + row * a.ldxc + 8 * l, xv);
                    if (is_fused(MODE)) st_store_out(a.xc + row * a.ldxc + 8 * l, pack_act<F16>(f));  // x + res
                }
            }
        }
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
    }
    pdl_release();
}

// ---------------------------------------------------------------------------
// Backward pass 1. Stage = RS rows of g, x (and g_res or z) plus their rstd.
// ---------------------------------------------------------------------------
template <int MODE, int G>
__global__ void __launch_bounds__(kNarrowThreads + 32, RMSN_NARROW_BWD_MINB)
narrow_bwd_kernel(const BwdArgs a, const __grid_constant__ NarrowMaps m, const int S) {
    constexpr int M = base_mode(MODE);
    constexpr bool F16 = is_f16(MODE);
    constexpr bool SIG = is_sigmoid_gate(MODE);
    constexpr int NIN = bwd_inputs(MODE);
    constexpr int P = narrow_pass_rows<G>();
    constexpr int RS = narrow_stage_rows<G>();
    constexpr int NP = RS / P;
    constexpr int CN = narrow_chunk_rows<G>();
    constexpr int NSC = CN / RS;  // stages per chunk
    constexpr bool RY = is_recompute(MODE);  // also write y (a.y is then not null)
    extern __shared__ __align__(128) unsigned char smem[];
    const int D = a.D;
    const int NV = D >> 3;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int gr = tid / G, l = tid % G;
    const bool lane_valid = l < NV;
    const int64_t T = a.T;
    const int nblocks = static_cast<int>((T + RS - 1) / RS);
    const int nchunks = static_cast<int>((T + CN - 1) / CN);
    const int Gd = gridDim.x;
    const int cta = blockIdx.x;
    const uint32_t tile_bytes = static_cast<uint32_t>(RS) * D * 2u;
    const uint32_t stage_bytes = NIN * tile_bytes + RS * 4u;  // + rstd tile
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
    uint64_t* empty = full + S;
    float* comb = reinterpret_cast<float*>(empty + S);  // [2][P][D]

    // Chunks cta, cta+Gd, ...; NSC stages each, except that the globally last
    // chunk may have fewer (it is this CTA's last chunk if it owns it).
    int n_it = 0;
    if (cta < nchunks) {
        const int cnt = (nchunks - 1 - cta) / Gd + 1;
        const int last = cta + (cnt - 1) * Gd;
        n_it = (cnt - 1) * NSC + min(NSC, nblocks - last * NSC);
    }
    auto block_of = [&](int i) { return (cta + (i / NSC) * Gd) * NSC + (i % NSC); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kNarrowThreads / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();  // first global memory access below

    if (warp == kNarrowThreads / 32) {  // producer warp
        if (lane == 0) {
            prefetch_tensormap(&m.a);
            prefetch_tensormap(&m.b);
            if (NIN >= 3) prefetch_tensormap(&m.c);
            if (NIN == 4) prefetch_tensormap(&m.d);
            prefetch_tensormap(&m.rstd);
            const uint64_t pol = policy_evict_normal();  // as in the forward
            narrow_produce(full, empty, S, n_it, [&](int i, int s) {
                unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
                const int row0 = block_of(i) * RS;
                mbar_arrive_expect_tx(&full[s], stage_bytes);
                tensor2d_g2s(st, &m.a, 0, row0, &full[s], pol);
                tensor2d_g2s(st + tile_bytes, &m.b, 0, row0, &full[s], pol);
                if (NIN >= 3) tensor2d_g2s(st + 2 * tile_bytes, &m.c, 0, row0, &full[s], pol);
                if (NIN == 4) tensor2d_g2s(st + 3 * tile_bytes, &m.d, 0, row0, &full[s], pol);
                tensor1d_g2s(st + NIN * tile_bytes, &m.rstd, row0, &full[s], pol);
            });
        }
        return;
    }

    float we[8];
    load_weights8(a.w, a.zc, lane_valid, l, we);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;

    bool ok = true;
    int s = 0, cbuf = 0;
    uint32_t ph = 0;
    for (int i = 0; i < n_it; ++i) {
        ok = mbar_wait(&full[s], ph) && ok;
        const unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
        const float* rtile = reinterpret_cast<const float*>(st + NIN * tile_bytes);
        const int64_t row0 = static_cast<int64_t>(block_of(i)) * RS;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int rs_ = p * P + gr;
            uint4 gv = make_uint4(0, 0, 0, 0), xv = gv, tv = gv, fv = gv;
            if (lane_valid) {
                const size_t off = (static_cast<size_t>(rs_) * D + 8 * l) * 2;
                gv = ld_shared_v4(st + off);
                xv = ld_shared_v4(st + tile_bytes + off);
                if (NIN >= 3) tv = ld_shared_v4(st + 2 * tile_bytes + off);
                if (NIN == 4) fv = ld_shared_v4(st + 3 * tile_bytes + off);
            }
            const float r = rtile[rs_];
            if (p == NP - 1) {  // whole stage read: release it
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            // gf: g, or g q(z) (gated); gd (gated): g q'(z). The gate is evaluated
            // once, before the row reduction; after it only gf, gd, x and the
            // packed z (for the optional y) are needed.
            float gf[8], xf[8], tf[8], ff[8], gd[8];
            unpack_act<F16>(gv, gf);
            narrow_norm_input<MODE>(xv, tv, xf);  // x, or h = x + res
            if (M == kResidual) unpack_act<F16>(tv, tf);
            if (M == kFusedAdd) unpack_act<F16>(fv, ff);
            if (M == kGated) {
                float zf[8], q[8], dq[8];
                unpack_act<F16>(tv, zf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    gate_eval<SIG>(zf[e], q[e], dq[e]);
                    gd[e] = fmul(gf[e], dq[e]);  // g q'(z)
                    gf[e] = fmul(gf[e], q[e]);   // g q(z)
                }
            }
            float gw[8];
            float sp = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                gw[e] = fmul(gf[e], we[e]);
                sp = fadd(sp, fmul(gw[e], xf[e]));
            }
            sp = group_sum<G>(sp);
            const float coef = fmul(div_by_d(fmul(fmul(r, r), r), D, a.inv_d_pow2), sp);
            const int64_t row = row0 + rs_;
            if (row < T && lane_valid) {
                float o[8];
                if (M == kGated) {
                    // dx; dw term (g q) (x r); dz = (g q') u with u = (x r) w_eff; y = u q.
                    float dzv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        o[e] = fsub(fmul(gw[e], r), fmul(xf[e], coef));
                        const float xr = fmul(xf[e], r);
                        acc[e] = fadd(acc[e], fmul(gf[e], xr));
                        dzv[e] = fmul(gd[e], fmul(xr, we[e]));
                    }
                    st_store_out(a.dx + row * a.lddx + 8 * l, pack_act<F16>(o));
                    st_store_out(a.dz + row * a.lddz + 8 * l, pack_act<F16>(dzv));
                    if constexpr (RY) {
                        // The forward output again (the forward's operations, same bits).
                        float zf[8], yv[8];
                        unpack_act<F16>(tv, zf);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            yv[e] = fmul(fmul(fmul(xf[e], r), we[e]), gate_value<SIG>(zf[e]));
                        st_store_out(a.y + row * a.ldy + 8 * l, pack_act<F16>(yv));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float d = fsub(fmul(gw[e], r), fmul(xf[e], coef));
                        if (M == kResidual) d = fadd(d, tf[e]);
                        if (M == kFusedAdd) d = fadd(d, ff[e]);
                        o[e] = d;
                        acc[e] = fadd(acc[e], fmul(fmul(gf[e], xf[e]), r));
                    }
                    st_store_out(a.dx + row * a.lddx + 8 * l, pack_act<F16>(o));
                    if constexpr (RY) {
                        // The forward output again, from the saved rstd (same bits as the forward).
                        float yv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) yv[e] = fmul(fmul(xf[e], r), we[e]);
                        st_store_out(a.y + row * a.ldy + 8 * l, pack_act<F16>(yv));
                    }
                }
            }
        }
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
        // End of a chunk: add the P lane-group totals in group order.
        if ((i % NSC) == NSC - 1 || i == n_it - 1) {
            float* cb = comb + cbuf * (P * D);
            if (lane_valid) {
#pragma unroll
                for (int e = 0; e < 8; ++e) cb[gr * D + 8 * l + e] = acc[e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
            if (!named_bar_and(kNarrowConsumerBarrier, kNarrowThreads, ok ? 1 : 0)) {
                if (tid == 0) atomicOr(&g_narrow_error, kErrWaitTimeout);
                return;
            }
            const int64_t chunk = cta + static_cast<int64_t>(i / NSC) * Gd;
            const uint64_t keep = policy_evict_last();  // re-read by pass 2 right away
            for (int col = tid; col < D; col += kNarrowThreads) {
                float t = cb[col];
                for (int q = 1; q < P; ++q) t = fadd(t, cb[q * D + col]);
                st_global_f1_hint(a.partials + chunk * D + col, t, keep);
            }
            cbuf ^= 1;
        }
    }
    pdl_release();
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------

constexpr int kMaxSmem = 227 * 1024;

int narrow_stages(size_t budget, size_t stage, size_t fixed) {
    size_t s = budget / stage;
    if (s > 16) s = 16;
    while (s > 2 && s * (stage + 16) + fixed > static_cast<size_t>(kMaxSmem)) --s;
    return static_cast<int>(s < 2 ? 2 : s);
}

template <int MODE, int G>
cudaError_t nfwd_t(const FwdArgs& a, cudaStream_t st) {
    constexpr int RS = narrow_fwd_stage_rows<G>();
    constexpr int NIN = fwd_inputs(MODE);
    NarrowMaps m;
    std::memset(&m, 0, sizeof(m));
    constexpr bool F16 = is_f16(MODE);
    cudaError_t e = encode_rows_2d(&m.a, a.x, a.T, a.D, a.ldx, RS, F16);
    if (e == cudaSuccess && is_gated(MODE)) e = encode_rows_2d(&m.b, a.z, a.T, a.D, a.ldz, RS, F16);
    if (e == cudaSuccess && is_fused(MODE)) e = encode_rows_2d(&m.b, a.res, a.T, a.D, a.ldres, RS, F16);
    if (e != cudaSuccess) return e;
    const size_t stage = static_cast<size_t>(NIN) * RS * a.D * 2;
    const int S = narrow_stages(RMSN_NARROW_FWD_SMEM, stage, 0);
    const size_t smem = S * (stage + 16);
    if (smem > static_cast<size_t>(kMaxSmem)) return cudaErrorInvalidConfiguration;
    const void* kern = reinterpret_cast<const void*>(narrow_fwd_kernel<MODE, G>);
    e = ensure_smem_attr(kern, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int threads = kNarrowThreads + 32;
    const int occ = std::min(ctas_per_sm(kern, threads, static_cast<int>(smem)), RMSN_NARROW_FWD_CTAS_PER_SM);
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int64_t nblocks = (a.T + RS - 1) / RS;
    const int64_t grid = std::min<int64_t>(nblocks, static_cast<int64_t>(sm_count()) * occ);
    return launch_kernel(narrow_fwd_kernel<MODE, G>, static_cast<unsigned>(grid), threads, smem, st, a, m, S);
}

template <int MODE, int G>
cudaError_t nbwd_t(const BwdArgs& a, cudaStream_t st) {
    constexpr int RS = narrow_stage_rows<G>();
    constexpr int CN = narrow_chunk_rows<G>();
    constexpr int P = narrow_pass_rows<G>();
    constexpr int NIN = bwd_inputs(MODE);
    NarrowMaps m;
    std::memset(&m, 0, sizeof(m));
    constexpr int M = base_mode(MODE);
    constexpr bool F16 = is_f16(MODE);
    cudaError_t e = encode_rows_2d(&m.a, a.g, a.T, a.D, a.ldg, RS, F16);
    if (e == cudaSuccess) e = encode_rows_2d(&m.b, a.x, a.T, a.D, a.ldx, RS, F16);
    if (e == cudaSuccess && M == kResidual) e = encode_rows_2d(&m.c, a.gres, a.T, a.D, a.ldgr, RS, F16);
    if (e == cudaSuccess && M == kGated) e = encode_rows_2d(&m.c, a.z, a.T, a.D, a.ldz, RS, F16);
    if (e == cudaSuccess && is_fused(MODE)) e = encode_rows_2d(&m.c, a.res, a.T, a.D, a.ldres, RS, F16);
    if (e == cudaSuccess && M == kFusedAdd) e = encode_rows_2d(&m.d, a.gres, a.T, a.D, a.ldgr, RS, F16);
    if (e == cudaSuccess) e = encode_vec_1d(&m.rstd, a.rstd, a.T, RS);
    if (e != cudaSuccess) return e;
    const size_t stage = static_cast<size_t>(NIN) * RS * a.D * 2 + RS * 4;
    const size_t fixed = static_cast<size_t>(2) * P * a.D * 4;
    const int S = narrow_stages(RMSN_NARROW_BWD_SMEM, stage, fixed);
    const size_t smem = S * (stage + 16) + fixed;
    if (smem > static_cast<size_t>(kMaxSmem)) return cudaErrorInvalidConfiguration;
    const void* kern = reinterpret_cast<const void*>(narrow_bwd_kernel<MODE, G>);
    e = ensure_smem_attr(kern, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int threads = kNarrowThreads + 32;
    const int occ = std::min(ctas_per_sm(kern, threads, static_cast<int>(smem)), RMSN_NARROW_BWD_CTAS_PER_SM);
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int64_t nchunks = (a.T + CN - 1) / CN;
    const int64_t grid = std::min<int64_t>(nchunks, static_cast<int64_t>(sm_count()) * occ);
    return launch_kernel(narrow_bwd_kernel<MODE, G>, static_cast<unsigned>(grid), threads, smem, st, a, m, S);
}

template <int MODE>
cudaError_t nfwd_dispatch(const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    switch (c.group) {
        case 1: return nfwd_t<MODE, 1>(a, st);
        case 2: return nfwd_t<MODE, 2>(a, st);
        case 4: return nfwd_t<MODE, 4>(a, st);
        case 8: return nfwd_t<MODE, 8>(a, st);
        case 16: return nfwd_t<MODE, 16>(a, st);
        case 32: return nfwd_t<MODE, 32>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

template <int MODE>
cudaError_t nbwd_dispatch(const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    switch (c.group) {
        case 1: return nbwd_t<MODE, 1>(a, st);
        case 2: return nbwd_t<MODE, 2>(a, st);
        case 4: return nbwd_t<MODE, 4>(a, st);
        case 8: return nbwd_t<MODE, 8>(a, st);
        case 16: return nbwd_t<MODE, 16>(a, st);
        case 32: return nbwd_t<MODE, 32>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

}  // namespace rmsn
