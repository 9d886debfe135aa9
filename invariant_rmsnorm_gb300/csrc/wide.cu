// Wide-row kernels (D > 256): one CTA reduces one row at a time.
//
// Design (GB300, HBM-bound):
//   * Persistent grid: at most (SM count x resident CTAs) CTAs walk a fixed
//     sequence of rows. Thread 0 keeps S rows in flight with 1-D bulk TMA copies
//     (cp.async.bulk global->shared, completion counted on a per-stage
//     mbarrier), so loads never wait on the arithmetic.
//   * Each thread owns VPT 16-byte vectors of the row at slots v = k*NT + tid
//     (coalesced, conflict-free shared reads). Row values stay in registers
//     between the reduction and the output.
//   * Fixed reduction tree (a function of D only): per-thread ascending sum
//     over its slots and the 8 lanes of each vector, an xor-butterfly over the
//     warp (offsets 16..1), then the per-warp totals added in warp order. The
//     same row therefore gives the same bits whatever T, its position, the
//     other rows, the grid or the GPU.
//   * fp32 arithmetic with every multiply and add rounded separately (no FMA
//     contraction), rsqrtf for the inverse RMS, bf16 round-to-nearest-even
//     outputs written with 128-bit streaming stores.
//   * Backward weight gradient: a CTA owns whole chunks of kWideChunkRows rows,
//     accumulates g*x*r per column in ascending row order in registers and
//     writes one fp32 partial row per chunk; no atomics anywhere.
//
// Sources: Megatron-LM pull request 6859 "Fix the batch-invariant RMSNorm
// forward and its input gradient" (What does this PR do, items 1-2);
// RL-Kernel pull request 414 "[DSv4][P1-5] rmsnorm_residual" (Implementation:
// rsqrt, (x*r)*gamma, ascending fp32 reductions, separate rounding, no atomics;
// Summary: the residual variant returns a copy of x); RL-Kernel pull request
// 467 "...zero-centred RMSNorm references and CUDA kernel" (+1 in fp32, gated
// norm with the weight multiply in fp32).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

#ifndef RMSN_WIDE_FWD_SMEM
#define RMSN_WIDE_FWD_SMEM (64 * 1024)   // target ring bytes per CTA (forward)
#endif
#ifndef RMSN_WIDE_FWD_CTAS_PER_SM
#define RMSN_WIDE_FWD_CTAS_PER_SM 4
#endif
#ifndef RMSN_WIDE_BWD_SMEM
#define RMSN_WIDE_BWD_SMEM (192 * 1024)  // target ring bytes per CTA (backward)
#endif
#ifndef RMSN_WIDE_BWD_CTAS_PER_SM
#define RMSN_WIDE_BWD_CTAS_PER_SM 1
#endif
#ifndef RMSN_MAX_STAGES
#define RMSN_MAX_STAGES 16
#endif

namespace rmsn {

static __device__ unsigned int g_wide_error;

cudaError_t wide_read_error(unsigned* flags, bool clear) {
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

namespace {

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

// First half of the block-wide fixed tree: butterfly within each warp, lane 0
// parks the warp total in `red` (a 32-float slot owned by this row). The
// barrier doubles as the error vote: returns the CTA-wide AND of `ok`.
__device__ __forceinline__ int block_partial(float v, float* red, int lane, int warp, bool ok) {
    v = group_sum<32>(v);
    if (lane == 0) red[warp] = v;
    return __syncthreads_and(ok ? 1 : 0);
}

// Second half: the warp totals added in warp order (same bits in every thread).
__device__ __forceinline__ float block_total(const float* red, int nw) {
    float t = red[0];
    for (int i = 1; i < nw; ++i) t = fadd(t, red[i]);
    return t;
}

// On a timed-out wait: thread 0 waits (bounded) for every copy it still has in
// flight so that no TMA write lands after the CTA exits, then raises the flag.
__device__ void drain_and_flag(uint64_t* mbar, int S, int64_t k, int64_t n_issued) {
    for (int64_t j = k; j < n_issued; ++j) (void)mbar_wait(&mbar[j % S], (uint32_t)((j / S) & 1));
    atomicOr(&g_wide_error, kErrWaitTimeout);
}

}  // namespace

// ---------------------------------------------------------------------------
// Forward: plain / zero-centred, residual (adds the copy), gated (reads z).
// ---------------------------------------------------------------------------
template <int VPT, int MODE, int MAXT>
__global__ void __launch_bounds__(MAXT) wide_fwd_kernel(const FwdArgs a, const int S) {
    constexpr int NIN = (MODE == kGated) ? 2 : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    const int D = a.D;
    const int NV = D >> 3;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int64_t T = a.T;
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const uint32_t row_bytes = static_cast<uint32_t>(D) * 2u;
    const uint32_t stage_bytes = NIN * row_bytes;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
    float* red = reinterpret_cast<float*>(mbar + S);  // [2][32]

    const int64_t n_my = (cta < T) ? (T - 1 - cta) / G + 1 : 0;  // rows cta, cta+G, ...

    float we[VPT][8];
    load_weights<VPT>(a.w, a.zc, NV, nt, tid, we);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&mbar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    auto issue = [&](int64_t k) {
        const int s = static_cast<int>(k % S);
        const int64_t row = cta + k * G;
        unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
        mbar_arrive_expect_tx(&mbar[s], stage_bytes);
        bulk_g2s(st, a.x + row * a.ldx, row_bytes, &mbar[s], pol);
        if (MODE == kGated) bulk_g2s(st + row_bytes, a.z + row * a.ldz, row_bytes, &mbar[s], pol);
    };
    int64_t n_issued = 0;
    if (tid == 0) {
        n_issued = n_my < S ? n_my : S;
        for (int64_t k = 0; k < n_issued; ++k) issue(k);
    }

    for (int64_t k = 0; k < n_my; ++k) {
        const int s = static_cast<int>(k % S);
        const bool ok = mbar_wait(&mbar[s], static_cast<uint32_t>((k / S) & 1));
        const unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;

        uint4 xv[VPT];
        uint4 zv[VPT];
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = j * nt + tid;
            if (v < NV) {
                xv[j] = ld_shared_v4(st + 16 * v);
                if (MODE == kGated) zv[j] = ld_shared_v4(st + row_bytes + 16 * v);
                float f[8];
                unpack8(xv[j], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fadd(ss, fmul(f[e], f[e]));
            }
        }
        float* rb = red + ((k & 1) << 5);
        if (!block_partial(ss, rb, lane, warp, ok)) {
            if (tid == 0) drain_and_flag(mbar, S, k, n_issued);
            return;
        }
        // Every thread has read stage s: refill it with the row S ahead.
        if (tid == 0 && k + S < n_my) {
            fence_proxy_async_smem();
            issue(k + S);
            n_issued = k + S + 1;
        }
        const float tot = block_total(rb, nw);
        const float r = rsqrtf(fadd(__fdiv_rn(tot, static_cast<float>(D)), a.eps));
        const int64_t row = cta + k * G;
        if (tid == 0) a.rstd[row] = r;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = j * nt + tid;
            if (v < NV) {
                float f[8], o[8];
                unpack8(xv[j], f);
                if (MODE == kGated) {
                    float zf[8];
                    unpack8(zv[j], zf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float q = fmul(zf[e], sigmoidf_rn(zf[e]));
                        o[e] = fmul(fmul(fmul(f[e], r), we[j][e]), q);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = fmul(fmul(f[e], r), we[j][e]);
                }
                st_global_cs(a.y + row * a.ldy + 8 * v, pack8(o));
                if (MODE == kResidual) st_global_cs(a.xc + row * a.ldxc + 8 * v, xv[j]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Backward pass 1: dx (and dz), plus one weight-gradient partial per chunk.
// Stage layout: [g row][x row][g_res or z row]; the row's rstd arrives in the
// same stage through a 4-byte cp.async whose completion is a no-increment
// arrive on the stage's mbarrier (expected count 2).
// ---------------------------------------------------------------------------
template <int VPT, int MODE, int MAXT>
__global__ void __launch_bounds__(MAXT) wide_bwd_kernel(const BwdArgs a, const int S) {
    constexpr int NIN = (MODE == kPlain) ? 2 : 3;
    constexpr int C = kWideChunkRows;
    extern __shared__ __align__(128) unsigned char smem[];
    const int D = a.D;
    const int NV = D >> 3;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int64_t T = a.T;
    const int64_t G = gridDim.x;
    const int64_t cta = blockIdx.x;
    const int64_t nchunks = (T + C - 1) / C;
    const uint32_t row_bytes = static_cast<uint32_t>(D) * 2u;
    const uint32_t stage_bytes = NIN * row_bytes;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * stage_bytes);
    float* rs = reinterpret_cast<float*>(mbar + S);  // [S]
    float* red = rs + S;                             // [2][32]

    // This CTA's chunks: cta, cta+G, ...; only the globally last chunk can be
    // short, and if this CTA owns it, it is its last one.
    int64_t n_my = 0;
    if (cta < nchunks) {
        const int64_t cnt = (nchunks - 1 - cta) / G + 1;
        const int64_t last = cta + (cnt - 1) * G;
        const int64_t last_rows = (T - last * C) < C ? (T - last * C) : C;
        n_my = (cnt - 1) * C + last_rows;
    }
    auto row_of = [&](int64_t k) -> int64_t { return (cta + (k / C) * G) * C + (k % C); };

    float we[VPT][8];
    load_weights<VPT>(a.w, a.zc, NV, nt, tid, we);
    float acc[VPT][8];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&mbar[s], 2);
        fence_mbar_init();
    }
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    const uint16_t* third = (MODE == kResidual) ? a.gres : a.z;
    const int64_t ld_third = (MODE == kResidual) ? a.ldgr : a.ldz;
    auto issue = [&](int64_t k) {
        const int s = static_cast<int>(k % S);
        const int64_t row = row_of(k);
        unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
        mbar_arrive_expect_tx(&mbar[s], stage_bytes);
        cp_async4_arrive(&rs[s], a.rstd + row, &mbar[s]);
        bulk_g2s(st, a.g + row * a.ldg, row_bytes, &mbar[s], pol);
        bulk_g2s(st + row_bytes, a.x + row * a.ldx, row_bytes, &mbar[s], pol);
        if (MODE != kPlain) bulk_g2s(st + 2 * row_bytes, third + row * ld_third, row_bytes, &mbar[s], pol);
    };
    int64_t n_issued = 0;
    if (tid == 0) {
        n_issued = n_my < S ? n_my : S;
        for (int64_t k = 0; k < n_issued; ++k) issue(k);
    }

    for (int64_t k = 0; k < n_my; ++k) {
        const int s = static_cast<int>(k % S);
        const bool ok = mbar_wait(&mbar[s], static_cast<uint32_t>((k / S) & 1));
        const unsigned char* st = smem + static_cast<size_t>(s) * stage_bytes;
        const float r = rs[s];

        uint4 gv[VPT], xv[VPT], tv[VPT];
        float sig[VPT][8];  // gated: sigmoid(z)
        float sp = 0.0f;    // this thread's part of s = sum g x w_eff (gated: g q x w_eff)
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = j * nt + tid;
            if (v < NV) {
                gv[j] = ld_shared_v4(st + 16 * v);
                xv[j] = ld_shared_v4(st + row_bytes + 16 * v);
                if (MODE != kPlain) tv[j] = ld_shared_v4(st + 2 * row_bytes + 16 * v);
                float gf[8], xf[8];
                unpack8(gv[j], gf);
                unpack8(xv[j], xf);
                if (MODE == kGated) {
                    float zf[8];
                    unpack8(tv[j], zf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        sig[j][e] = sigmoidf_rn(zf[e]);
                        gf[e] = fmul(gf[e], fmul(zf[e], sig[j][e]));  // g * silu(z)
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) sp = fadd(sp, fmul(fmul(gf[e], we[j][e]), xf[e]));
            }
        }
        float* rb = red + ((k & 1) << 5);
        if (!block_partial(sp, rb, lane, warp, ok)) {
            if (tid == 0) drain_and_flag(mbar, S, k, n_issued);
            return;
        }
        if (tid == 0 && k + S < n_my) {
            fence_proxy_async_smem();
            issue(k + S);
            n_issued = k + S + 1;
        }
        const float s_tot = block_total(rb, nw);
        const float coef = fmul(__fdiv_rn(fmul(fmul(r, r), r), static_cast<float>(D)), s_tot);
        const int64_t row = row_of(k);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = j * nt + tid;
            if (v < NV) {
                float gf[8], xf[8], o[8];
                unpack8(gv[j], gf);
                unpack8(xv[j], xf);
                if (MODE == kGated) {
                    float zf[8], dzv[8];
                    unpack8(tv[j], zf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float u = fmul(fmul(xf[e], r), we[j][e]);
                        const float dsilu = fmul(sig[j][e], fadd(1.0f, fmul(zf[e], fsub(1.0f, sig[j][e]))));
                        dzv[e] = fmul(fmul(gf[e], u), dsilu);
                        gf[e] = fmul(gf[e], fmul(zf[e], sig[j][e]));  // g * silu(z)
                    }
                    st_global_cs(a.dz + row * a.lddz + 8 * v, pack8(dzv));
                }
                float gr[8];
                if (MODE == kResidual) unpack8(tv[j], gr);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float d = fsub(fmul(fmul(gf[e], we[j][e]), r), fmul(xf[e], coef));
                    if (MODE == kResidual) d = fadd(d, gr[e]);
                    o[e] = d;
                    acc[j][e] = fadd(acc[j][e], fmul(fmul(gf[e], xf[e]), r));
                }
                st_global_cs(a.dx + row * a.lddx + 8 * v, pack8(o));
            }
        }
        // End of a chunk: write its partial row and restart the accumulators.
        if ((k % C) == C - 1 || k == n_my - 1) {
            const int64_t chunk = cta + (k / C) * G;
            float4* prow = reinterpret_cast<float4*>(a.partials + chunk * D);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = j * nt + tid;
                if (v < NV) {
                    prow[2 * v] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
                    prow[2 * v + 1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[j][e] = 0.0f;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
namespace {

inline int stages_for(size_t budget, size_t stage_bytes) {
    size_t s = budget / stage_bytes;
    if (s < 2) s = 2;
    if (s > RMSN_MAX_STAGES) s = RMSN_MAX_STAGES;
    return static_cast<int>(s);
}

template <int VPT, int MODE, int MAXT>
cudaError_t fwd_t(const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    constexpr int NIN = (MODE == kGated) ? 2 : 1;
    const size_t stage = static_cast<size_t>(NIN) * a.D * 2;
    const int S = stages_for(RMSN_WIDE_FWD_SMEM, stage);
    const int smem = static_cast<int>(S * stage + S * 8 + 2 * 32 * 4);
    const void* kern = reinterpret_cast<const void*>(wide_fwd_kernel<VPT, MODE, MAXT>);
    cudaError_t e = ensure_smem_attr(kern, smem);
    if (e != cudaSuccess) return e;
    const int occ = std::min(ctas_per_sm(kern, c.threads, smem), RMSN_WIDE_FWD_CTAS_PER_SM);
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int64_t grid = std::min<int64_t>(a.T, static_cast<int64_t>(sm_count()) * occ);
    wide_fwd_kernel<VPT, MODE, MAXT><<<static_cast<unsigned>(grid), c.threads, smem, st>>>(a, S);
    return cudaGetLastError();
}

template <int VPT, int MODE, int MAXT>
cudaError_t bwd_t(const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    constexpr int NIN = (MODE == kPlain) ? 2 : 3;
    const size_t stage = static_cast<size_t>(NIN) * a.D * 2;
    const int S = stages_for(RMSN_WIDE_BWD_SMEM, stage);
    const int smem = static_cast<int>(S * stage + S * 8 + S * 4 + 2 * 32 * 4);
    const void* kern = reinterpret_cast<const void*>(wide_bwd_kernel<VPT, MODE, MAXT>);
    cudaError_t e = ensure_smem_attr(kern, smem);
    if (e != cudaSuccess) return e;
    const int occ = std::min(ctas_per_sm(kern, c.threads, smem), RMSN_WIDE_BWD_CTAS_PER_SM);
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int64_t nchunks = (a.T + kWideChunkRows - 1) / kWideChunkRows;
    const int64_t grid = std::min<int64_t>(nchunks, static_cast<int64_t>(sm_count()) * occ);
    wide_bwd_kernel<VPT, MODE, MAXT><<<static_cast<unsigned>(grid), c.threads, smem, st>>>(a, S);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t fwd_dispatch(const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    if (c.threads > 256) return fwd_t<4, MODE, 512>(a, c, st);
    switch (c.vpt) {
        case 1: return fwd_t<1, MODE, 256>(a, c, st);
        case 2: return fwd_t<2, MODE, 256>(a, c, st);
        case 4: return fwd_t<4, MODE, 256>(a, c, st);
        default: return cudaErrorInvalidValue;
    }
}

template <int MODE>
cudaError_t bwd_dispatch(const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    if (c.threads > 256) return bwd_t<4, MODE, 512>(a, c, st);
    switch (c.vpt) {
        case 1: return bwd_t<1, MODE, 256>(a, c, st);
        case 2: return bwd_t<2, MODE, 256>(a, c, st);
        case 4: return bwd_t<4, MODE, 256>(a, c, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_wide_fwd(Mode m, const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    switch (m) {
        case kPlain: return fwd_dispatch<kPlain>(a, c, st);
        case kResidual: return fwd_dispatch<kResidual>(a, c, st);
        case kGated: return fwd_dispatch<kGated>(a, c, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_wide_bwd(Mode m, const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    switch (m) {
        case kPlain: return bwd_dispatch<kPlain>(a, c, st);
        case kResidual: return bwd_dispatch<kResidual>(a, c, st);
        case kGated: return bwd_dispatch<kGated>(a, c, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
