// Weight-gradient pass 2: dgamma[j] = sum over chunks c of partials[c][j].
//
// Fixed order, no atomics (RL-Kernel pull request 414 "[DSv4][P1-5]
// rmsnorm_residual", Implementation: ascending fp32 reductions, no atomic
// reductions / Split-K / Stream-K). For every column the chunk axis is cut
// into kReduceWarps contiguous ranges of ceil(n / kReduceWarps) chunks; each
// range is added in ascending order, then the range totals in range order.
// The tree depends only on the number of chunks (a function of T and D) and
// on compile-time constants, so the result is bitwise reproducible on any GPU.
//
// A CTA owns CW adjacent columns (CW = 32, 16 or 8) and all the ranges of
// them: thread (range w, column k) adds range w of column k, and the CTA's
// first CW threads add the range totals. CW changes only which thread does
// which range, never the tree, so every CW gives the same bits; narrower CTAs
// spread small D over more SMs (D = 128: 16 CTAs instead of 4). Every thread
// keeps kUnroll independent loads in flight.
#include "common.cuh"
#include "kernels.h"

namespace rmsn {

namespace {
#ifndef RMSN_REDUCE_UNROLL
#define RMSN_REDUCE_UNROLL 32
#endif
constexpr int kUnroll = RMSN_REDUCE_UNROLL;  // loads in flight per thread
}

template <int CW>
__global__ void __launch_bounds__(kReduceWarps * CW)
dgamma_reduce_kernel(const float* __restrict__ partials, int64_t nchunks, int D, float* __restrict__ out) {
    __shared__ float tot[kReduceWarps][CW];
    pdl_wait();
    const int k = threadIdx.x % CW, w = threadIdx.x / CW;  // column within the CTA, range
    const int col = blockIdx.x * CW + k;
    const int64_t per = (nchunks + kReduceWarps - 1) / kReduceWarps;
    const int64_t c0 = w * per;
    const int64_t c1 = (c0 + per < nchunks) ? c0 + per : nchunks;
    float acc = 0.0f;
    if (col < D) {
        const float* p = partials + col;
        int64_t c = c0;
        for (; c + kUnroll <= c1; c += kUnroll) {
            float v[kUnroll];
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) v[i] = __ldcs(p + (c + i) * D);
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) acc = fadd(acc, v[i]);
        }
        for (; c < c1; ++c) acc = fadd(acc, __ldcs(p + c * D));
    }
    pdl_release();
    tot[w][k] = acc;
    __syncthreads();
    if (w == 0 && col < D) {
        float s = tot[0][k];
#pragma unroll
        for (int r = 1; r < kReduceWarps; ++r) s = fadd(s, tot[r][k]);
        out[col] = s;
    }
}

// Columns per CTA: the widest of 32, 16, 8 that still gives at least one CTA
// per SM (D is a multiple of 8).
cudaError_t launch_dgamma_reduce(const float* partials, int64_t nchunks, int D, float* out, cudaStream_t s) {
    const int sms = sm_count();
    if (D / 32 >= sms)
        return launch_kernel(dgamma_reduce_kernel<32>, static_cast<unsigned>((D + 31) / 32), 32 * kReduceWarps, 0, s,
                             partials, nchunks, D, out);
    if (D / 16 >= sms)
        return launch_kernel(dgamma_reduce_kernel<16>, static_cast<unsigned>((D + 15) / 16), 16 * kReduceWarps, 0, s,
                             partials, nchunks, D, out);
    return launch_kernel(dgamma_reduce_kernel<8>, static_cast<unsigned>((D + 7) / 8), 8 * kReduceWarps, 0, s,
                         partials, nchunks, D, out);
}

}  // namespace rmsn
