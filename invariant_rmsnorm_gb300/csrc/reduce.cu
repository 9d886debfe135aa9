// Weight-gradient pass 2: dgamma[j] = sum over chunks c of partials[c][j].
//
// Fixed order, no atomics (RL-Kernel pull request 414 "[DSv4][P1-5]
// rmsnorm_residual", Implementation: ascending fp32 reductions, no atomic
// reductions / Split-K / Stream-K). One CTA owns 32 adjacent columns, one per
// lane. For every column the chunk axis is cut into kReduceWarps contiguous
// ranges of ceil(n / kReduceWarps) chunks; warp w adds range w in ascending
// order, then lane j of warp 0 adds the warp totals in warp order. The tree
// depends only on the number of chunks (a function of T and D) and on
// compile-time constants, so the result is bitwise reproducible on any GPU.
// Every lane keeps kUnroll independent loads in flight, so the whole partial
// array is read in a few memory round trips.
#include "common.cuh"
#include "kernels.h"

namespace rmsn {

namespace {
#ifndef RMSN_REDUCE_UNROLL
#define RMSN_REDUCE_UNROLL 32
#endif
constexpr int kUnroll = RMSN_REDUCE_UNROLL;  // loads in flight per lane
}

__global__ void __launch_bounds__(32 * kReduceWarps)
dgamma_reduce_kernel(const float* __restrict__ partials, int64_t nchunks, int D, float* __restrict__ out) {
    __shared__ float tot[kReduceWarps][32];
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + lane;
    const int64_t per = (nchunks + kReduceWarps - 1) / kReduceWarps;
    const int64_t c0 = warp * per;
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
    tot[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && col < D) {
        float s = tot[0][lane];
#pragma unroll
        for (int w = 1; w < kReduceWarps; ++w) s = fadd(s, tot[w][lane]);
        out[col] = s;
    }
}

cudaError_t launch_dgamma_reduce(const float* partials, int64_t nchunks, int D, float* out, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>((D + 31) / 32);
    return launch_kernel(dgamma_reduce_kernel, grid, 32 * kReduceWarps, 0, s, partials, nchunks, D, out);
}

}  // namespace rmsn
