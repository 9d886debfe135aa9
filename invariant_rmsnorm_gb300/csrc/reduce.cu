// Weight-gradient pass 2: dgamma[j] = sum over chunks c of partials[c][j].
//
// Fixed order, no atomics (RL-Kernel pull request 414 "[DSv4][P1-5]
// rmsnorm_residual", Implementation: ascending fp32 reductions, no atomic
// reductions / Split-K / Stream-K). For every column the chunk axis is cut into
// kReduceWarps contiguous ranges of ceil(n / kReduceWarps) chunks; warp w adds
// range w in ascending order, then the warp totals are added in warp order.
// The tree depends only on the number of chunks (a function of T and D) and on
// compile-time constants, so the result is bitwise reproducible on any GPU.
// How many columns a lane carries (1 or 4, chosen from D for parallelism)
// does not change the tree.
#include "common.cuh"
#include "kernels.h"

namespace rmsn {

namespace {
constexpr int kUnroll = 16;  // loads in flight per lane

template <int VEC>
struct Vec;
template <>
struct Vec<1> {
    using T = float;
    static __device__ __forceinline__ T zero() { return 0.0f; }
    static __device__ __forceinline__ T load(const float* p) { return __ldcs(p); }
    static __device__ __forceinline__ T add(T a, T b) { return fadd(a, b); }
    static __device__ __forceinline__ void store(float* p, T v) { *p = v; }
};
template <>
struct Vec<4> {
    using T = float4;
    static __device__ __forceinline__ T zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    static __device__ __forceinline__ T load(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
    static __device__ __forceinline__ T add(T a, T b) {
        return make_float4(fadd(a.x, b.x), fadd(a.y, b.y), fadd(a.z, b.z), fadd(a.w, b.w));
    }
    static __device__ __forceinline__ void store(float* p, T v) { *reinterpret_cast<float4*>(p) = v; }
};
}  // namespace

template <int VEC>
__global__ void __launch_bounds__(32 * kReduceWarps)
dgamma_reduce_kernel(const float* __restrict__ partials, int64_t nchunks, int D, float* __restrict__ out) {
    using V = Vec<VEC>;
    using T = typename V::T;
    __shared__ T tot[kReduceWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int col = (blockIdx.x * 32 + lane) * VEC;
    const int64_t per = (nchunks + kReduceWarps - 1) / kReduceWarps;
    const int64_t c0 = warp * per;
    const int64_t c1 = (c0 + per < nchunks) ? c0 + per : nchunks;
    T acc = V::zero();
    if (col < D) {
        const float* p = partials + col;
        int64_t c = c0;
        for (; c + kUnroll <= c1; c += kUnroll) {
            T v[kUnroll];
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) v[i] = V::load(p + (c + i) * D);
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) acc = V::add(acc, v[i]);
        }
        for (; c < c1; ++c) acc = V::add(acc, V::load(p + c * D));
    }
    tot[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && col < D) {
        T s = tot[0][lane];
#pragma unroll
        for (int w = 1; w < kReduceWarps; ++w) s = V::add(s, tot[w][lane]);
        V::store(out + col, s);
    }
}

cudaError_t launch_dgamma_reduce(const float* partials, int64_t nchunks, int D, float* out, cudaStream_t s) {
    if (D >= 2048) {
        const unsigned grid = static_cast<unsigned>((D + 127) / 128);
        dgamma_reduce_kernel<4><<<grid, 32 * kReduceWarps, 0, s>>>(partials, nchunks, D, out);
    } else {
        const unsigned grid = static_cast<unsigned>((D + 31) / 32);
        dgamma_reduce_kernel<1><<<grid, 32 * kReduceWarps, 0, s>>>(partials, nchunks, D, out);
    }
    return cudaGetLastError();
}

}  // namespace rmsn
