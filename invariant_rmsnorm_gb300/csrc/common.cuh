// Shared device-side building blocks for the sm_103a RMSNorm kernels:
// inline-PTX wrappers for mbarriers, bulk (TMA) copies and cp.async, bf16 and
// fp16 packing, separately rounded fp32 arithmetic, the gate functions, and
// the fixed butterfly sum.
//
// Every wait on an mbarrier is bounded: a waiter that sees no progress for
// kWaitTimeoutNs of global time gives up and reports failure, and the kernels
// turn that into an error flag plus a clean exit (no trap, no endless spin).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "rmsnorm.h"

namespace rmsn {

// ---------------------------------------------------------------------------
// Constants that fix the numerics. They depend on nothing but D, never on T,
// the row index, the grid or the GPU's SM count.
// ---------------------------------------------------------------------------
#ifndef RMSN_WIDE_CHUNK
#define RMSN_WIDE_CHUNK 32
#endif
constexpr int kWideChunkRows = RMSN_WIDE_CHUNK;  // weight-gradient chunk (rows), wide path
constexpr int kNarrowThreads = 256;      // narrow path CTA size
constexpr int kNarrowChunkRowsMin = 128;  // weight-gradient chunk (rows), narrow path (at least)
constexpr int kMaxD = 16384;
constexpr int kReduceWarps = 32;         // weight-gradient pass 2: warps (chunk ranges) per 32 columns

// Device-side error codes (bit flags OR-ed into the library's error words).
constexpr unsigned kErrWaitTimeout = RMSN_DEVICE_ERR_WAIT_TIMEOUT;

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel is launched with programmatic
// stream serialization allowed (launch_kernel below), so it may become
// resident while the previous kernel of its stream drains. It runs only its
// prologue (shared-memory barriers; no global memory), then waits in
// pdl_wait() until that kernel has completed and its memory is visible. Each
// CTA calls pdl_release() once its main loop is done, so the next kernel of
// the stream starts launching when every CTA is in its epilogue: its launch
// latency and prologue overlap this kernel's end, while its CTAs still land on
// SMs that are (almost) free, as in an ordinary launch. Kernels launched
// without the attribute see both as no-ops.
// ---------------------------------------------------------------------------
#ifndef RMSN_PDL
#define RMSN_PDL 1
#endif

__device__ __forceinline__ void pdl_wait() {
#if RMSN_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

__device__ __forceinline__ void pdl_release() {
#if RMSN_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Launch `kern` on `st` (programmatic stream serialization allowed when
// RMSN_PDL is set), in thread-block clusters of `cluster` consecutive CTAs
// when `cluster` > 1 (`grid` a multiple of it). Returns the launch's error.
template <typename... Params, typename... Args>
cudaError_t launch_kernel_clustered(void (*kern)(Params...), unsigned cluster, unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (RMSN_PDL) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kern)(Params...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                          Args&&... args) {
    return launch_kernel_clustered(kern, 1u, grid, block, smem, st, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order earlier generic-proxy shared-memory accesses (made visible to this
// thread by a barrier) before its later async-proxy (TMA) writes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Plain arrive (release) on `bar`.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Named barrier `id` over `nthreads` threads (a multiple of 32) that also
// returns the AND of every participant's predicate.
__device__ __forceinline__ int named_bar_and(int id, int nthreads, int pred) {
    int res;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(res) : "r"(pred), "r"(id), "r"(nthreads) : "memory");
    return res;
}

// Thread-block clusters: this CTA's rank in its cluster, the cluster's index
// along x and the number of clusters along x.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// The shared::cluster address of the location `p` (in this CTA's shared
// memory) has in the CTA of rank `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Store 4 bytes into another CTA's shared memory (both addresses from
// cluster_map, in that CTA); its mbarrier counts them as transaction bytes.
__device__ __forceinline__ void st_async_f32(uint32_t remote_dst, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 ::"r"(remote_dst), "r"(__float_as_uint(v)), "r"(remote_bar) : "memory");
}

// Every thread of every CTA of the cluster (release, then acquire). A CTA pair
// meets there twice: after the shared-memory barriers are initialised, before
// either CTA touches the other's shared memory, and at the end, before either
// exits while the other may still store into it.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bounded wait for the phase with parity `parity` to complete, with an acquire
// at CTA scope, or with kCluster at cluster scope (for a phase completed by
// another CTA of the cluster, st_async_f32, whose data is then read here).
// Returns false if `limit_ns` of global time elapsed without completion.
template <bool kCluster>
__device__ __forceinline__ bool mbar_wait_scoped(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    const uint32_t addr = smem_u32(bar);
    uint32_t done = 0;
    unsigned long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if constexpr (kCluster)
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(done) : "r"(addr), "r"(parity) : "memory");
        else
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(done) : "r"(addr), "r"(parity) : "memory");
        if (done) return true;
        if ((it & 255u) == 0u) {
            const unsigned long long now = global_timer_ns();
            if (it == 0) t0 = now;
            else if (now - t0 > limit_ns) return false;
        }
    }
}

// The kernels' waits: kWaitTimeoutNs unless a test gives another limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitTimeoutNs) {
    return mbar_wait_scoped<false>(bar, parity, limit_ns);
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
    return mbar_wait_scoped<true>(bar, parity, kWaitTimeoutNs);
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
// dst and src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// 2-D tiled tensor copy global -> shared (box described by the tensor map).
// c0 = innermost (column) coordinate, c1 = row coordinate.
__device__ __forceinline__ void tensor2d_g2s(void* dst, const CUtensorMap* map, int c0, int c1,
                                             uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// 1-D tiled tensor copy global -> shared.
__device__ __forceinline__ void tensor1d_g2s(void* dst, const CUtensorMap* map, int c0, uint64_t* bar,
                                             uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2}], [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 4-byte asynchronous copy global -> shared (cp.async, L1-allocating).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// One arrive on `bar`, triggered once all of this thread's earlier cp.async
// copies have landed; no-increment, so the barrier's expected count includes it.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// L2 policy for streamed data read once.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy of ordinary priority (explicitly).
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy for data written now and read back soon (kept resident in L2).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 128-bit global store of four floats with an L2 cache policy.
__device__ __forceinline__ void st_global_f4_hint(float* p, float a, float b, float c, float d, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;"
                 ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d), "l"(pol) : "memory");
}

// 32-bit global store with an L2 cache policy.
__device__ __forceinline__ void st_global_f1_hint(float* p, float a, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(a), "l"(pol) : "memory");
}

// 128-bit streaming global store.
__device__ __forceinline__ void st_global_cs(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)) : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// bf16 <-> fp32 (exact widening; round-to-nearest-even narrowing)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void unpack8(const uint4 v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);  // .x = low half
        w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// fp16 <-> fp32: exact widening; round-to-nearest-even narrowing (subnormals
// kept, overflow to infinity).
__device__ __forceinline__ void unpack8_f16(const uint4 v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));  // .x = low half
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8_f16(const float f[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Eight activations of the kernel's storage format (fp16 if F16, else bf16).
template <bool F16>
__device__ __forceinline__ void unpack_act(const uint4 v, float f[8]) {
    if constexpr (F16) unpack8_f16(v, f);
    else unpack8(v, f);
}
template <bool F16>
__device__ __forceinline__ uint4 pack_act(const float f[8]) {
    if constexpr (F16) return pack8_f16(f);
    else return pack8(f);
}

// An fp32 value rounded to bf16 (nearest even) and widened back.
__device__ __forceinline__ float round_bf16f(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// ---------------------------------------------------------------------------
// Separately rounded fp32 arithmetic (never contracted into FMA).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }

// Two independent fp32 operations at once, through the packed instructions
// `mul.rn.f32x2` / `add.rn.f32x2` (sm_100 and later): each half is an IEEE
// fp32 operation rounded to nearest even, without flushing subnormals, so
// fmul2(a, b) is bit for bit {fmul(a.x, b.x), fmul(a.y, b.y)} at half the
// instruction count (checked on 2^24 random pairs of every class).
// One rule keeps every multiply and add separately rounded: ptxas contracts a
// packed multiply whose result feeds a packed add or subtract into one fused
// multiply-add, even under -fmad=false (measured: about 6 % of such chains
// round differently). So a sum or difference that takes a product is always
// computed with the scalar fadd/fsub, whose explicit rounding ptxas keeps;
// fadd2 only ever adds values that are not products. With RMSN_F32X2 = 0 both
// are the scalar pairs.
#ifndef RMSN_F32X2
#define RMSN_F32X2 1
#endif
#if RMSN_F32X2
#define RMSN_DEFINE_OP2(name, op)                                                             \
    __device__ __forceinline__ float2 name(float2 a, float2 b) {                              \
        float2 d;                                                                             \
        asm("{\n\t.reg .b64 ra, rb, rd;\n\t"                                                  \
            "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t" op                           \
            " rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"                                      \
            : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                 \
        return d;                                                                             \
    }
RMSN_DEFINE_OP2(fmul2, "mul.rn.f32x2")
RMSN_DEFINE_OP2(fadd2, "add.rn.f32x2")
#undef RMSN_DEFINE_OP2
#else
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return make_float2(fmul(a.x, b.x), fmul(a.y, b.y)); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return make_float2(fadd(a.x, b.x), fadd(a.y, b.y)); }
#endif
// Elements e and e+1 of an fp32 array as a pair, and a value twice.
__device__ __forceinline__ float2 pair(const float* v, int e) { return make_float2(v[e], v[e + 1]); }
__device__ __forceinline__ float2 both(float v) { return make_float2(v, v); }

// e^-a for a >= 0, from the PTX instruction ex2.approx.ftz.f32 (2^x, which
// flushes subnormal results to zero), as the square of a half-way power:
// h = 2^(-a log2(e) / 2), e^-a = h * h. h stays a normal number for every a
// up to about 174, so the flush never bites where e^-a is still an fp32
// value (down to the smallest subnormal, reached at a of about 103): the
// square, an ordinary multiply that keeps subnormals, rounds those tails.
// Relative error about (5 + a) * 2^-24: twice the instruction's error plus the
// rounding of the exponent, doubled by the square, plus the square's rounding.
#ifndef RMSN_FAST_EXP
#define RMSN_FAST_EXP 1
#endif
__device__ __forceinline__ float exp_neg(float a) {
#if RMSN_FAST_EXP
    float h;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(h) : "f"(fmul(a, -0.72134752044448170f)));
    return fmul(h, h);
#else
    return __expf(-a);
#endif
}

// 1 / d for d in [1, 2] (never subnormal, so flushing changes nothing), from
// the PTX instruction rcp.approx.ftz.f32 (error <= 1 ulp).
__device__ __forceinline__ float rcp_1to2(float d) {
#if RMSN_FAST_EXP
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
#else
    return __fdividef(1.0f, d);
#endif
}

// sigmoid(z) = 1 / (1 + exp(-z)) in fp32, in the stable two-sided form: with
// e = exp(-|z|) in (0, 1] and s = 1 / (1 + e), sigmoid is s for z >= 0 and
// e * s (= e^z / (1 + e^z)) for z < 0, so the divisor stays in [1, 2]. A
// relative error of about (8 + |z|) * 2^-24 on sigmoid, for every finite z.
__device__ __forceinline__ float sigmoidf_rn(float z) {
    const float e = exp_neg(fabsf(z));
    const float s = rcp_1to2(fadd(1.0f, e));
    return z >= 0.0f ? s : fmul(e, s);
}

// The gate q(z) of the gated norm and its derivative, from one exponential.
// With e, s as in sigmoidf_rn, both sigmoid(z) and sigmoid(-z) = 1 - sigmoid(z)
// come without a subtraction: one is s, the other e * s.
//   silu:    q = z sigmoid(z),  q' = sigmoid(z) + q sigmoid(-z)
//   sigmoid: q = sigmoid(z),    q' = sigmoid(z) sigmoid(-z) = (e s) s
// (q is bit for bit gate_value's; neither form cancels in a tail, where
// 1 - sigmoid(z) would lose every bit for z >> 0).
template <bool SIG>
__device__ __forceinline__ float gate_value(float z) {
    return SIG ? sigmoidf_rn(z) : fmul(z, sigmoidf_rn(z));
}
template <bool SIG>
__device__ __forceinline__ void gate_eval(float z, float& q, float& dq) {
    const float e = exp_neg(fabsf(z));
    const float s = rcp_1to2(fadd(1.0f, e));
    const float es = fmul(e, s);
    const bool pos = z >= 0.0f;
    const float sg = pos ? s : es;  // sigmoid(z)
    if (SIG) {
        q = sg;
        dq = fmul(es, s);
    } else {
        q = fmul(z, sg);
        dq = fadd(sg, fmul(q, pos ? es : s));
    }
}

// x / D, correctly rounded. When D is a power of two the host passes its exact
// reciprocal `inv_pow2` and the quotient is that single exact scaling (same
// bits as the division); otherwise inv_pow2 is 0 and an IEEE division runs.
__device__ __forceinline__ float div_by_d(float x, int D, float inv_pow2) {
    return inv_pow2 != 0.0f ? fmul(x, inv_pow2) : __fdiv_rn(x, static_cast<float>(D));
}

// Butterfly sum over aligned groups of WIDTH lanes (a power of two <= 32).
// Every lane of a group ends with the same bits (IEEE addition commutes).
template <int WIDTH>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) v = fadd(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace rmsn
