// C-ABI layer: argument validation, row-shape selection, device caches and
// dispatch to the kernel launchers. Every check runs on the host before any
// launch; there is no fallback path.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace rmsn {

// ---------------------------------------------------------------------------
// Row shape: a pure function of D (this is what makes a row's reduction tree,
// and therefore its bits, independent of everything but D; run_bwd adjusts the
// backward's shape by the variant, which a call fixes).
// ---------------------------------------------------------------------------
#ifndef RMSN_FWD_NTMAX
#define RMSN_FWD_NTMAX 256
#endif
#ifndef RMSN_BWD_PAIR_PLAIN_UPTO
#define RMSN_BWD_PAIR_PLAIN_UPTO 1152  // plain backward rows of 1025..this many vectors on CTA pairs
#endif
#ifndef RMSN_BWD_NTMAX
#define RMSN_BWD_NTMAX 256
#endif
#ifndef RMSN_BWD_NT128_UPTO
#define RMSN_BWD_NT128_UPTO 256  // plain backward rows of at most this many 16-byte vectors (D <= 2048): <= 128 threads
#endif
#ifndef RMSN_BWD_NT512_FROM
#define RMSN_BWD_NT512_FROM 897  // backward rows of 897..1024 vectors (7168 < D <= 8192): 512 threads, 2 vectors each
#endif

// Threads and 16-byte vectors per thread for one row of NV vectors: at most
// `ntmax` threads (512 beyond 1024 vectors), VPT in {1, 2, 4}, threads rounded
// up to whole warps; slots past the row end are idle.
static void wide_shape(int NV, int ntmax, int* threads, int* vpt) {
    if (NV > 4 * ntmax) ntmax = 512;
    const int need = (NV + ntmax - 1) / ntmax;
    *vpt = need <= 1 ? 1 : (need <= 2 ? 2 : 4);
    *threads = ((NV + *vpt - 1) / *vpt + 31) / 32 * 32;
}

RowCfg row_cfg(int D) {
    RowCfg c{};
    const int NV = D / 8;  // 16-byte vectors per row
    if (NV <= 32) {
        // Narrow rows: one group of G lanes (a power of two) per row.
        int G = 1;
        while (G < NV) G *= 2;
        c.narrow = true;
        c.threads = c.bwd_threads = kNarrowThreads;
        c.vpt = c.bwd_vpt = 1;
        c.group = G;
        c.rows_per_stage = narrow_stage_rows_for_group(G);
        c.chunk_rows = narrow_chunk_rows_for_group(G);
        return c;
    }
    c.narrow = false;
    wide_shape(NV, RMSN_FWD_NTMAX, &c.threads, &c.vpt);
    wide_shape(NV, RMSN_BWD_NTMAX, &c.bwd_threads, &c.bwd_vpt);
    c.group = 0;
    c.rows_per_stage = 1;
    c.chunk_rows = kWideChunkRows;
    return c;
}

// The wide backward's weight-gradient chunk. A CTA owns whole chunks, so with
// 32-row chunks the last round of a persistent grid can leave many CTAs idle
// (T=32768, D=4096: 1024 chunks over 304 CTAs, 112 of them with a fourth).
// For 2048 < D <= 7168, where the backward runs 2 CTAs per SM whatever the
// mode, a chunk count that fills less than 90 % of its rounds of
// kBalanceSms x 2 CTAs is evened out by shortening the chunk just enough that
// the chunks come in whole rounds (T=32768, D=4096: 27 rows, 1214 chunks,
// pass 1 166 -> 160 us). kBalanceSms is a constant, not the GPU's SM count:
// the chunk, and so dgamma's bits, depend on T and D alone. Other widths and
// well-filled rounds keep 32-row chunks (and the kernels' fixed-chunk code).
constexpr int64_t kBalanceSms = 152;

int64_t wide_chunk_rows(int64_t T, int D) {
    constexpr int64_t c0 = kWideChunkRows;
    if (D <= 2048 || D > 7168 || T <= 0) return c0;
    const int64_t ctas = kBalanceSms * 2;
    const int64_t n0 = (T + c0 - 1) / c0;
    if (n0 <= ctas) return c0;
    const int64_t rounds = (n0 + ctas - 1) / ctas;
    if (10 * n0 >= 9 * rounds * ctas) return c0;
    return (T + rounds * ctas - 1) / (rounds * ctas);  // < 32
}

// The largest number of wide-path chunks over every row count 1..T_max, in
// closed form (a loop over at most nine rounds). Chunks are shortened only in
// rounds R = 2..9 of the nominal grid (from ten rounds on, 32-row chunks fill
// over 90 % of their rounds), and there a row count t gets
// c = ceil(t / (R K)) rows a chunk (K = 2 kBalanceSms) and ceil(t / c) <= R K
// chunks, with exactly R K whenever t is a multiple of R K. So over the
// shortened row counts of round R up to T_max (t_lo..t_top), the largest
// count is R K if a multiple of R K lies in that range, and otherwise
// ceil(t_top / c), since c is then the same for all of them and ceil(t / c)
// grows with t. Every other row count has 32-row chunks, at most as many as
// T_max has with 32-row chunks.
int64_t wide_chunks_max(int64_t T_max, int D) {
    constexpr int64_t c0 = kWideChunkRows;
    if (T_max <= 0) return 0;
    int64_t best = (T_max + wide_chunk_rows(T_max, D) - 1) / wide_chunk_rows(T_max, D);
    best = std::max(best, (T_max + c0 - 1) / c0);
    if (D <= 2048 || D > 7168) return best;
    const int64_t K = kBalanceSms * 2;
    for (int64_t R = 2; R <= 9; ++R) {
        const int64_t t_lo = c0 * (R - 1) * K + 1;     // first row count of round R
        const int64_t n_hi = (9 * R * K - 1) / 10;     // most 32-row chunks still under 90 % of R K
        const int64_t t_top = std::min(T_max, c0 * n_hi);
        if (t_top < t_lo) break;
        const int64_t c_top = (t_top + R * K - 1) / (R * K);
        if ((c_top - 1) * R * K >= t_lo) best = std::max(best, R * K);  // a multiple of R K in range
        else best = std::max(best, (t_top + c_top - 1) / c_top);
    }
    return best;
}

int64_t num_chunks(int64_t T, int D) {
    const int64_t c = row_cfg(D).narrow ? row_cfg(D).chunk_rows : wide_chunk_rows(T, D);
    return (T + c - 1) / c;
}

// ---------------------------------------------------------------------------
// Per-device caches
// ---------------------------------------------------------------------------
namespace {
std::mutex g_mu;
std::map<int, int> g_sms;
std::map<std::tuple<int, unsigned long long, const void*>, int> g_smem_set;
std::map<std::tuple<int, const void*, int, int>, int> g_occ;
std::map<std::tuple<int, const void*, int, int>, int> g_pairs;

int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d;
}
}  // namespace

// The current context's unique id, through the driver entry points (the
// library does not link libcuda); false if there is no current context yet or
// the driver does not provide them. A context destroyed and created again
// (cudaDeviceReset) gets a new id, so state kept per context can tell.
bool current_context_id(unsigned long long* id) {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return false;
    return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

int sm_count() {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sms.find(dev);
    if (it != g_sms.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    g_sms[dev] = n;
    return n;
}

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    const int dev = current_device();
    // The attribute belongs to the function in the current context: keyed on
    // the context too, so that it is set again after a device reset (without a
    // context id it is set on every call).
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    if (!have_ctx) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(dev, ctx, kernel);
    auto it = g_smem_set.find(key);
    if (it != g_smem_set.end() && it->second >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_smem_set[key] = bytes;
    return e;
}

int ctas_per_sm(const void* kernel, int threads, int smem_bytes) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(dev, kernel, threads, smem_bytes);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem_bytes) != cudaSuccess) n = 0;
    g_occ[key] = n;
    return n;
}

int pair_clusters(const void* kernel, int threads, int smem_bytes) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(dev, kernel, threads, smem_bytes);
    auto it = g_pairs.find(key);
    if (it != g_pairs.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
    g_pairs[key] = n;
    return n;
}

}  // namespace rmsn

using namespace rmsn;

// ---------------------------------------------------------------------------
// Validation helpers
// ---------------------------------------------------------------------------
namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int64_t T, int64_t D) {
    if (T < 0 || T >= (int64_t(1) << 31)) return RMSN_EINVAL;
    if (D < 8 || D > kMaxD || (D % 8) != 0) return RMSN_EUNSUPPORTED;
    return RMSN_OK;
}

// An activation matrix [T][ld] of bf16 (required = must be non-null).
int check_act(const void* p, int64_t ld, int64_t D) {
    if (p == nullptr) return RMSN_EINVAL;
    if (ld < D || ld > (int64_t(1) << 40)) return RMSN_EINVAL;
    if (!aligned16(p) || (ld % 8) != 0) return RMSN_EALIGN;
    return RMSN_OK;
}

int check_vec(const void* p) {
    if (p == nullptr) return RMSN_EINVAL;
    if (!aligned16(p)) return RMSN_EALIGN;
    return RMSN_OK;
}

int check_eps(float eps) { return (std::isfinite(eps) && eps >= 0.0f) ? RMSN_OK : RMSN_EINVAL; }

int check_ws(const void* ws, size_t ws_bytes, int64_t T, int64_t D) {
    const size_t need = static_cast<size_t>(num_chunks(T, static_cast<int>(D))) * static_cast<size_t>(D) * 4u;
    if (ws == nullptr || ws_bytes < need) return RMSN_EWORKSPACE;
    if (!aligned16(ws)) return RMSN_EALIGN;
    return RMSN_OK;
}

#define RMSN_TRY(expr)                  \
    do {                                \
        const int _st = (expr);         \
        if (_st != RMSN_OK) return _st; \
    } while (0)

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? RMSN_OK : RMSN_ECUDA; }

float inv_pow2(int D) { return (D & (D - 1)) == 0 ? 1.0f / static_cast<float>(D) : 0.0f; }

// Variant flags of an activation dtype / gate argument (RMSN_EINVAL if unknown).
int dtype_flags(int dtype, int* flags) {
    if (dtype == RMSN_DTYPE_BF16) { *flags = 0; return RMSN_OK; }
    if (dtype == RMSN_DTYPE_F16) { *flags = kFlagF16; return RMSN_OK; }
    return RMSN_EINVAL;
}

int gate_flags(int gate, int* flags) {
    if (gate == RMSN_GATE_SILU) { *flags = 0; return RMSN_OK; }
    if (gate == RMSN_GATE_SIGMOID) { *flags = kFlagSigmoid; return RMSN_OK; }
    return RMSN_EINVAL;
}

// `m` = Mode | variant flags.
int run_fwd(int m, FwdArgs a, cudaStream_t s) {
    a.inv_d_pow2 = inv_pow2(a.D);
    const RowCfg c = row_cfg(a.D);
    cudaError_t e;
    if (is_f16(m)) e = c.narrow ? launch_narrow_fwd_f16(m, a, c, s) : launch_wide_fwd_f16(m, a, c, s);
    else e = c.narrow ? launch_narrow_fwd(m, a, c, s) : launch_wide_fwd(m, a, c, s);
    return cuda_status(e);
}

int run_bwd(int m, BwdArgs a, float* dgamma, cudaStream_t s) {
    a.inv_d_pow2 = inv_pow2(a.D);
    RowCfg c = row_cfg(a.D);
    if (a.chunk == 0) a.chunk = static_cast<int>(wide_chunk_rows(a.T, a.D));
    // The plain backward of rows up to 2048 values runs them on at most 128
    // threads, two vectors each (a fixed function of D for this mode; measured
    // 131072 x 2048: 291 -> 282 us). The modes streaming more operands per row
    // measured slower that way and keep the shared shape.
    if (!c.narrow && base_mode(m) == kPlain && a.D / 8 <= RMSN_BWD_NT128_UPTO)
        wide_shape(a.D / 8, 128, &c.bwd_threads, &c.bwd_vpt);
    // Rows of 7168 < D <= 8192 run on 512 threads, two vectors each, rather than
    // 256 threads with four: the four-vector kernel needs 168 registers, so a
    // single 9-warp CTA fits on an SM, where this one keeps 16 consumer warps
    // (measured 131072 x 8192: 1124 -> 1101 us, with the larger ring the
    // one-CTA-per-SM backward gets).
    if (!c.narrow && a.D / 8 >= RMSN_BWD_NT512_FROM && a.D / 8 <= 4 * RMSN_BWD_NTMAX)
        wide_shape(a.D / 8, 512, &c.bwd_threads, &c.bwd_vpt);
    // The modes that stream three or four operands take that shape from
    // 4096 < D on (two vectors on up to 512 threads, one CTA per SM) instead of
    // four vectors on 224 threads at two CTAs per SM (32768 x 7168, backward
    // with pass 2: fused add 499 -> 359 us, residual 323 -> 309, gated
    // 541 -> 529); the plain backward keeps the 224-thread kernel (232 us either
    // way). Like every launch shape here it is a function of D and the mode.
    if (!c.narrow && base_mode(m) != kPlain && a.D / 8 > 512 && a.D / 8 < RMSN_BWD_NT512_FROM)
        wide_shape(a.D / 8, 512, &c.bwd_threads, &c.bwd_vpt);
    // Rows of more than 1024 vectors (D > 8192): each row split between the two
    // CTAs of a cluster, ceil(NV/2) vectors on up to 512 threads, two vectors
    // each, in place of four vectors a thread on 512 threads (which spilled in
    // the modes that stream three or four operands). 32768 rows, backward with
    // pass 2, D=16384: residual 944 -> 738 us, gated 1926 -> 1118, fused add
    // 1570 -> 858. The plain mode takes pairs only up to 1152 vectors (D=9216:
    // 412 -> 393 us): wider, its one CTA pair per two SMs measured slower than
    // the four-vector kernel (D=16384: 622 against 665 us).
    if (!c.narrow && a.D / 8 > 4 * RMSN_BWD_NTMAX && (base_mode(m) != kPlain || a.D / 8 <= RMSN_BWD_PAIR_PLAIN_UPTO)) {
        wide_shape((a.D / 8 + 1) / 2, 512, &c.bwd_threads, &c.bwd_vpt);
        c.bwd_pair = true;
    }
    // The recompute of y is a compile-time flag of the kernels: the backward
    // without it carries no y code (nor its registers).
    const int mr = a.y != nullptr ? (m | kFlagRecompute) : m;
    cudaError_t e;
    if (is_f16(m)) e = c.narrow ? launch_narrow_bwd_f16(mr, a, c, s) : launch_wide_bwd_f16(mr, a, c, s);
    else e = c.narrow ? launch_narrow_bwd(mr, a, c, s) : launch_wide_bwd(mr, a, c, s);
    if (e != cudaSuccess) return RMSN_ECUDA;
    const int64_t nchunks = c.narrow ? num_chunks(a.T, a.D) : (a.T + a.chunk - 1) / a.chunk;
    if (dgamma != nullptr) e = launch_dgamma_reduce(a.partials, nchunks, a.D, dgamma, s);
    return cuda_status(e);
}

}  // namespace

// The backward's checks that come after the shape's and before the
// workspace's, in rmsnorm_bwd's order (T >= 1 and D already checked).
int rmsn::bwd_check_args(const uint16_t* g, int64_t ldg, const uint16_t* x, int64_t ldx, const float* w,
                         const float* rstd, const uint16_t* dx, int64_t lddx, const float* dgamma, int64_t T,
                         int64_t D) {
    (void)T;
    RMSN_TRY(check_act(g, ldg, D));
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(dx, lddx, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    if (dgamma) RMSN_TRY(check_vec(dgamma));
    return RMSN_OK;
}

// ---------------------------------------------------------------------------
// The operations, with the variant flags (activation dtype, gate) as the first
// argument; the entry points below validate those and call these.
// ---------------------------------------------------------------------------
namespace {

int rmsnorm_fwd_impl(int flags, const rmsn_act16* x, int64_t ldx, const float* w, rmsn_act16* y, int64_t ldy,
                     float* rstd, int64_t T, int64_t D, float eps, int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(y, ldy, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    RMSN_TRY(check_eps(eps));
    FwdArgs a{};
    a.x = x; a.ldx = ldx; a.w = w; a.y = y; a.ldy = ldy; a.rstd = rstd;
    a.T = T; a.D = static_cast<int>(D); a.eps = eps; a.zc = zero_centered_gamma ? 1 : 0;
    return run_fwd(kPlain | flags, a, stream);
}

int rmsnorm_residual_fwd_impl(int flags, const rmsn_act16* x, int64_t ldx, const float* w, rmsn_act16* y,
                              int64_t ldy, float* rstd, rmsn_act16* x_copy, int64_t ldxc, int64_t T, int64_t D,
                              float eps, int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(y, ldy, D));
    RMSN_TRY(check_act(x_copy, ldxc, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    RMSN_TRY(check_eps(eps));
    FwdArgs a{};
    a.x = x; a.ldx = ldx; a.w = w; a.y = y; a.ldy = ldy; a.rstd = rstd; a.xc = x_copy; a.ldxc = ldxc;
    a.T = T; a.D = static_cast<int>(D); a.eps = eps; a.zc = zero_centered_gamma ? 1 : 0;
    return run_fwd(kResidual | flags, a, stream);
}

int rmsnorm_gated_fwd_impl(int flags, const rmsn_act16* x, int64_t ldx, const rmsn_act16* z, int64_t ldz,
                           const float* w, rmsn_act16* y, int64_t ldy, float* rstd, int64_t T, int64_t D, float eps,
                           int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(z, ldz, D));
    RMSN_TRY(check_act(y, ldy, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    RMSN_TRY(check_eps(eps));
    FwdArgs a{};
    a.x = x; a.ldx = ldx; a.z = z; a.ldz = ldz; a.w = w; a.y = y; a.ldy = ldy; a.rstd = rstd;
    a.T = T; a.D = static_cast<int>(D); a.eps = eps; a.zc = zero_centered_gamma ? 1 : 0;
    return run_fwd(kGated | flags, a, stream);
}

int rmsnorm_bwd_impl(int flags, const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx, const float* w,
                     const float* rstd, rmsn_act16* dx, int64_t lddx, float* dgamma, void* ws, size_t ws_bytes,
                     int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(bwd_check_args(g, ldg, x, ldx, w, rstd, dx, lddx, dgamma, T, D));
    RMSN_TRY(check_ws(ws, ws_bytes, T, D));
    BwdArgs a{};
    a.g = g; a.ldg = ldg; a.x = x; a.ldx = ldx; a.w = w; a.rstd = rstd; a.dx = dx; a.lddx = lddx;
    a.partials = static_cast<float*>(ws); a.T = T; a.D = static_cast<int>(D); a.zc = zero_centered_gamma ? 1 : 0;
    return run_bwd(kPlain | flags, a, dgamma, stream);
}

int rmsnorm_residual_bwd_impl(int flags, const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                              const float* w, const float* rstd, const rmsn_act16* g_res, int64_t ldgr,
                              rmsn_act16* dx, int64_t lddx, float* dgamma, void* ws, size_t ws_bytes, int64_t T,
                              int64_t D, int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(g, ldg, D));
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(dx, lddx, D));
    if (g_res) RMSN_TRY(check_act(g_res, ldgr, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    if (dgamma) RMSN_TRY(check_vec(dgamma));
    RMSN_TRY(check_ws(ws, ws_bytes, T, D));
    BwdArgs a{};
    a.g = g; a.ldg = ldg; a.x = x; a.ldx = ldx; a.gres = g_res; a.ldgr = ldgr; a.w = w; a.rstd = rstd;
    a.dx = dx; a.lddx = lddx; a.partials = static_cast<float*>(ws);
    a.T = T; a.D = static_cast<int>(D); a.zc = zero_centered_gamma ? 1 : 0;
    // A zero residual gradient is the plain backward.
    return run_bwd((g_res ? kResidual : kPlain) | flags, a, dgamma, stream);
}

int rmsnorm_gated_bwd_impl(int flags, const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                           const rmsn_act16* z, int64_t ldz, const float* w, const float* rstd, rmsn_act16* dx,
                           int64_t lddx, rmsn_act16* dz, int64_t lddz, float* dw, void* ws, size_t ws_bytes,
                           int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(g, ldg, D));
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(z, ldz, D));
    RMSN_TRY(check_act(dx, lddx, D));
    RMSN_TRY(check_act(dz, lddz, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    if (dw) RMSN_TRY(check_vec(dw));
    RMSN_TRY(check_ws(ws, ws_bytes, T, D));
    BwdArgs a{};
    a.g = g; a.ldg = ldg; a.x = x; a.ldx = ldx; a.z = z; a.ldz = ldz; a.w = w; a.rstd = rstd;
    a.dx = dx; a.lddx = lddx; a.dz = dz; a.lddz = lddz; a.partials = static_cast<float*>(ws);
    a.T = T; a.D = static_cast<int>(D); a.zc = zero_centered_gamma ? 1 : 0;
    return run_bwd(kGated | flags, a, dw, stream);
}

int rmsnorm_fused_add_fwd_impl(int flags, const rmsn_act16* x, int64_t ldx, const rmsn_act16* res, int64_t ldres,
                               const float* w, rmsn_act16* y, int64_t ldy, float* rstd, rmsn_act16* res_out,
                               int64_t ldro, int64_t T, int64_t D, float eps, int zero_centered_gamma,
                               rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(res, ldres, D));
    RMSN_TRY(check_act(y, ldy, D));
    RMSN_TRY(check_act(res_out, ldro, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    RMSN_TRY(check_eps(eps));
    FwdArgs a{};
    a.x = x; a.ldx = ldx; a.res = res; a.ldres = ldres; a.w = w; a.y = y; a.ldy = ldy; a.rstd = rstd;
    a.xc = res_out; a.ldxc = ldro;
    a.T = T; a.D = static_cast<int>(D); a.eps = eps; a.zc = zero_centered_gamma ? 1 : 0;
    return run_fwd(kFusedAdd | flags, a, stream);
}

int rmsnorm_fused_add_bwd_impl(int flags, const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                               const rmsn_act16* res, int64_t ldres, const float* w, const float* rstd,
                               const rmsn_act16* g_res, int64_t ldgr, rmsn_act16* dh, int64_t lddh, float* dgamma,
                               void* ws, size_t ws_bytes, int64_t T, int64_t D, int zero_centered_gamma,
                               rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(g, ldg, D));
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(res, ldres, D));
    RMSN_TRY(check_act(dh, lddh, D));
    if (g_res) RMSN_TRY(check_act(g_res, ldgr, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    if (dgamma) RMSN_TRY(check_vec(dgamma));
    RMSN_TRY(check_ws(ws, ws_bytes, T, D));
    BwdArgs a{};
    a.g = g; a.ldg = ldg; a.x = x; a.ldx = ldx; a.res = res; a.ldres = ldres; a.gres = g_res; a.ldgr = ldgr;
    a.w = w; a.rstd = rstd; a.dx = dh; a.lddx = lddh; a.partials = static_cast<float*>(ws);
    a.T = T; a.D = static_cast<int>(D); a.zc = zero_centered_gamma ? 1 : 0;
    return run_bwd((g_res ? kFusedAdd : kFusedAddNoGres) | flags, a, dgamma, stream);
}

int rmsnorm_bwd_recompute_impl(int flags, const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                               const float* w, const float* rstd, const rmsn_act16* g_res, int64_t ldgr,
                               rmsn_act16* dx, int64_t lddx, float* dgamma, rmsn_act16* y, int64_t ldy, void* ws,
                               size_t ws_bytes, int64_t T, int64_t D, int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(g, ldg, D));
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(dx, lddx, D));
    RMSN_TRY(check_act(y, ldy, D));
    if (g_res) RMSN_TRY(check_act(g_res, ldgr, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    if (dgamma) RMSN_TRY(check_vec(dgamma));
    RMSN_TRY(check_ws(ws, ws_bytes, T, D));
    BwdArgs a{};
    a.g = g; a.ldg = ldg; a.x = x; a.ldx = ldx; a.gres = g_res; a.ldgr = ldgr; a.w = w; a.rstd = rstd;
    a.dx = dx; a.lddx = lddx; a.y = y; a.ldy = ldy; a.partials = static_cast<float*>(ws);
    a.T = T; a.D = static_cast<int>(D); a.zc = zero_centered_gamma ? 1 : 0;
    return run_bwd((g_res ? kResidual : kPlain) | flags, a, dgamma, stream);
}

int rmsnorm_gated_bwd_recompute_impl(int flags, const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                                     const rmsn_act16* z, int64_t ldz, const float* w, const float* rstd,
                                     rmsn_act16* dx, int64_t lddx, rmsn_act16* dz, int64_t lddz, float* dw,
                                     rmsn_act16* y, int64_t ldy, void* ws, size_t ws_bytes, int64_t T, int64_t D,
                                     int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(g, ldg, D));
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(z, ldz, D));
    RMSN_TRY(check_act(dx, lddx, D));
    RMSN_TRY(check_act(dz, lddz, D));
    RMSN_TRY(check_act(y, ldy, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    if (dw) RMSN_TRY(check_vec(dw));
    RMSN_TRY(check_ws(ws, ws_bytes, T, D));
    BwdArgs a{};
    a.g = g; a.ldg = ldg; a.x = x; a.ldx = ldx; a.z = z; a.ldz = ldz; a.w = w; a.rstd = rstd;
    a.dx = dx; a.lddx = lddx; a.dz = dz; a.lddz = lddz; a.y = y; a.ldy = ldy; a.partials = static_cast<float*>(ws);
    a.T = T; a.D = static_cast<int>(D); a.zc = zero_centered_gamma ? 1 : 0;
    return run_bwd(kGated | flags, a, dw, stream);
}

}  // namespace

// The rmsnorm_residual backward of T rows with the weight-gradient chunk of a
// chunk_T-row problem (for the host-buffer step, whose slabs must write the
// chunk partials of the whole problem). Only pass 1 runs.
int rmsn::residual_bwd_chunk_of(int64_t chunk_T, const uint16_t* g, int64_t ldg, const uint16_t* x, int64_t ldx,
                                const float* w, const float* rstd, const uint16_t* g_res, int64_t ldgr, uint16_t* dx,
                                int64_t lddx, void* ws, size_t ws_bytes, int64_t T, int64_t D,
                                int zero_centered_gamma, int dtype, cudaStream_t stream) {
    int flags = 0;
    RMSN_TRY(dtype_flags(dtype, &flags));
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(g, ldg, D));
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(dx, lddx, D));
    if (g_res) RMSN_TRY(check_act(g_res, ldgr, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    const RowCfg c = row_cfg(static_cast<int>(D));
    const int64_t chunk = c.narrow ? c.chunk_rows : wide_chunk_rows(chunk_T, static_cast<int>(D));
    const size_t need = static_cast<size_t>((T + chunk - 1) / chunk) * static_cast<size_t>(D) * 4u;
    if (ws == nullptr || ws_bytes < need) return RMSN_EWORKSPACE;
    if (!aligned16(ws)) return RMSN_EALIGN;
    BwdArgs a{};
    a.g = g; a.ldg = ldg; a.x = x; a.ldx = ldx; a.gres = g_res; a.ldgr = ldgr; a.w = w; a.rstd = rstd;
    a.dx = dx; a.lddx = lddx; a.partials = static_cast<float*>(ws);
    a.T = T; a.D = static_cast<int>(D); a.zc = zero_centered_gamma ? 1 : 0;
    a.chunk = c.narrow ? 0 : static_cast<int>(chunk);
    return run_bwd((g_res ? kResidual : kPlain) | flags, a, nullptr, stream);
}

// ---------------------------------------------------------------------------
// Entry points
// ---------------------------------------------------------------------------
extern "C" {

const char* rmsnorm_status_string(int status) {
    switch (status) {
        case RMSN_OK: return "RMSN_OK";
        case RMSN_EINVAL: return "RMSN_EINVAL: invalid argument (null pointer, size, stride or eps)";
        case RMSN_EALIGN: return "RMSN_EALIGN: pointer or row stride not 16-byte aligned";
        case RMSN_EUNSUPPORTED: return "RMSN_EUNSUPPORTED: D must be a multiple of 8 in [8, 16384]";
        case RMSN_ECUDA: return "RMSN_ECUDA: a CUDA call failed";
        case RMSN_EWORKSPACE: return "RMSN_EWORKSPACE: workspace missing or too small";
        default: return "unknown rmsnorm status";
    }
}

size_t rmsnorm_bwd_workspace_bytes(int64_t T, int64_t D) {
    if (check_shape(T, D) != RMSN_OK || T == 0) return 0;
    return static_cast<size_t>(num_chunks(T, static_cast<int>(D))) * static_cast<size_t>(D) * 4u;
}

int rmsnorm_fwd(const rmsn_bf16* x, int64_t ldx, const float* w, rmsn_bf16* y, int64_t ldy, float* rstd, int64_t T,
                int64_t D, float eps, int zero_centered_gamma, rmsn_stream stream) {
    return rmsnorm_fwd_impl(0, x, ldx, w, y, ldy, rstd, T, D, eps, zero_centered_gamma, stream);
}

int rmsnorm_fwd_ex(const rmsn_act16* x, int64_t ldx, const float* w, rmsn_act16* y, int64_t ldy, float* rstd,
                   int64_t T, int64_t D, float eps, int zero_centered_gamma, int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    return rmsnorm_fwd_impl(f, x, ldx, w, y, ldy, rstd, T, D, eps, zero_centered_gamma, stream);
}

int rmsnorm_residual_fwd(const rmsn_bf16* x, int64_t ldx, const float* w, rmsn_bf16* y, int64_t ldy, float* rstd,
                         rmsn_bf16* x_copy, int64_t ldxc, int64_t T, int64_t D, float eps, int zero_centered_gamma,
                         rmsn_stream stream) {
    return rmsnorm_residual_fwd_impl(0, x, ldx, w, y, ldy, rstd, x_copy, ldxc, T, D, eps, zero_centered_gamma,
                                     stream);
}

int rmsnorm_residual_fwd_ex(const rmsn_act16* x, int64_t ldx, const float* w, rmsn_act16* y, int64_t ldy,
                            float* rstd, rmsn_act16* x_copy, int64_t ldxc, int64_t T, int64_t D, float eps,
                            int zero_centered_gamma, int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    return rmsnorm_residual_fwd_impl(f, x, ldx, w, y, ldy, rstd, x_copy, ldxc, T, D, eps, zero_centered_gamma,
                                     stream);
}

int rmsnorm_gated_fwd(const rmsn_bf16* x, int64_t ldx, const rmsn_bf16* z, int64_t ldz, const float* w,
                      rmsn_bf16* y, int64_t ldy, float* rstd, int64_t T, int64_t D, float eps,
                      int zero_centered_gamma, rmsn_stream stream) {
    return rmsnorm_gated_fwd_impl(0, x, ldx, z, ldz, w, y, ldy, rstd, T, D, eps, zero_centered_gamma, stream);
}

int rmsnorm_gated_fwd_ex(const rmsn_act16* x, int64_t ldx, const rmsn_act16* z, int64_t ldz, const float* w,
                         rmsn_act16* y, int64_t ldy, float* rstd, int64_t T, int64_t D, float eps,
                         int zero_centered_gamma, int gate, int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    int fg = 0;
    RMSN_TRY(gate_flags(gate, &fg));
    f |= fg;
    return rmsnorm_gated_fwd_impl(f, x, ldx, z, ldz, w, y, ldy, rstd, T, D, eps, zero_centered_gamma, stream);
}

int rmsnorm_gated_hf_fwd(const rmsn_bf16* x, int64_t ldx, const rmsn_bf16* z, int64_t ldz, const float* w,
                         rmsn_bf16* y, int64_t ldy, float* rstd, int64_t T, int64_t D, float eps,
                         int zero_centered_gamma, rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_act(x, ldx, D));
    RMSN_TRY(check_act(z, ldz, D));
    RMSN_TRY(check_act(y, ldy, D));
    RMSN_TRY(check_vec(w));
    RMSN_TRY(check_vec(rstd));
    RMSN_TRY(check_eps(eps));
    FwdArgs a{};
    a.x = x; a.ldx = ldx; a.z = z; a.ldz = ldz; a.w = w; a.y = y; a.ldy = ldy; a.rstd = rstd;
    a.T = T; a.D = static_cast<int>(D); a.eps = eps; a.zc = zero_centered_gamma ? 1 : 0;
    return run_fwd(kGatedHF, a, stream);
}

int rmsnorm_bwd(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx, const float* w, const float* rstd,
                rmsn_bf16* dx, int64_t lddx, float* dgamma, void* ws, size_t ws_bytes, int64_t T, int64_t D,
                int zero_centered_gamma, rmsn_stream stream) {
    return rmsnorm_bwd_impl(0, g, ldg, x, ldx, w, rstd, dx, lddx, dgamma, ws, ws_bytes, T, D, zero_centered_gamma,
                            stream);
}

int rmsnorm_bwd_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx, const float* w,
                   const float* rstd, rmsn_act16* dx, int64_t lddx, float* dgamma, void* ws, size_t ws_bytes,
                   int64_t T, int64_t D, int zero_centered_gamma, int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    return rmsnorm_bwd_impl(f, g, ldg, x, ldx, w, rstd, dx, lddx, dgamma, ws, ws_bytes, T, D, zero_centered_gamma,
                            stream);
}

int rmsnorm_residual_bwd(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx, const float* w,
                         const float* rstd, const rmsn_bf16* g_res, int64_t ldgr, rmsn_bf16* dx, int64_t lddx,
                         float* dgamma, void* ws, size_t ws_bytes, int64_t T, int64_t D, int zero_centered_gamma,
                         rmsn_stream stream) {
    return rmsnorm_residual_bwd_impl(0, g, ldg, x, ldx, w, rstd, g_res, ldgr, dx, lddx, dgamma, ws, ws_bytes, T, D,
                                     zero_centered_gamma, stream);
}

int rmsnorm_residual_bwd_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx, const float* w,
                            const float* rstd, const rmsn_act16* g_res, int64_t ldgr, rmsn_act16* dx, int64_t lddx,
                            float* dgamma, void* ws, size_t ws_bytes, int64_t T, int64_t D, int zero_centered_gamma,
                            int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    return rmsnorm_residual_bwd_impl(f, g, ldg, x, ldx, w, rstd, g_res, ldgr, dx, lddx, dgamma, ws, ws_bytes, T, D,
                                     zero_centered_gamma, stream);
}

int rmsnorm_gated_bwd(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx, const rmsn_bf16* z,
                      int64_t ldz, const float* w, const float* rstd, rmsn_bf16* dx, int64_t lddx, rmsn_bf16* dz,
                      int64_t lddz, float* dw, void* ws, size_t ws_bytes, int64_t T, int64_t D,
                      int zero_centered_gamma, rmsn_stream stream) {
    return rmsnorm_gated_bwd_impl(0, g, ldg, x, ldx, z, ldz, w, rstd, dx, lddx, dz, lddz, dw, ws, ws_bytes, T, D,
                                  zero_centered_gamma, stream);
}

int rmsnorm_gated_bwd_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx, const rmsn_act16* z,
                         int64_t ldz, const float* w, const float* rstd, rmsn_act16* dx, int64_t lddx,
                         rmsn_act16* dz, int64_t lddz, float* dw, void* ws, size_t ws_bytes, int64_t T, int64_t D,
                         int zero_centered_gamma, int gate, int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    int fg = 0;
    RMSN_TRY(gate_flags(gate, &fg));
    f |= fg;
    return rmsnorm_gated_bwd_impl(f, g, ldg, x, ldx, z, ldz, w, rstd, dx, lddx, dz, lddz, dw, ws, ws_bytes, T, D,
                                  zero_centered_gamma, stream);
}

int rmsnorm_fused_add_fwd(const rmsn_bf16* x, int64_t ldx, const rmsn_bf16* res, int64_t ldres, const float* w,
                          rmsn_bf16* y, int64_t ldy, float* rstd, rmsn_bf16* res_out, int64_t ldro, int64_t T,
                          int64_t D, float eps, int zero_centered_gamma, rmsn_stream stream) {
    return rmsnorm_fused_add_fwd_impl(0, x, ldx, res, ldres, w, y, ldy, rstd, res_out, ldro, T, D, eps,
                                      zero_centered_gamma, stream);
}

int rmsnorm_fused_add_fwd_ex(const rmsn_act16* x, int64_t ldx, const rmsn_act16* res, int64_t ldres, const float* w,
                             rmsn_act16* y, int64_t ldy, float* rstd, rmsn_act16* res_out, int64_t ldro, int64_t T,
                             int64_t D, float eps, int zero_centered_gamma, int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    return rmsnorm_fused_add_fwd_impl(f, x, ldx, res, ldres, w, y, ldy, rstd, res_out, ldro, T, D, eps,
                                      zero_centered_gamma, stream);
}

int rmsnorm_fused_add_bwd(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx, const rmsn_bf16* res,
                          int64_t ldres, const float* w, const float* rstd, const rmsn_bf16* g_res, int64_t ldgr,
                          rmsn_bf16* dh, int64_t lddh, float* dgamma, void* ws, size_t ws_bytes, int64_t T,
                          int64_t D, int zero_centered_gamma, rmsn_stream stream) {
    return rmsnorm_fused_add_bwd_impl(0, g, ldg, x, ldx, res, ldres, w, rstd, g_res, ldgr, dh, lddh, dgamma, ws,
                                      ws_bytes, T, D, zero_centered_gamma, stream);
}

int rmsnorm_fused_add_bwd_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                             const rmsn_act16* res, int64_t ldres, const float* w, const float* rstd,
                             const rmsn_act16* g_res, int64_t ldgr, rmsn_act16* dh, int64_t lddh, float* dgamma,
                             void* ws, size_t ws_bytes, int64_t T, int64_t D, int zero_centered_gamma, int dtype,
                             rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    return rmsnorm_fused_add_bwd_impl(f, g, ldg, x, ldx, res, ldres, w, rstd, g_res, ldgr, dh, lddh, dgamma, ws,
                                      ws_bytes, T, D, zero_centered_gamma, stream);
}

int rmsnorm_bwd_recompute(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx, const float* w,
                          const float* rstd, const rmsn_bf16* g_res, int64_t ldgr, rmsn_bf16* dx, int64_t lddx,
                          float* dgamma, rmsn_bf16* y, int64_t ldy, void* ws, size_t ws_bytes, int64_t T, int64_t D,
                          int zero_centered_gamma, rmsn_stream stream) {
    return rmsnorm_bwd_recompute_impl(0, g, ldg, x, ldx, w, rstd, g_res, ldgr, dx, lddx, dgamma, y, ldy, ws,
                                      ws_bytes, T, D, zero_centered_gamma, stream);
}

int rmsnorm_bwd_recompute_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx, const float* w,
                             const float* rstd, const rmsn_act16* g_res, int64_t ldgr, rmsn_act16* dx, int64_t lddx,
                             float* dgamma, rmsn_act16* y, int64_t ldy, void* ws, size_t ws_bytes, int64_t T,
                             int64_t D, int zero_centered_gamma, int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    return rmsnorm_bwd_recompute_impl(f, g, ldg, x, ldx, w, rstd, g_res, ldgr, dx, lddx, dgamma, y, ldy, ws,
                                      ws_bytes, T, D, zero_centered_gamma, stream);
}

int rmsnorm_gated_bwd_recompute(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                                const rmsn_bf16* z, int64_t ldz, const float* w, const float* rstd, rmsn_bf16* dx,
                                int64_t lddx, rmsn_bf16* dz, int64_t lddz, float* dw, rmsn_bf16* y, int64_t ldy,
                                void* ws, size_t ws_bytes, int64_t T, int64_t D, int zero_centered_gamma,
                                rmsn_stream stream) {
    return rmsnorm_gated_bwd_recompute_impl(0, g, ldg, x, ldx, z, ldz, w, rstd, dx, lddx, dz, lddz, dw, y, ldy, ws,
                                            ws_bytes, T, D, zero_centered_gamma, stream);
}

int rmsnorm_gated_bwd_recompute_ex(const rmsn_act16* g, int64_t ldg, const rmsn_act16* x, int64_t ldx,
                                   const rmsn_act16* z, int64_t ldz, const float* w, const float* rstd,
                                   rmsn_act16* dx, int64_t lddx, rmsn_act16* dz, int64_t lddz, float* dw,
                                   rmsn_act16* y, int64_t ldy, void* ws, size_t ws_bytes, int64_t T, int64_t D,
                                   int zero_centered_gamma, int gate, int dtype, rmsn_stream stream) {
    int f = 0;
    RMSN_TRY(dtype_flags(dtype, &f));
    int fg = 0;
    RMSN_TRY(gate_flags(gate, &fg));
    f |= fg;
    return rmsnorm_gated_bwd_recompute_impl(f, g, ldg, x, ldx, z, ldz, w, rstd, dx, lddx, dz, lddz, dw, y, ldy, ws,
                                            ws_bytes, T, D, zero_centered_gamma, stream);
}

int rmsnorm_dgamma_reduce(const void* ws, size_t ws_bytes, int64_t T, int64_t D, float* dgamma,
                          rmsn_stream stream) {
    RMSN_TRY(check_shape(T, D));
    if (T == 0) return RMSN_OK;
    RMSN_TRY(check_vec(dgamma));
    RMSN_TRY(check_ws(ws, ws_bytes, T, D));
    return cuda_status(launch_dgamma_reduce(static_cast<const float*>(ws), num_chunks(T, static_cast<int>(D)),
                                            static_cast<int>(D), dgamma, stream));
}

int rmsnorm_device_error(unsigned int* flags, int clear) {
    if (flags == nullptr) return RMSN_EINVAL;
    *flags = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = wide_read_error(flags, clear != 0);
    if (e == cudaSuccess) e = narrow_read_error(flags, clear != 0);
    if (e == cudaSuccess) e = wide_f16_read_error(flags, clear != 0);
    if (e == cudaSuccess) e = narrow_f16_read_error(flags, clear != 0);
    if (e == cudaSuccess) e = selftest_read_error(flags, clear != 0);
    return cuda_status(e);
}

}  // extern "C"
