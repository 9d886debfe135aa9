// rmsnorm_residual step on host-resident buffers.
//
// A caller whose activations live in host memory (a data loader's pinned
// staging buffers, a host-side optimiser, a test harness) would otherwise
// copy every input to the device, run the forward and the backward, and copy
// every output back, one after the other, leaving the PCIe/C2C link idle while
// the kernels run and the kernels idle while the link runs. This entry point
// does the whole step in one call and overlaps the three: the rows are cut
// into slabs, and while the kernels of slab k run, the inputs of slab k+1 come
// in on one stream and the outputs of slab k-1 go out on another.
//
// Device memory is a caller-provided work buffer: a ring of three slab slots
// (inputs and outputs of one slab each), the weights, the weight gradient and
// the per-chunk weight-gradient partials of all T rows. Slabs are whole
// weight-gradient chunks, so each slab's backward writes exactly its own
// chunks' partials, and one pass 2 over all chunks gives the weight gradient
// of the unsliced step bit for bit; the row outputs are the same bits as the
// unsliced step's because every row is reduced independently of the others.
//
// Streams and events: the kernels run on the caller's stream; the copies run
// on two non-blocking streams per device that the library creates on first use
// and keeps until the process exits, with events ordering the three. Slot
// reuse is ordered by those events: slab k's inputs wait until the kernels of
// slab k-3 (same slot) have read theirs, and slab k's kernels wait until the
// outputs of slab k-3 have left. The call begins after all earlier work on the
// caller's stream and the caller's stream waits for the last copy, so calls on
// one stream are ordered like any other stream work.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace rmsn {
namespace {

constexpr int kSlots = 3;                 // ring of slab slots in the work buffer
constexpr int64_t kDefaultSlabRows = 4096;
constexpr int kMaxDevices = 64;

size_t round256(size_t n) { return (n + 255u) & ~static_cast<size_t>(255u); }

// Byte offsets of the parts of the work buffer for one problem.
struct WorkLayout {
    int64_t slab_rows = 0;  // rows per slab (whole chunks)
    int64_t nslabs = 0;
    int slots = 0;          // slab slots actually used (<= kSlots)
    size_t act_bytes = 0;   // one [slab_rows][D] activation buffer, rounded
    size_t rstd_bytes = 0;  // one [slab_rows] fp32 buffer, rounded
    size_t w = 0, dgamma = 0, partials = 0, slot0 = 0, slot_bytes = 0, total = 0;
};

// Rows per weight-gradient chunk of the whole T-row problem: every slab starts
// on a chunk boundary and its backward writes the whole problem's chunks.
int64_t step_chunk_rows(int64_t T, int64_t D) {
    const RowCfg c = row_cfg(static_cast<int>(D));
    return c.narrow ? c.chunk_rows : wide_chunk_rows(T, static_cast<int>(D));
}

// Slab rows: the request (0 = default), rounded up to whole chunks and capped
// at the chunk-rounded T.
WorkLayout layout(int64_t T, int64_t D, int64_t slab_rows) {
    WorkLayout L{};
    const int64_t chunk = step_chunk_rows(T, D);
    int64_t s = slab_rows > 0 ? slab_rows : kDefaultSlabRows;
    if (s > T) s = T;  // first, so that the rounding below cannot overflow
    s = (s + chunk - 1) / chunk * chunk;
    const int64_t t_chunks = (T + chunk - 1) / chunk * chunk;
    if (s > t_chunks) s = t_chunks;
    if (s <= 0) s = chunk;
    L.slab_rows = s;
    L.nslabs = (T + s - 1) / s;
    L.slots = static_cast<int>(L.nslabs < kSlots ? L.nslabs : kSlots);
    if (L.slots < 1) L.slots = 1;
    L.act_bytes = round256(static_cast<size_t>(s) * static_cast<size_t>(D) * 2u);
    L.rstd_bytes = round256(static_cast<size_t>(s) * 4u);
    L.w = 0;
    L.dgamma = L.w + round256(static_cast<size_t>(D) * 4u);
    L.partials = L.dgamma + round256(static_cast<size_t>(D) * 4u);
    L.slot0 = L.partials + round256(rmsnorm_bwd_workspace_bytes(T, D));
    L.slot_bytes = 6 * L.act_bytes + L.rstd_bytes;  // x, g, g_res, y, x_copy, dx, rstd
    L.total = L.slot0 + static_cast<size_t>(L.slots) * L.slot_bytes;
    return L;
}

// Per-device copy streams and the events that order them, created on first
// use with that device current and kept until the process exits.
struct StepCtx {
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, w_in = nullptr, reduced = nullptr, done = nullptr;
    cudaEvent_t in[kSlots] = {}, computed[kSlots] = {}, out[kSlots] = {};
};

std::mutex g_step_mu;  // held while a call creates or enqueues on the shared context
StepCtx* g_step_ctx[kMaxDevices] = {};

int make_event(cudaEvent_t* e) {
    return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess ? RMSN_OK : RMSN_ECUDA;
}

// Caller holds g_step_mu.
int step_ctx(StepCtx** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RMSN_ECUDA;
    if (g_step_ctx[dev] == nullptr) {
        StepCtx* c = new StepCtx();
        int st = RMSN_OK;
        if (cudaStreamCreateWithFlags(&c->s_in, cudaStreamNonBlocking) != cudaSuccess) st = RMSN_ECUDA;
        if (st == RMSN_OK && cudaStreamCreateWithFlags(&c->s_out, cudaStreamNonBlocking) != cudaSuccess)
            st = RMSN_ECUDA;
        for (cudaEvent_t* e : {&c->start, &c->w_in, &c->reduced, &c->done})
            if (st == RMSN_OK) st = make_event(e);
        for (int i = 0; i < kSlots && st == RMSN_OK; ++i) {
            st = make_event(&c->in[i]);
            if (st == RMSN_OK) st = make_event(&c->computed[i]);
            if (st == RMSN_OK) st = make_event(&c->out[i]);
        }
        if (st != RMSN_OK) return st;  // the partly built context is leaked, never used
        g_step_ctx[dev] = c;
    }
    *out = g_step_ctx[dev];
    return RMSN_OK;
}

#define RMSN_STEP_CUDA(expr)                            \
    do {                                                \
        if ((expr) != cudaSuccess) return RMSN_ECUDA;   \
    } while (0)
#define RMSN_STEP_TRY(expr)                 \
    do {                                    \
        const int _st = (expr);             \
        if (_st != RMSN_OK) return _st;     \
    } while (0)

inline cudaError_t h2d(void* dst, const void* src, size_t n, cudaStream_t s) {
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s);
}
inline cudaError_t d2h(void* dst, const void* src, size_t n, cudaStream_t s) {
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, s);
}

}  // namespace
}  // namespace rmsn

extern "C" size_t rmsnorm_residual_step_host_work_bytes(int64_t T, int64_t D, int64_t slab_rows) {
    if (T <= 0 || T >= (int64_t(1) << 31) || D < 8 || D > 16384 || (D % 8) != 0 || slab_rows < 0) return 0;
    return rmsn::layout(T, D, slab_rows).total;
}

extern "C" int rmsnorm_residual_step_host(const rmsn_act16* x, const rmsn_act16* g, const rmsn_act16* g_res,
                                          const float* w, rmsn_act16* y, rmsn_act16* x_copy, float* rstd,
                                          rmsn_act16* dx, float* dgamma, int64_t T, int64_t D, float eps,
                                          int zero_centered_gamma, int dtype, int64_t slab_rows, void* work,
                                          size_t work_bytes, rmsn_stream stream) {
    using namespace rmsn;
    // Every argument is checked before anything is enqueued.
    if (dtype != RMSN_DTYPE_BF16 && dtype != RMSN_DTYPE_F16) return RMSN_EINVAL;
    if (T < 0 || T >= (int64_t(1) << 31) || slab_rows < 0) return RMSN_EINVAL;
    if (D < 8 || D > 16384 || (D % 8) != 0) return RMSN_EUNSUPPORTED;
    if (!std::isfinite(eps) || eps < 0.0f) return RMSN_EINVAL;
    if (T == 0) return RMSN_OK;
    if (x == nullptr || g == nullptr || w == nullptr || y == nullptr || x_copy == nullptr || rstd == nullptr ||
        dx == nullptr || dgamma == nullptr)
        return RMSN_EINVAL;
    const WorkLayout L = layout(T, D, slab_rows);
    if (work == nullptr || work_bytes < L.total) return RMSN_EWORKSPACE;
    if ((reinterpret_cast<uintptr_t>(work) & 255u) != 0) return RMSN_EALIGN;

    unsigned char* base = static_cast<unsigned char*>(work);
    float* d_w = reinterpret_cast<float*>(base + L.w);
    float* d_dgamma = reinterpret_cast<float*>(base + L.dgamma);
    unsigned char* d_partials = base + L.partials;
    const size_t partials_bytes = rmsnorm_bwd_workspace_bytes(T, D);
    const int64_t chunk = step_chunk_rows(T, D);
    const size_t row_bytes = static_cast<size_t>(D) * 2u;
    const size_t chunk_partial_bytes = static_cast<size_t>(D) * 4u;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lk(g_step_mu);
    StepCtx* c = nullptr;
    RMSN_STEP_TRY(step_ctx(&c));

    // Begin after the caller's earlier work; weights first.
    RMSN_STEP_CUDA(cudaEventRecord(c->start, s));
    RMSN_STEP_CUDA(cudaStreamWaitEvent(c->s_in, c->start, 0));
    RMSN_STEP_CUDA(cudaStreamWaitEvent(c->s_out, c->start, 0));
    RMSN_STEP_CUDA(h2d(d_w, w, static_cast<size_t>(D) * 4u, c->s_in));
    RMSN_STEP_CUDA(cudaEventRecord(c->w_in, c->s_in));
    RMSN_STEP_CUDA(cudaStreamWaitEvent(s, c->w_in, 0));

    for (int64_t k = 0; k < L.nslabs; ++k) {
        const int slot = static_cast<int>(k % L.slots);
        const int64_t a = k * L.slab_rows;
        const int64_t rows = (T - a < L.slab_rows) ? (T - a) : L.slab_rows;
        const size_t nb = static_cast<size_t>(rows) * row_bytes;
        const size_t host_off = static_cast<size_t>(a) * row_bytes;
        unsigned char* sb = base + L.slot0 + static_cast<size_t>(slot) * L.slot_bytes;
        rmsn_act16* s_x = reinterpret_cast<rmsn_act16*>(sb + 0 * L.act_bytes);
        rmsn_act16* s_g = reinterpret_cast<rmsn_act16*>(sb + 1 * L.act_bytes);
        rmsn_act16* s_gr = reinterpret_cast<rmsn_act16*>(sb + 2 * L.act_bytes);
        rmsn_act16* s_y = reinterpret_cast<rmsn_act16*>(sb + 3 * L.act_bytes);
        rmsn_act16* s_xc = reinterpret_cast<rmsn_act16*>(sb + 4 * L.act_bytes);
        rmsn_act16* s_dx = reinterpret_cast<rmsn_act16*>(sb + 5 * L.act_bytes);
        float* s_rstd = reinterpret_cast<float*>(sb + 6 * L.act_bytes);
        const bool reuse = k >= L.slots;  // the slot held slab k - slots

        // Inputs in, once the slot's previous slab has been read by its kernels.
        if (reuse) RMSN_STEP_CUDA(cudaStreamWaitEvent(c->s_in, c->computed[slot], 0));
        RMSN_STEP_CUDA(h2d(s_x, reinterpret_cast<const unsigned char*>(x) + host_off, nb, c->s_in));
        RMSN_STEP_CUDA(h2d(s_g, reinterpret_cast<const unsigned char*>(g) + host_off, nb, c->s_in));
        if (g_res != nullptr)
            RMSN_STEP_CUDA(h2d(s_gr, reinterpret_cast<const unsigned char*>(g_res) + host_off, nb, c->s_in));
        RMSN_STEP_CUDA(cudaEventRecord(c->in[slot], c->s_in));

        // Kernels, once the inputs are in and the slot's previous outputs are out.
        RMSN_STEP_CUDA(cudaStreamWaitEvent(s, c->in[slot], 0));
        if (reuse) RMSN_STEP_CUDA(cudaStreamWaitEvent(s, c->out[slot], 0));
        RMSN_STEP_TRY(rmsnorm_residual_fwd_ex(s_x, D, d_w, s_y, D, s_rstd, s_xc, D, rows, D, eps,
                                              zero_centered_gamma, dtype, stream));
        const size_t p_off = static_cast<size_t>(a / chunk) * chunk_partial_bytes;
        RMSN_STEP_TRY(residual_bwd_chunk_of(T, s_g, D, s_x, D, d_w, s_rstd, g_res != nullptr ? s_gr : nullptr, D,
                                            s_dx, D, d_partials + p_off, partials_bytes - p_off, rows, D,
                                            zero_centered_gamma, dtype, s));
        RMSN_STEP_CUDA(cudaEventRecord(c->computed[slot], s));

        // Outputs out.
        RMSN_STEP_CUDA(cudaStreamWaitEvent(c->s_out, c->computed[slot], 0));
        RMSN_STEP_CUDA(d2h(reinterpret_cast<unsigned char*>(y) + host_off, s_y, nb, c->s_out));
        RMSN_STEP_CUDA(d2h(reinterpret_cast<unsigned char*>(x_copy) + host_off, s_xc, nb, c->s_out));
        RMSN_STEP_CUDA(d2h(reinterpret_cast<unsigned char*>(dx) + host_off, s_dx, nb, c->s_out));
        RMSN_STEP_CUDA(d2h(rstd + a, s_rstd, static_cast<size_t>(rows) * 4u, c->s_out));
        RMSN_STEP_CUDA(cudaEventRecord(c->out[slot], c->s_out));
    }

    // Weight-gradient pass 2 over every chunk, then the result out; the
    // caller's stream ends the step when the last copy has landed.
    RMSN_STEP_TRY(rmsnorm_dgamma_reduce(d_partials, partials_bytes, T, D, d_dgamma, stream));
    RMSN_STEP_CUDA(cudaEventRecord(c->reduced, s));
    RMSN_STEP_CUDA(cudaStreamWaitEvent(c->s_out, c->reduced, 0));
    RMSN_STEP_CUDA(d2h(dgamma, d_dgamma, static_cast<size_t>(D) * 4u, c->s_out));
    RMSN_STEP_CUDA(cudaEventRecord(c->done, c->s_out));
    RMSN_STEP_CUDA(cudaStreamWaitEvent(s, c->done, 0));
    return RMSN_OK;
}
