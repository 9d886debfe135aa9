// Backward entry point for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device buffer for the weight-gradient
// scratch: code running where cudaMalloc is forbidden or unavailable (inside a
// framework hook that only hands out its own input and output tensors, a
// plugin whose host owns all allocation, or a runtime that must not allocate
// after start-up so that its memory footprint stays fixed). This entry point
// serves them: it keeps the scratch in a fixed array that is part of this
// library's device image, so the call itself allocates nothing.
//
// The array is RMSN_NOALLOC_SCRATCH_BYTES (32 MiB) on every GPU where the
// library's device code is loaded, held until the process exits. Its device
// address is looked up once per device, on the first call made with that
// device current (so that first call should come before any stream capture),
// and again after the device's context has been destroyed and recreated
// (cudaDeviceReset), which reloads the module and can move the array: the
// address is kept with the context's unique id and used only in that context.
// All calls share the array: two calls that overlap on the GPU (different
// streams, or different host threads, without ordering between them) race on
// it and give wrong weight gradients. Nothing in the array has to start at
// zero: every partial row the backward reads was written earlier in the same
// call, so the contents a previous call left behind are never used.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace rmsn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RMSN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct ScratchEntry {
    unsigned long long ctx_id;  // unique id of the context the address belongs to (0: none yet)
    void* ptr;
};
ScratchEntry g_noalloc[kMaxDevices] = {};

// Device address of the scratch array in the current device's context. In
// host code the array's name is only a host-side stand-in; the real address
// must come from cudaGetSymbolAddress, made with the device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RMSN_ECUDA;
    // Before the runtime has made the device's context current there is no id:
    // the lookup below then runs, and the id is kept from a later call.
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    ScratchEntry& e = g_noalloc[dev];
    if (!have_ctx || e.ptr == nullptr || e.ctx_id != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return RMSN_ECUDA;
        e.ptr = p;
        e.ctx_id = have_ctx ? ctx : 0;  // without a context id, look it up on every call
    }
    *out = e.ptr;
    return RMSN_OK;
}

}  // namespace
}  // namespace rmsn

extern "C" int rmsnorm_bwd_noalloc(const rmsn_bf16* g, int64_t ldg, const rmsn_bf16* x, int64_t ldx,
                                   const float* w, const float* rstd, rmsn_bf16* dx, int64_t lddx,
                                   float* dgamma, int64_t T, int64_t D, int zero_centered_gamma,
                                   rmsn_stream stream) {
    // rmsnorm_bwd's own checks first, in its order, so that a call fails with
    // the status rmsnorm_bwd would give; then this entry point's two limits.
    const size_t need = rmsnorm_bwd_workspace_bytes(T, D);
    if (need == 0) {
        // T == 0 (nothing to do) or an invalid shape: the regular entry point
        // returns the right status without touching the device.
        return rmsnorm_bwd(g, ldg, x, ldx, w, rstd, dx, lddx, dgamma, nullptr, 0, T, D, zero_centered_gamma,
                           stream);
    }
    const int st = rmsn::bwd_check_args(g, ldg, x, ldx, w, rstd, dx, lddx, dgamma, T, D);
    if (st != RMSN_OK) return st;
    if (dgamma == nullptr) return RMSN_EINVAL;                     // partials cannot be left in the shared array
    if (need > RMSN_NOALLOC_SCRATCH_BYTES) return RMSN_EWORKSPACE;  // problem too large for the array
    void* scratch = nullptr;
    const int sa = rmsn::scratch_address(&scratch);
    if (sa != RMSN_OK) return sa;
    return rmsnorm_bwd(g, ldg, x, ldx, w, rstd, dx, lddx, dgamma, scratch, RMSN_NOALLOC_SCRATCH_BYTES, T, D,
                       zero_centered_gamma, stream);
}
