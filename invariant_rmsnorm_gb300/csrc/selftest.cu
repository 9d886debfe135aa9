// Self-test of the bounded waits' error path.
//
// Every wait of the kernels on an mbarrier gives up after a time limit,
// raises a device error flag and lets its kernel return, so that a stalled
// copy never hangs the GPU and the host learns of it through
// rmsnorm_device_error(). This entry point exercises that path on purpose and
// without any fault: one thread waits, with the kernels' own wait routine and
// a caller-chosen limit, on a fresh mbarrier that nothing ever arrives on. The
// wait runs out, the thread raises the flag the kernels raise
// (RMSN_DEVICE_ERR_WAIT_TIMEOUT) and the kernel ends normally; the context
// stays usable.
#include "common.cuh"
#include "kernels.h"

namespace rmsn {
namespace {

__device__ unsigned int g_selftest_error;

constexpr unsigned long long kSelftestMaxLimitNs = 1000000000ull;  // 1 s

__global__ void wait_timeout_probe_kernel(unsigned long long limit_ns, unsigned long long* waited_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // expects one arrive; none ever comes
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned long long t0 = global_timer_ns();
        const bool done = mbar_wait(&bar, 0u, limit_ns);
        if (waited_ns != nullptr) *waited_ns = global_timer_ns() - t0;
        if (!done) atomicOr(&g_selftest_error, kErrWaitTimeout);
    }
}

}  // namespace

cudaError_t selftest_read_error(unsigned* flags, bool clear) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_selftest_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *flags |= v;
    if (clear && v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace rmsn

extern "C" int rmsnorm_selftest_wait_timeout(unsigned long long limit_ns, unsigned long long* waited_ns,
                                             rmsn_stream stream) {
    if (limit_ns == 0 || limit_ns > rmsn::kSelftestMaxLimitNs) return RMSN_EINVAL;
    if (waited_ns != nullptr && (reinterpret_cast<uintptr_t>(waited_ns) & 7u) != 0) return RMSN_EALIGN;
    rmsn::wait_timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, waited_ns);
    return cudaGetLastError() == cudaSuccess ? RMSN_OK : RMSN_ECUDA;
}
