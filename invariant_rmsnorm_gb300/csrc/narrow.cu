// Narrow-row support (D <= 256) and tensor-map encoding.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace rmsn {

static __device__ unsigned int g_narrow_error;

cudaError_t narrow_read_error(unsigned* flags, bool clear) {
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

cudaError_t launch_narrow_fwd(Mode, const FwdArgs&, const RowCfg&, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t launch_narrow_bwd(Mode, const BwdArgs&, const RowCfg&, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace rmsn
