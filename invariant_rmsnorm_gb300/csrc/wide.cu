// Wide-row kernels (D > 256) with bf16 activations: the instantiations of
// wide_impl.cuh for every bf16 mode, and their launch entry points.
#include "wide_impl.cuh"

namespace rmsn {

cudaError_t wide_read_error(unsigned* flags, bool clear) { return read_wide_error_word(flags, clear); }

cudaError_t launch_wide_fwd(int m, const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    switch (m) {
        case kPlain: return fwd_dispatch<kPlain>(a, c, st);
        case kResidual: return fwd_dispatch<kResidual>(a, c, st);
        case kGated: return fwd_dispatch<kGated>(a, c, st);
        case kGated | kFlagSigmoid: return fwd_dispatch<kGated | kFlagSigmoid>(a, c, st);
        case kFusedAdd:
        case kFusedAddNoGres: return fwd_dispatch<kFusedAdd>(a, c, st);
        case kGatedHF: return fwd_dispatch<kGatedHF>(a, c, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_wide_bwd(int m, const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    switch (m) {
        case kPlain: return bwd_dispatch<kPlain>(a, c, st);
        case kResidual: return bwd_dispatch<kResidual>(a, c, st);
        case kGated: return bwd_dispatch<kGated>(a, c, st);
        case kGated | kFlagSigmoid: return bwd_dispatch<kGated | kFlagSigmoid>(a, c, st);
        case kPlain | kFlagRecompute: return bwd_dispatch<kPlain | kFlagRecompute>(a, c, st);
        case kResidual | kFlagRecompute: return bwd_dispatch<kResidual | kFlagRecompute>(a, c, st);
        case kGated | kFlagRecompute: return bwd_dispatch<kGated | kFlagRecompute>(a, c, st);
        case kGated | kFlagSigmoid | kFlagRecompute: return bwd_dispatch<kGated | kFlagSigmoid | kFlagRecompute>(a, c, st);
        case kFusedAdd: return bwd_dispatch<kFusedAdd>(a, c, st);
        case kFusedAddNoGres: return bwd_dispatch<kFusedAddNoGres>(a, c, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
