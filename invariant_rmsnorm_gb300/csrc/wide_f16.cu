// Wide-row kernels (D > 256) with fp16 activations: the instantiations of
// wide_impl.cuh for the fp16 modes (the HF-convention witness is bf16 only),
// compiled apart from the bf16 ones so that the two build in parallel.
#include "wide_impl.cuh"

namespace rmsn {

cudaError_t wide_f16_read_error(unsigned* flags, bool clear) { return read_wide_error_word(flags, clear); }

cudaError_t launch_wide_fwd_f16(int m, const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    constexpr int H = kFlagF16;
    switch (m) {
        case kPlain | H: return fwd_dispatch<kPlain | H>(a, c, st);
        case kResidual | H: return fwd_dispatch<kResidual | H>(a, c, st);
        case kGated | H: return fwd_dispatch<kGated | H>(a, c, st);
        case kGated | kFlagSigmoid | H: return fwd_dispatch<kGated | kFlagSigmoid | H>(a, c, st);
        case kFusedAdd | H:
        case kFusedAddNoGres | H: return fwd_dispatch<kFusedAdd | H>(a, c, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_wide_bwd_f16(int m, const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    constexpr int H = kFlagF16;
    switch (m) {
        case kPlain | H: return bwd_dispatch<kPlain | H>(a, c, st);
        case kResidual | H: return bwd_dispatch<kResidual | H>(a, c, st);
        case kGated | H: return bwd_dispatch<kGated | H>(a, c, st);
        case kGated | kFlagSigmoid | H: return bwd_dispatch<kGated | kFlagSigmoid | H>(a, c, st);
        case kPlain | kFlagRecompute | H: return bwd_dispatch<kPlain | kFlagRecompute | H>(a, c, st);
        case kResidual | kFlagRecompute | H: return bwd_dispatch<kResidual | kFlagRecompute | H>(a, c, st);
        case kGated | kFlagRecompute | H: return bwd_dispatch<kGated | kFlagRecompute | H>(a, c, st);
        case kGated | kFlagSigmoid | kFlagRecompute | H: return bwd_dispatch<kGated | kFlagSigmoid | kFlagRecompute | H>(a, c, st);
        case kFusedAdd | H: return bwd_dispatch<kFusedAdd | H>(a, c, st);
        case kFusedAddNoGres | H: return bwd_dispatch<kFusedAddNoGres | H>(a, c, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
