// Narrow-row kernels (D <= 256) with fp16 activations: the instantiations of
// narrow_impl.cuh for the fp16 modes (the HF-convention witness is bf16 only),
// compiled apart from the bf16 ones so that the two build in parallel.
#include "narrow_impl.cuh"

namespace rmsn {

cudaError_t narrow_f16_read_error(unsigned* flags, bool clear) { return read_narrow_error_word(flags, clear); }

cudaError_t launch_narrow_fwd_f16(int md, const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    constexpr int H = kFlagF16;
    switch (md) {
        case kPlain | H: return nfwd_dispatch<kPlain | H>(a, c, st);
        case kResidual | H: return nfwd_dispatch<kResidual | H>(a, c, st);
        case kGated | H: return nfwd_dispatch<kGated | H>(a, c, st);
        case kGated | kFlagSigmoid | H: return nfwd_dispatch<kGated | kFlagSigmoid | H>(a, c, st);
        case kFusedAdd | H:
        case kFusedAddNoGres | H: return nfwd_dispatch<kFusedAdd | H>(a, c, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_narrow_bwd_f16(int md, const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    constexpr int H = kFlagF16;
    switch (md) {
        case kPlain | H: return nbwd_dispatch<kPlain | H>(a, c, st);
        case kResidual | H: return nbwd_dispatch<kResidual | H>(a, c, st);
        case kGated | H: return nbwd_dispatch<kGated | H>(a, c, st);
        case kGated | kFlagSigmoid | H: return nbwd_dispatch<kGated | kFlagSigmoid | H>(a, c, st);
        case kPlain | kFlagRecompute | H: return nbwd_dispatch<kPlain | kFlagRecompute | H>(a, c, st);
        case kResidual | kFlagRecompute | H: return nbwd_dispatch<kResidual | kFlagRecompute | H>(a, c, st);
        case kGated | kFlagRecompute | H: return nbwd_dispatch<kGated | kFlagRecompute | H>(a, c, st);
        case kGated | kFlagSigmoid | kFlagRecompute | H: return nbwd_dispatch<kGated | kFlagSigmoid | kFlagRecompute | H>(a, c, st);
        case kFusedAdd | H: return nbwd_dispatch<kFusedAdd | H>(a, c, st);
        case kFusedAddNoGres | H: return nbwd_dispatch<kFusedAddNoGres | H>(a, c, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
