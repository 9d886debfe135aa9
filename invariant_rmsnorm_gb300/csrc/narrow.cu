// Narrow-row kernels (D <= 256) with bf16 activations: the instantiations of
// narrow_impl.cuh for every bf16 mode and their launch entry points, plus the
// host-side tensor-map encoding shared with narrow_f16.cu.
#include <cudaTypedefs.h>

#include <mutex>

#include "narrow_impl.cuh"

namespace rmsn {

cudaError_t narrow_read_error(unsigned* flags, bool clear) { return read_narrow_error_word(flags, clear); }

// ---------------------------------------------------------------------------
// Tensor maps (encoded on the host through the driver entry point)
// ---------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

cudaError_t encode_rows_2d(CUtensorMap* map, const void* base, int64_t T, int D, int64_t ld_elems, int box_rows,
                           bool f16) {
    auto fn = encode_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_elems) * 2u};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_vec_1d(CUtensorMap* map, const float* base, int64_t T, int box) {
    auto fn = encode_fn();
    if (fn == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[1] = {static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {4};  // unused for rank 1
    const cuuint32_t boxd[1] = {static_cast<cuuint32_t>(box)};
    const cuuint32_t estr[1] = {1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, const_cast<float*>(base), dims, strides, boxd, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int narrow_chunk_rows_for_group(int G) {
    switch (G) {
        case 1: return narrow_chunk_rows<1>();
        case 2: return narrow_chunk_rows<2>();
        case 4: return narrow_chunk_rows<4>();
        case 8: return narrow_chunk_rows<8>();
        case 16: return narrow_chunk_rows<16>();
        default: return narrow_chunk_rows<32>();
    }
}

int narrow_stage_rows_for_group(int G) {
    switch (G) {
        case 1: return narrow_stage_rows<1>();
        case 2: return narrow_stage_rows<2>();
        case 4: return narrow_stage_rows<4>();
        case 8: return narrow_stage_rows<8>();
        case 16: return narrow_stage_rows<16>();
        default: return narrow_stage_rows<32>();
    }
}

cudaError_t launch_narrow_fwd(int md, const FwdArgs& a, const RowCfg& c, cudaStream_t st) {
    switch (md) {
        case kPlain: return nfwd_dispatch<kPlain>(a, c, st);
        case kResidual: return nfwd_dispatch<kResidual>(a, c, st);
        case kGated: return nfwd_dispatch<kGated>(a, c, st);
        case kGated | kFlagSigmoid: return nfwd_dispatch<kGated | kFlagSigmoid>(a, c, st);
        case kFusedAdd:
        case kFusedAddNoGres: return nfwd_dispatch<kFusedAdd>(a, c, st);
        case kGatedHF: return nfwd_dispatch<kGatedHF>(a, c, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_narrow_bwd(int md, const BwdArgs& a, const RowCfg& c, cudaStream_t st) {
    switch (md) {
        case kPlain: return nbwd_dispatch<kPlain>(a, c, st);
        case kResidual: return nbwd_dispatch<kResidual>(a, c, st);
        case kGated: return nbwd_dispatch<kGated>(a, c, st);
        case kGated | kFlagSigmoid: return nbwd_dispatch<kGated | kFlagSigmoid>(a, c, st);
        case kPlain | kFlagRecompute: return nbwd_dispatch<kPlain | kFlagRecompute>(a, c, st);
        case kResidual | kFlagRecompute: return nbwd_dispatch<kResidual | kFlagRecompute>(a, c, st);
        case kGated | kFlagRecompute: return nbwd_dispatch<kGated | kFlagRecompute>(a, c, st);
        case kGated | kFlagSigmoid | kFlagRecompute: return nbwd_dispatch<kGated | kFlagSigmoid | kFlagRecompute>(a, c, st);
        case kFusedAdd: return nbwd_dispatch<kFusedAdd>(a, c, st);
        case kFusedAddNoGres: return nbwd_dispatch<kFusedAddNoGres>(a, c, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace rmsn
