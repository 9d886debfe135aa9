// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rmsn {

// kFusedAdd / kFusedAddNoGres: the norm of h = x + res (fp32), forward also
// returning bf16(h); the backward with or without the gradient of that output.
// kGatedHF: the gated forward in the HF convention (bf16 casts around the
// weight multiply); forward only.
enum Mode : int { kPlain = 0, kResidual = 1, kGated = 2, kFusedAdd = 3, kFusedAddNoGres = 4, kGatedHF = 5 };

// Variant flags OR-ed into a mode (the kernels' MODE template argument):
// fp16 activations instead of bf16, and for kGated the sigmoid gate instead of
// silu. The arithmetic between load and store is the same fp32 in every case.
constexpr int kModeMask = 0xff;
constexpr int kFlagF16 = 0x100;
constexpr int kFlagSigmoid = 0x200;
// The backward that also writes the forward output y again (recompute), as a
// compile-time flag, so that the other backward kernels carry no y code.
constexpr int kFlagRecompute = 0x400;

__host__ __device__ constexpr int base_mode(int mode) { return mode & kModeMask; }
__host__ __device__ constexpr bool is_f16(int mode) { return (mode & kFlagF16) != 0; }
__host__ __device__ constexpr bool is_sigmoid_gate(int mode) { return (mode & kFlagSigmoid) != 0; }
__host__ __device__ constexpr bool is_recompute(int mode) { return (mode & kFlagRecompute) != 0; }
__host__ __device__ constexpr bool is_fused(int mode) {
    return base_mode(mode) == kFusedAdd || base_mode(mode) == kFusedAddNoGres;
}
__host__ __device__ constexpr bool is_gated(int mode) {
    return base_mode(mode) == kGated || base_mode(mode) == kGatedHF;
}

// Operands streamed per row, by mode.
__host__ __device__ constexpr int fwd_inputs(int mode) { return (is_gated(mode) || is_fused(mode)) ? 2 : 1; }
__host__ __device__ constexpr int bwd_inputs(int mode) {
    return base_mode(mode) == kPlain ? 2
           : (base_mode(mode) == kResidual || base_mode(mode) == kGated || base_mode(mode) == kFusedAddNoGres) ? 3
                                                                                                                : 4;
}
__host__ __device__ constexpr bool has_gres(int mode) {
    return base_mode(mode) == kResidual || base_mode(mode) == kFusedAdd;
}

// Everything a forward launch needs (unused pointers are null).
struct FwdArgs {
    const uint16_t* x; int64_t ldx;
    const uint16_t* z; int64_t ldz;     // gate (gated)
    const float* w;
    uint16_t* y; int64_t ldy;
    float* rstd;
    uint16_t* xc; int64_t ldxc;         // input copy (residual) / bf16(x + res) (fused add)
    const uint16_t* res; int64_t ldres; // residual stream (fused add)
    int64_t T; int D; float eps; int zc;
    float inv_d_pow2;                   // 1/D if D is a power of two, else 0
};

// Everything a backward (pass 1) launch needs.
struct BwdArgs {
    const uint16_t* g; int64_t ldg;
    const uint16_t* x; int64_t ldx;
    const uint16_t* z; int64_t ldz;     // gate (gated)
    const uint16_t* gres; int64_t ldgr; // gradient of the input copy (residual) / of bf16(x+res) (fused)
    const uint16_t* res; int64_t ldres; // residual stream (fused add)
    const float* w;
    const float* rstd;
    uint16_t* dx; int64_t lddx;
    uint16_t* dz; int64_t lddz;         // gated
    float* partials;                    // [nchunks][D] fp32 (workspace)
    uint16_t* y; int64_t ldy;           // optional: the forward output, recomputed (null = skip)
    int64_t T; int D; int zc;
    float inv_d_pow2;                   // 1/D if D is a power of two, else 0
    int chunk;                          // wide path: rows per weight-gradient chunk (0: wide_chunk_rows(T, D))
};

// Row-shape configuration: a pure function of D.
struct RowCfg {
    bool narrow;         // D <= 256: several rows per CTA, one lane group per row
    int threads;         // CTA size (forward)
    int vpt;             // 16-byte vectors per thread per row (wide forward); 1 (narrow)
    int bwd_threads;     // CTA size (wide backward)
    int bwd_vpt;         // 16-byte vectors per thread per row (wide backward)
    bool bwd_pair;       // wide backward: each row split between the two CTAs of a cluster
    int group;           // lanes per row (narrow), a power of two <= 32
    int rows_per_stage;  // rows per pipeline stage (narrow); 1 (wide)
    int chunk_rows;      // rows per weight-gradient partial
};

RowCfg row_cfg(int D);
int narrow_chunk_rows_for_group(int G);
int narrow_stage_rows_for_group(int G);
int64_t num_chunks(int64_t T, int D);
// Rows per weight-gradient chunk of the wide backward (D > 256) for T rows:
// a function of T and D only (see api.cu).
int64_t wide_chunk_rows(int64_t T, int D);
// The most chunks any row count 1..T_max gets on the wide path (closed form).
int64_t wide_chunks_max(int64_t T_max, int D);
// The rmsnorm_residual backward with the weight-gradient chunk of `chunk_T`
// rows' problem instead of its own T (so that a slice of rows writes the same
// chunk partials as the whole problem would); otherwise rmsnorm_residual_bwd_ex.
int residual_bwd_chunk_of(int64_t chunk_T, const uint16_t* g, int64_t ldg, const uint16_t* x, int64_t ldx,
                          const float* w, const float* rstd, const uint16_t* g_res, int64_t ldgr, uint16_t* dx,
                          int64_t lddx, void* ws, size_t ws_bytes, int64_t T, int64_t D, int zero_centered_gamma,
                          int dtype, cudaStream_t stream);

// rmsnorm_bwd's argument checks after the shape's and before the workspace's
// (pointers, row strides, alignment), in its order; RMSN_OK if all pass.
int bwd_check_args(const uint16_t* g, int64_t ldg, const uint16_t* x, int64_t ldx, const float* w,
                   const float* rstd, const uint16_t* dx, int64_t lddx, const float* dgamma, int64_t T, int64_t D);

// Launchers (return the launch's cudaError_t; arguments already validated).
// `m` is a Mode with its variant flags. The bf16 variants are instantiated in
// wide.cu / narrow.cu, the fp16 ones in wide_f16.cu / narrow_f16.cu.
cudaError_t launch_wide_fwd(int m, const FwdArgs& a, const RowCfg& c, cudaStream_t s);
cudaError_t launch_wide_bwd(int m, const BwdArgs& a, const RowCfg& c, cudaStream_t s);
cudaError_t launch_narrow_fwd(int m, const FwdArgs& a, const RowCfg& c, cudaStream_t s);
cudaError_t launch_narrow_bwd(int m, const BwdArgs& a, const RowCfg& c, cudaStream_t s);
cudaError_t launch_wide_fwd_f16(int m, const FwdArgs& a, const RowCfg& c, cudaStream_t s);
cudaError_t launch_wide_bwd_f16(int m, const BwdArgs& a, const RowCfg& c, cudaStream_t s);
cudaError_t launch_narrow_fwd_f16(int m, const FwdArgs& a, const RowCfg& c, cudaStream_t s);
cudaError_t launch_narrow_bwd_f16(int m, const BwdArgs& a, const RowCfg& c, cudaStream_t s);
cudaError_t launch_dgamma_reduce(const float* partials, int64_t nchunks, int D, float* out,
                                 cudaStream_t s);

// Device properties, cached per device.
int sm_count();
// The current context's unique id (false if none is current or the driver
// cannot say); see api.cu.
bool current_context_id(unsigned long long* id);
cudaError_t ensure_smem_attr(const void* kernel, int bytes);
int ctas_per_sm(const void* kernel, int threads, int smem_bytes);
// Clusters of two CTAs of `kernel` that can be resident at once.
int pair_clusters(const void* kernel, int threads, int smem_bytes);

// Error-word access for each kernel translation unit.
cudaError_t wide_read_error(unsigned* flags, bool clear);
cudaError_t narrow_read_error(unsigned* flags, bool clear);
cudaError_t selftest_read_error(unsigned* flags, bool clear);
cudaError_t wide_f16_read_error(unsigned* flags, bool clear);
cudaError_t narrow_f16_read_error(unsigned* flags, bool clear);

// Tensor-map encoding through the driver entry point (no libcuda link needed).
// Rows of 16-bit activations (bf16, or fp16 if `f16`): box = [box_rows][D].
// Vector of fp32: box = [box].
cudaError_t encode_rows_2d(CUtensorMap* map, const void* base, int64_t T, int D, int64_t ld_elems,
                           int box_rows, bool f16);
cudaError_t encode_vec_1d(CUtensorMap* map, const float* base, int64_t T, int box);

}  // namespace rmsn
