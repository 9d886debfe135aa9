// Workspace sizing over a range of row counts.
//
// rmsnorm_bwd_workspace_bytes(T, D) is not monotone in T: where the wide
// backward's weight-gradient chunk is shortened so that chunks fill whole
// rounds of its grid (wide_chunk_rows), a larger T can need fewer partial rows
// than a smaller one. A caller that keeps one workspace for every T up to a
// maximum needs the largest size over that range, which this query returns
// in closed form (wide_chunks_max in api.cu; no scan over T).
#include "common.cuh"
#include "kernels.h"

extern "C" size_t rmsnorm_bwd_workspace_bytes_max(int64_t T_max, int64_t D) {
    const size_t at_max = T_max > 0 ? rmsnorm_bwd_workspace_bytes(T_max, D) : 0;
    if (at_max == 0) return 0;  // T_max <= 0 or an unsupported D
    if (rmsn::row_cfg(static_cast<int>(D)).narrow) return at_max;  // fixed chunks: the size grows with T
    return static_cast<size_t>(rmsn::wide_chunks_max(T_max, static_cast<int>(D))) * static_cast<size_t>(D) * 4u;
}
