// Workspace sizing over a range of row counts.
//
// rmsnorm_bwd_workspace_bytes(T, D) is not monotone in T: where the wide
// backward's weight-gradient chunk is shortened so that chunks fill whole
// rounds of its grid (wide_chunk_rows), a larger T can need fewer partial rows
// than a smaller one. A caller that keeps one workspace for every T up to a
// maximum needs the largest size over that range, which this query returns.
#include "common.cuh"
#include "kernels.h"

extern "C" size_t rmsnorm_bwd_workspace_bytes_max(int64_t T_max, int64_t D) {
    const size_t at_max = T_max > 0 ? rmsnorm_bwd_workspace_bytes(T_max, D) : 0;
    if (at_max == 0) return 0;  // T_max <= 0 or an unsupported D
    if (rmsn::row_cfg(static_cast<int>(D)).narrow) return at_max;  // fixed chunks: the size grows with T
    // Chunks are shortened only while 32-row chunks fill fewer than ten rounds
    // of the 304-CTA grid (from ten rounds on, even a nearly empty last round
    // leaves them over 90 % full), in fact only for T <= 78784; beyond, the
    // size grows with T and exceeds every size below. Scanning the first
    // 131072 row counts covers that band.
    size_t best = at_max;
    const int64_t scan_to = T_max < 131072 ? T_max : 131072;
    for (int64_t t = 1; t <= scan_to; ++t) {
        const size_t b = rmsnorm_bwd_workspace_bytes(t, D);
        if (b > best) best = b;
    }
    return best;
}
