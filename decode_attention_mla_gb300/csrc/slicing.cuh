// slicing.cuh -- how the attended entries of one request are cut into split
// slices.  Used by the partial kernel (which computes the slices) and by the
// combine kernel (which skips the slices that are empty), so both agree.
#pragma once

#include "mla_internal.h"

namespace mla {

// Entries of request b: the dense context n_ctx = d_pos[b] + 1 clamped to the
// rows that exist past the request's first row, or the sparse list length.
__device__ __forceinline__ long long request_entries(int sparse, int topk, const int* d_pos,
                                                     const long long* row_offset, long long kv_rows, int b,
                                                     long long* base_out) {
    const long long base = row_offset ? row_offset[b] : 0;
    *base_out = base;
    if (sparse) return topk;
    long long n = static_cast<long long>(d_pos[b]) + 1;   // n_ctx = *d_pos + 1
    const long long cap = kv_rows - base;
    if (n > cap) n = cap;
    if (n < 0) n = 0;
    return n;
}

// Entries per slice: ceil(n / S) rounded up to a whole number of granules
// (the kernel's row step: 32 for the warp-MMA kernel, 16 for tcgen05).
__host__ __device__ __forceinline__ long long slice_entries(long long n, int splits, int granule) {
    long long per = (n + splits - 1) / splits;
    return (per + granule - 1) / granule * granule;
}

}  // namespace mla
