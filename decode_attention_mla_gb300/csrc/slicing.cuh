// slicing.cuh -- how the attended entries of one request are cut into split
// slices.  Used by the partial kernel (which computes the slices) and by the
// combine kernel (which skips the slices that are empty), so both agree.
#pragma once

#include <cmath>

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

// The same cut in 32-bit arithmetic for counts below 2^31 with a power-of-two
// granule (the tcgen05 kernel's item decode runs on the critical path of
// every CTA's first load; 64-bit division there costs hundreds of cycles).
__device__ __forceinline__ uint32_t slice_entries_u32(uint32_t n, uint32_t splits, uint32_t granule_pow2) {
    const uint32_t per = (n + splits - 1u) / splits;
    return (per + granule_pow2 - 1u) & ~(granule_pow2 - 1u);
}

// A slice without entries still gets its partial written: lse_s = -inf and
// o_s = 0 for the 16 heads of the item, so the combine reads every slice
// without re-deriving which ones are empty.  row0 = the partial row of head 0
// ((b * H + first head) * S + s); `tid` / `nthreads` split the stores.
__device__ __forceinline__ void write_empty_partial(float* o_part, float* lse_part, long long row0, int splits,
                                                    int tid, int nthreads) {
    constexpr int kVec = kDLatent / 4;                   // float4 per partial row
    for (int i = tid; i < kHeadGroup * kVec; i += nthreads) {
        const int h = i / kVec;
        const int v = i - h * kVec;
        reinterpret_cast<float4*>(o_part + (row0 + static_cast<long long>(h) * splits) * kDLatent)[v] =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < kHeadGroup) lse_part[row0 + static_cast<long long>(tid) * splits] = -INFINITY;
}

}  // namespace mla
