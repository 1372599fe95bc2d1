// mla_combine.cu -- log-sum-exp merge of the split partials.
//
// For every (request, head):  M = max_s lse_s,  lse = M + ln sum_s exp(lse_s - M),
// out = sum_s exp(lse_s - lse) * o_s
// ("Graph-resident decode", Lecture 08, s.6: the merge is its own kernel with
// a grid wider than n_head and no serial thread-0 prologue).
//
// Grid (ceil(B*H / U), 512/128) of 8-warp CTAs: a unit of W = 1, 2, 4 or 8
// warps (fewer for fewer slices; U = 8 / W units per CTA, so batched decode
// with short split lists runs few, full CTAs) merges 128 output features of
// one (request, head) over all S slices (a slice without entries carries lse = -inf and
// o = 0, written by the partial kernel, so the merge needs neither the
// context length nor the slicing).  The 8 warps take contiguous runs of
// slices; each lane owns 4 consecutive features and loads its run's partials
// (all of a run of up to 20 at once, else 16 at a time) before the weights
// are known, so those loads are in flight together with the lse loads.  The max and the sum of exponentials are taken
// in one pass of (max, sum) pairs.  Each warp adds its run in ascending slice
// order and the run sums are added in warp order: a fixed association, so
// the result is reproducible bit for bit.  An all-empty row set gives
// lse = -inf, out = 0.
#include <algorithm>
#include <cmath>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kWarps = 8;                                        // most warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kBatch = 16;                                       // partials a lane loads at once (two batches)
constexpr int kWideBatch = 20;                                   // ... or all of a run of up to 20, at once
static_assert(MLA_MAX_SPLITS <= kThreads, "one lse per thread of an 8-warp unit");
static_assert(MLA_MAX_SPLITS <= kWarps * 2 * kBatch, "a warp's run fits two load batches");

template <int W, int B>
__global__ void __launch_bounds__(kThreads) mla_combine_kernel(const CombineParams p, int rows) {
    __shared__ float weight[kThreads];                  // unit u's weights at u * 32 * unit_warps
    __shared__ float red_max[kWarps];
    __shared__ float red_sum[kWarps];
    __shared__ float4 part[kWarps][32];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // W = warps per (request, head): 1, 2, 4 or 8
    const int unit = warp / W;
    const int wl = warp - unit * W;                    // warp within the unit
    const int bh = blockIdx.x * (kWarps / W) + unit;   // (request, head) of this unit
    const bool live = bh < rows;
    const int chunk = blockIdx.y;
    const int S = p.splits;
    // while the partial kernel finishes: the lines (and address translations)
    // this thread reads first
    if (live) {
        if (threadIdx.x % 32 == 0) prefetch_l2(p.lse_part + static_cast<long long>(bh) * S);
        const int s = (S + W - 1) / W * wl;
        if (s < S)
            prefetch_l2(p.o_part + (static_cast<long long>(bh) * S + s) * kDLatent + chunk * kCombineChunk + 4 * lane);
    }
    grid_dependency_wait();          // the partials come from the preceding kernel
    allow_dependent_launch();
    // fused state update (dense): the partial kernel took each request's new row
    // from new_rows; now that it is done reading the cache, CTA (0, 0) writes the
    // row to cache row d_pos[b] (for the steps after this one) and advances
    // d_pos.  Nothing in this grid reads either, and the next kernel on the
    // stream waits for this grid to finish before it does.
    if (p.new_rows && blockIdx.x == 0 && blockIdx.y == 0) {
        constexpr int kUnits = kRowBytes / 16;
        for (int i = threadIdx.x; i < p.batch * kUnits; i += kThreads) {
            const int b = i / kUnits;
            const int u = i - b * kUnits;
            const long long row = (p.row_offset ? p.row_offset[b] : 0) + p.d_pos[b];
            if (row >= 0 && row < p.kv_rows)
                reinterpret_cast<uint4*>(p.kv + row * p.row_stride)[u] =
                    reinterpret_cast<const uint4*>(p.new_rows + static_cast<long long>(b) * kDRow)[u];
        }
        __syncthreads();             // every read of d_pos above precedes the increments
        if (p.advance)
            for (int b = threadIdx.x; b < p.batch; b += kThreads) p.d_pos_rw[b] += 1;
    }
    // Every slice holds a partial (the partial kernels write lse = -inf, o = 0
    // for slices without entries), so nothing here depends on the context length.
    const int tu = wl * 32 + lane;                     // thread within the unit: 32 * W >= S
    const float ls = (live && tu < S) ? p.lse_part[static_cast<long long>(bh) * S + tu] : -INFINITY;
    const int run = (S + W - 1) / W;                   // <= 2 * B (the host sizes W and B that way)
    const int s0 = wl * run;
    const int s1 = live ? min(S, s0 + run) : s0;

    // the first batch of this warp's partials, loaded before the weights are known
    const float4* src = reinterpret_cast<const float4*>(p.o_part + static_cast<long long>(bh) * S * kDLatent) +
                        chunk * (kCombineChunk / 4) + lane;
    float4 v[B];
#pragma unroll
    for (int i = 0; i < B; ++i) {
        const int s = s0 + i;
        v[i] = (s < s1) ? src[static_cast<long long>(s) * (kDLatent / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // (max, sum of exp relative to it) over the slices in one pass: a warp
    // butterfly on the pairs (both partners form the same, commutative merge,
    // so every lane ends with the same bits), then the unit's warps in order
    float m = ls;
    float e = (ls == -INFINITY) ? 0.f : 1.f;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float e2 = __shfl_xor_sync(0xffffffffu, e, off);
        const float nm = fmaxf(m, m2);
        e = (nm == -INFINITY) ? 0.f : e * expf(m - nm) + e2 * expf(m2 - nm);
        m = nm;
    }
    if (lane == 0) {
        red_max[warp] = m;
        red_sum[warp] = e;
    }
    __syncthreads();
    const int w0 = unit * W;
    float mx = red_max[w0];
#pragma unroll
    for (int w = 1; w < W; ++w) mx = fmaxf(mx, red_max[w0 + w]);
    float sum = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
        for (int w = 0; w < W; ++w) sum += red_sum[w0 + w] * expf(red_max[w0 + w] - mx);
    }
    const float total = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
    float* wt = weight + unit * 32 * W;
    if (tu < S) wt[tu] = (mx == -INFINITY) ? 0.f : expf(ls - total);
    __syncthreads();

    // this warp's run, ascending slice order
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < B; ++i) {
        const int s = s0 + i;
        if (s < s1) {
            const float w = wt[s];
            acc.x += w * v[i].x;
            acc.y += w * v[i].y;
            acc.z += w * v[i].z;
            acc.w += w * v[i].w;
        }
    }
    if (s0 + B < s1) {
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int s = s0 + B + i;
            v[i] = (s < s1) ? src[static_cast<long long>(s) * (kDLatent / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < B; ++i) {
            const int s = s0 + B + i;
            if (s < s1) {
                const float w = wt[s];
                acc.x += w * v[i].x;
                acc.y += w * v[i].y;
                acc.z += w * v[i].z;
                acc.w += w * v[i].w;
            }
        }
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (wl == 0 && live) {
        float4 o = part[w0][lane];
#pragma unroll
        for (int w = 1; w < W; ++w) {
            const float4 q = part[w0 + w][lane];
            o.x += q.x;
            o.y += q.y;
            o.z += q.z;
            o.w += q.w;
        }
        reinterpret_cast<float4*>(p.out + static_cast<long long>(bh) * kDLatent)[chunk * (kCombineChunk / 4) + lane] = o;
        if (chunk == 0 && lane == 0) p.lse[bh] = total;
    }
}

}  // namespace

// Warps per (request, head) for S slices: enough threads for one lse each and
// at most 20 slices per warp (one load batch) where 8 warps allow it, rounded
// up to a power of two so that 8 / W units share a CTA of 8 warps (measured
// against 16-slice runs: a dense H=128 decode step at T=32832, 37.65 -> 36.59
// us; H=16 T=131072, 30.80 -> 30.51 us per call).
int combine_unit_warps(int splits) {
    const int need = std::max((splits + 31) / 32, std::min((splits + kWideBatch - 1) / kWideBatch, kWarps));
    int w = 1;
    while (w < need) w *= 2;
    return w;
}
int combine_block_threads() { return kThreads; }
int combine_grid_rows(int rows, int splits) {
    const int per_cta = kWarps / combine_unit_warps(splits);
    return (rows + per_cta - 1) / per_cta;
}

// Shared memory reserved (unused) by each combine CTA of a grid no larger than
// the GPU, so that no two share an SM: launched early (programmatic dependent
// launch) while the partial kernel holds most SMs, the CTAs would otherwise
// pile onto the few idle ones and load the partials through a fraction of
// the GPU.  Larger grids run in waves anyway and are launched without it.
constexpr int kSpreadSmemBytes = 120 * 1024;

cudaError_t combine_prepare() {
    for (auto fn : {mla_combine_kernel<1, kBatch>, mla_combine_kernel<2, kBatch>, mla_combine_kernel<4, kBatch>,
                    mla_combine_kernel<8, kBatch>, mla_combine_kernel<1, kWideBatch>, mla_combine_kernel<2, kWideBatch>,
                    mla_combine_kernel<4, kWideBatch>, mla_combine_kernel<8, kWideBatch>}) {
        const cudaError_t e =
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpreadSmemBytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_combine(const CombineParams& p, dim3 grid, int block, bool pdl, bool spread,
                           cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = spread ? kSpreadSmemBytes : 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const int rows = p.batch * p.heads;
    const int w = combine_unit_warps(p.splits);
    const int run = (p.splits + w - 1) / w;
    if (run > kBatch && run <= kWideBatch) {
        // a run of 17-20 slices: one batch of 20 loads instead of two dependent ones
        switch (w) {
            case 1: return cudaLaunchKernelEx(&cfg, mla_combine_kernel<1, kWideBatch>, p, rows);
            case 2: return cudaLaunchKernelEx(&cfg, mla_combine_kernel<2, kWideBatch>, p, rows);
            case 4: return cudaLaunchKernelEx(&cfg, mla_combine_kernel<4, kWideBatch>, p, rows);
            default: return cudaLaunchKernelEx(&cfg, mla_combine_kernel<8, kWideBatch>, p, rows);
        }
    }
    switch (w) {
        case 1: return cudaLaunchKernelEx(&cfg, mla_combine_kernel<1, kBatch>, p, rows);
        case 2: return cudaLaunchKernelEx(&cfg, mla_combine_kernel<2, kBatch>, p, rows);
        case 4: return cudaLaunchKernelEx(&cfg, mla_combine_kernel<4, kBatch>, p, rows);
        default: return cudaLaunchKernelEx(&cfg, mla_combine_kernel<8, kBatch>, p, rows);
    }
}

}  // namespace mla
