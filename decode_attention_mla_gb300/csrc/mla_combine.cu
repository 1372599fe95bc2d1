// mla_combine.cu -- log-sum-exp merge of the split partials.
//
// For every (request, head):  M = max_s lse_s,  lse = M + ln sum_s exp(lse_s - M),
// out = sum_s exp(lse_s - lse) * o_s
// ("Graph-resident decode", Lecture 08, s.6: the merge is its own kernel with
// a grid wider than n_head and no serial thread-0 prologue).
//
// Grid (B*H, 512/128): a CTA merges 128 output features of one (request,
// head).  Only the slices that hold entries are read (the same slicing as the
// partial kernel).  The 8 warps take contiguous runs of those slices; each
// lane owns 4 consecutive features and loads its run's partials (16 at a time)
// before the weights are known, so those loads are in flight together with
// the lse loads.  Each warp adds its run in ascending slice order and the 8
// run sums are added in warp order: a fixed association, so the result is
// reproducible bit for bit.  An all-empty row set gives lse = -inf, out = 0.
#include <cmath>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"
#include "slicing.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kBatch = 16;                                       // partials a lane loads at once
static_assert(MLA_MAX_SPLITS <= kThreads, "one lse per thread");
static_assert(MLA_MAX_SPLITS <= kWarps * 2 * kBatch, "a warp's run fits two load batches");

__global__ void __launch_bounds__(kThreads) mla_combine_kernel(const CombineParams p) {
    __shared__ float weight[MLA_MAX_SPLITS];
    __shared__ float red_max[kWarps];
    __shared__ float red_sum[kWarps];
    __shared__ float4 part[kWarps][32];
    grid_dependency_wait();          // the partials come from the preceding kernel
    allow_dependent_launch();
    const int bh = blockIdx.x;
    const int b = bh / p.heads;
    const int chunk = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.splits;
    // only the slices that hold entries were written by the partial kernel
    long long base;
    const long long n = request_entries(p.sparse, p.topk, p.d_pos, p.row_offset, p.kv_rows, b, &base);
    const long long per = slice_entries(n, S, p.granule);
    const int S_used = per > 0 ? static_cast<int>(min(static_cast<long long>(S), (n + per - 1) / per)) : 0;
    const int run = (S_used + kWarps - 1) / kWarps;
    const int s0 = warp * run;
    const int s1 = min(S_used, s0 + run);

    // the first batch of this warp's partials, loaded before the weights are known
    const float4* src = reinterpret_cast<const float4*>(p.o_part + static_cast<long long>(bh) * S * kDLatent) +
                        chunk * (kCombineChunk / 4) + lane;
    float4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
        const int s = s0 + i;
        v[i] = (s < s1) ? src[static_cast<long long>(s) * (kDLatent / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // slice weights exp(lse_s - lse)
    const int t = threadIdx.x;
    const float ls = (t < S_used) ? p.lse_part[static_cast<long long>(bh) * S + t] : -INFINITY;
    float mx = ls;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red_max[warp] = mx;
    __syncthreads();
    mx = red_max[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, red_max[w]);
    float e = (mx == -INFINITY || t >= S_used) ? 0.f : expf(ls - mx);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) e += __shfl_xor_sync(0xffffffffu, e, off);
    if (lane == 0) red_sum[warp] = e;
    __syncthreads();
    float sum = red_sum[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) sum += red_sum[w];
    const float total = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
    if (t < S_used) weight[t] = (mx == -INFINITY) ? 0.f : expf(ls - total);
    __syncthreads();

    // this warp's run, ascending slice order
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
        const int s = s0 + i;
        if (s < s1) {
            const float w = weight[s];
            acc.x += w * v[i].x;
            acc.y += w * v[i].y;
            acc.z += w * v[i].z;
            acc.w += w * v[i].w;
        }
    }
    if (s0 + kBatch < s1) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int s = s0 + kBatch + i;
            v[i] = (s < s1) ? src[static_cast<long long>(s) * (kDLatent / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int s = s0 + kBatch + i;
            if (s < s1) {
                const float w = weight[s];
                acc.x += w * v[i].x;
                acc.y += w * v[i].y;
                acc.z += w * v[i].z;
                acc.w += w * v[i].w;
            }
        }
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float4 o = part[0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            const float4 q = part[w][lane];
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

int combine_block_threads() { return kThreads; }

cudaError_t launch_combine(const CombineParams& p, dim3 grid, int block, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mla_combine_kernel, p);
}

}  // namespace mla
