// mla_combine.cu -- log-sum-exp merge of the split partials.
//
// For every (request, head):  M = max_s lse_s,  lse = M + ln sum_s exp(lse_s - M),
// out = sum_s exp(lse_s - lse) * o_s, slices added in ascending order
// ("Graph-resident decode", Lecture 08, s.6: the merge is its own kernel with
// a grid wider than n_head, the slice sum runs in ascending slice order and
// there is no serial thread-0 prologue; here every lane of the warp computes
// the weights of its own slices and a fixed butterfly forms the normaliser).
//
// Grid (B*H, 512/128), one warp per CTA; each lane owns 4 consecutive output
// features (float4 loads of the partials, which stay in L2 between the two
// kernels).  An all-empty row set gives lse = -inf and out = 0.
#include <cmath>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"

namespace mla {
namespace {

__global__ void __launch_bounds__(32) mla_combine_kernel(const CombineParams p) {
    __shared__ float weight[MLA_MAX_SPLITS];
    grid_dependency_wait();          // the partials come from the preceding kernel
    allow_dependent_launch();
    const int bh = blockIdx.x;
    const int chunk = blockIdx.y;
    const int lane = threadIdx.x;
    const int S = p.splits;
    const float* lp = p.lse_part + static_cast<long long>(bh) * S;

    float mx = -INFINITY;
    for (int i = lane; i < S; i += 32) mx = fmaxf(mx, lp[i]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

    float sum = 0.f;
    if (mx != -INFINITY) {
        for (int i = lane; i < S; i += 32) sum += expf(lp[i] - mx);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float total = (mx == -INFINITY) ? -INFINITY : mx + logf(sum);
    for (int i = lane; i < S; i += 32) weight[i] = (mx == -INFINITY) ? 0.f : expf(lp[i] - total);
    __syncwarp();

    const float4* src = reinterpret_cast<const float4*>(p.o_part + static_cast<long long>(bh) * S * kDLatent) +
                        chunk * (kCombineChunk / 4) + lane;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int i = 0; i < S; ++i) {
        const float w = weight[i];
        const float4 v = src[static_cast<long long>(i) * (kDLatent / 4)];
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
    }
    reinterpret_cast<float4*>(p.out + static_cast<long long>(bh) * kDLatent)[chunk * (kCombineChunk / 4) + lane] = acc;
    if (chunk == 0 && lane == 0) p.lse[bh] = total;
}

}  // namespace

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
