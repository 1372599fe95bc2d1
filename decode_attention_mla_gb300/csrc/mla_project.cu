// mla_project.cu -- projection of the merged latent through wv_b:
//   y[b][h][v] = sum_r latent[b][h][r] * wv_b[h][v][r]      (r = 0 .. 511)
// ("Graph-resident decode", Lecture 08, s.6: the merge writes the normalised
// latent to scratch and a second kernel, grid (n_head, 16), projects it; each
// block owns a slice of v_dim and reads only its own wv_b rows, and the
// projection dot strides r by 32 across the warp.)
//
// Grid (H, 16, ceil(B / kBatchPerBlock)); a block has v_dim / 16 warps and
// warp w computes output v = blockIdx.y * (v_dim / 16) + w: lane l holds the
// 16 weights wv_b[h][v][256j + 8l + e] (j = 0, 1; e = 0 .. 7: two 16-byte
// loads, the warp reading its 1 KB row in two coalesced 512-byte sweeps),
// forms the sum over (j, e) in ascending order against the latent and the
// warp adds the 32 lane sums with a fixed butterfly, for each request b of
// the block.  (The pages stride r by 32 across the warp; 8-element groups
// keep every load 16 bytes wide.)  Every block reads 1/16 of its head's wv_b
// once; the weights stay in registers across the requests.  fp32 arithmetic,
// fixed association: the result is reproducible bit for bit.
#include "device_utils.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kSlices = 16;                  // v_dim slices (grid y)
constexpr int kRPerLane = kDLatent / 32;     // 16 latent entries per lane: two groups of 8
constexpr int kBatchPerBlock = 8;            // requests per block (grid z covers the rest)

__global__ void __launch_bounds__(1024) mla_project_kernel(const ProjectParams p) {
    grid_dependency_wait();                  // the latent comes from the preceding merge
    allow_dependent_launch();
    const int h = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int v = blockIdx.y * (p.v_dim / kSlices) + warp;
    const uint4* wrow =
        reinterpret_cast<const uint4*>(p.wv_b + (static_cast<long long>(h) * p.v_dim + v) * kDLatent);
    float wk[kRPerLane];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint4 u = wrow[32 * j + lane];           // bf16 r = 256j + 8*lane .. +7
        const uint32_t part[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {                  // exact widening: bf16 is the top half of fp32
            wk[8 * j + 2 * e] = __uint_as_float(part[e] << 16);
            wk[8 * j + 2 * e + 1] = __uint_as_float(part[e] & 0xffff0000u);
        }
    }
    const int b0 = blockIdx.z * kBatchPerBlock;
    const int b1 = min(p.batch, b0 + kBatchPerBlock);
    for (int b = b0; b < b1; ++b) {
        const float4* lat =
            reinterpret_cast<const float4*>(p.latent + (static_cast<long long>(b) * p.heads + h) * kDLatent);
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float4 a = lat[64 * j + 2 * lane];
            const float4 c = lat[64 * j + 2 * lane + 1];
            acc += a.x * wk[8 * j + 0];
            acc += a.y * wk[8 * j + 1];
            acc += a.z * wk[8 * j + 2];
            acc += a.w * wk[8 * j + 3];
            acc += c.x * wk[8 * j + 4];
            acc += c.y * wk[8 * j + 5];
            acc += c.z * wk[8 * j + 6];
            acc += c.w * wk[8 * j + 7];
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) p.y[(static_cast<long long>(b) * p.heads + h) * p.v_dim + v] = acc;
    }
}

}  // namespace

cudaError_t launch_project(const ProjectParams& p, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.heads, kSlices, (p.batch + kBatchPerBlock - 1) / kBatchPerBlock);
    cfg.blockDim = dim3(32 * (p.v_dim / kSlices), 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mla_project_kernel, p);
}

}  // namespace mla
