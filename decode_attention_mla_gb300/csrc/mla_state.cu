// mla_state.cu -- the two device-side state updates of graph-resident decode
// ("Graph-resident decode", Lecture 08, s.2):
//   append : the new token's cache row is written at the row derived on the
//            device from d_pos, so every replay of a captured graph writes a
//            different row (a host-computed row pointer would be frozen at
//            capture and rewrite one row forever);
//   advance: d_pos += 1 inside the captured region.
#include "device_utils.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kAppendThreads = 96;   // 72 x 16-byte pieces per 1152-byte row

__global__ void __launch_bounds__(kAppendThreads) mla_append_kernel(const AppendParams p) {
    grid_dependency_wait();          // d_pos may come from the preceding advance
    allow_dependent_launch();
    const int b = blockIdx.x;
    const long long base = p.row_offset ? p.row_offset[b] : 0;
    const long long row = base + p.d_pos[b];
    if (row < 0 || row >= p.kv_rows) return;
    const uint4* src = reinterpret_cast<const uint4*>(p.new_rows + static_cast<long long>(b) * kDRow);
    uint4* dst = reinterpret_cast<uint4*>(p.kv + row * p.row_stride);
    for (int i = threadIdx.x; i < kRowBytes / 16; i += blockDim.x) dst[i] = src[i];
}

__global__ void __launch_bounds__(256) mla_advance_kernel(int* d_pos, int batch) {
    grid_dependency_wait();          // readers of d_pos earlier on the stream must be done
    allow_dependent_launch();
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < batch; b += gridDim.x * blockDim.x) d_pos[b] += 1;
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, bool pdl, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, bool pdl, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg(dim3(p.batch), dim3(kAppendThreads), pdl, stream, attr);
    return cudaLaunchKernelEx(&cfg, mla_append_kernel, p);
}

cudaError_t launch_advance(int* d_pos, int batch, bool pdl, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    const int blocks = (batch + 255) / 256;
    cudaLaunchConfig_t cfg = make_cfg(dim3(blocks < 1 ? 1 : blocks), dim3(256), pdl, stream, attr);
    return cudaLaunchKernelEx(&cfg, mla_advance_kernel, d_pos, batch);
}

}  // namespace mla
