// mla_floor.cu -- floor probes of a decode call (declared in mla_floor.h):
// two empty kernels chained the way the partial and combine kernels are, one
// kernel that only reads a region of device memory over the whole GPU with
// bulk copies, and one that only gathers listed rows of a cache the way the
// sparse decode does.  Nothing here computes any part of the method; the
// measurement code times them beside the decode calls, so the share of a
// call's time that no kernel body can remove is measured, not assumed.
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "device_utils.cuh"
#include "mla_floor.h"

namespace {

constexpr int kMaxSmem = 227 * 1024;
constexpr int kCopyBytes = 32 * 1024;         // one bulk copy
constexpr int kCopies = 6;                    // copies in flight per CTA (192 KiB)
constexpr int kReadSmem = kCopies * kCopyBytes;
constexpr int kMaxDevices = 64;

__global__ void mla_floor_empty_kernel() {
    mla::grid_dependency_wait();
    mla::allow_dependent_launch();
}

// One warp per CTA; lane 0 issues the copies of the CTA's piece in rounds of
// up to kCopies, each round completing one phase of the CTA's mbarrier.
__global__ void __launch_bounds__(32, 1)
    mla_floor_read_kernel(const uint8_t* src, size_t bytes, size_t per_cta, unsigned* sink, int* status) {
    extern __shared__ __align__(128) uint8_t buf[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;                 // the bounded wait polls it; nothing raises it here
    if (threadIdx.x == 0) {
        mla::mbar_init(&bar, 1);
        abort_flag = 0;
        mla::mbar_init_fence();
    }
    __syncwarp();
    mla::grid_dependency_wait();
    mla::allow_dependent_launch();
    if (threadIdx.x != 0) return;
    const uint64_t policy = mla::l2_policy_evict_first();
    const size_t lo = static_cast<size_t>(blockIdx.x) * per_cta;
    const size_t hi = lo + per_cta < bytes ? lo + per_cta : bytes;
    unsigned acc = 0;
    uint32_t phase = 0;
    for (size_t off = lo; off < hi; off += kReadSmem) {
        const size_t left = hi - off;
        const uint32_t round = static_cast<uint32_t>(left < kReadSmem ? left : kReadSmem);
        mla::mbar_arrive_expect_tx(&bar, round);
        for (uint32_t k = 0; k < round; k += kCopyBytes) {
            const uint32_t n = round - k < kCopyBytes ? round - k : kCopyBytes;
            mla::bulk_copy_g2s(buf + k, src + off + k, n, &bar, policy);
        }
        if (!mla::mbar_wait_bounded(&bar, phase, &abort_flag)) {
            atomicCAS(status, 0, static_cast<int>(MLA_EDEVICE));
            mla::mbar_wait_bounded(&bar, phase, &abort_flag);   // the copies in flight, once more
            return;
        }
        phase ^= 1u;
        acc += *reinterpret_cast<const unsigned*>(buf);
    }
    sink[blockIdx.x] = acc;
}

// Row gather: one warp per CTA copies rows of a cache, one bulk copy per row,
// in rounds that fill half of the shared buffer each, two rounds in flight
// (one per half and mbarrier); each lane keeps the row numbers of its rows of
// the next round in registers, loaded while the current round is in flight.
constexpr int kGatherHalf = kReadSmem / 2;
constexpr int kGatherPerLane = 4;             // rows per lane and round (row_bytes >= kGatherHalf / 128)

__global__ void __launch_bounds__(32, 1)
    mla_floor_gather_kernel(const uint8_t* base, long long row_stride, long long kv_rows, uint32_t row_bytes,
                            const long long* rows, long long n_rows, long long per_cta, unsigned* sink,
                            int* status) {
    extern __shared__ __align__(128) uint8_t buf[];
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ int abort_flag;
    const int lane = threadIdx.x;
    if (lane == 0) {
        mla::mbar_init(&bar[0], 1);
        mla::mbar_init(&bar[1], 1);
        abort_flag = 0;
        mla::mbar_init_fence();
    }
    __syncwarp();
    mla::grid_dependency_wait();
    mla::allow_dependent_launch();
    const uint64_t policy = mla::l2_policy_evict_first();
    const int fit = kGatherHalf / static_cast<int>(row_bytes);
    const int per_round = fit < 32 * kGatherPerLane ? fit : 32 * kGatherPerLane;   // rows per round
    const long long lo = static_cast<long long>(blockIdx.x) * per_cta;
    const long long hi = lo + per_cta < n_rows ? lo + per_cta : n_rows;
    long long next[kGatherPerLane];
#pragma unroll
    for (int k = 0; k < kGatherPerLane; ++k) {
        const long long e = lo + lane + 32 * k;
        next[k] = (32 * k + lane < per_round && e < hi) ? rows[e] : -1;
    }
    unsigned acc = 0;
    bool ok = true;
    int round = 0;
    for (long long r0 = lo; r0 < hi && ok; r0 += per_round, ++round) {
        const int h = round & 1;
        if (round >= 2) {
            // the half is free once the round before last has landed
            ok = mla::mbar_wait_bounded(&bar[h], ((round - 2) >> 1) & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            acc += *reinterpret_cast<const unsigned*>(buf + h * kGatherHalf);
        }
        long long cur[kGatherPerLane];
        uint32_t mine = 0;
#pragma unroll
        for (int k = 0; k < kGatherPerLane; ++k) {
            cur[k] = next[k];
            if (cur[k] >= 0 && cur[k] < kv_rows) ++mine;
        }
        const uint32_t total = __reduce_add_sync(0xffffffffu, mine);
        if (lane == 0) mla::mbar_arrive_expect_tx(&bar[h], total * row_bytes);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < kGatherPerLane; ++k) {
            if (cur[k] >= 0 && cur[k] < kv_rows)
                mla::bulk_copy_g2s(buf + h * kGatherHalf + (32 * k + lane) * row_bytes, base + cur[k] * row_stride,
                                   row_bytes, &bar[h], policy);
        }
        // the next round's row numbers while this one is in flight
        const long long r1 = r0 + per_round;
#pragma unroll
        for (int k = 0; k < kGatherPerLane; ++k) {
            const long long e = r1 + lane + 32 * k;
            next[k] = (32 * k + lane < per_round && e < hi) ? rows[e] : -1;
        }
    }
    // every round issued lands before the CTA leaves (bounded, as above)
    for (int r = round - 2 < 0 ? 0 : round - 2; r < round; ++r) {
        const bool w = mla::mbar_wait_bounded(&bar[r & 1], (r >> 1) & 1, &abort_flag);
        if (!w) ok = false;
    }
    if (!ok) {
        if (lane == 0) atomicCAS(status, 0, static_cast<int>(MLA_EDEVICE));
        return;
    }
    if (lane == 0) sink[blockIdx.x] = acc + (round > 0 ? *reinterpret_cast<const unsigned*>(buf) : 0u);
}

std::atomic<int> g_floor_ready[kMaxDevices];
std::mutex g_floor_mutex;

// Shared-memory limits of the kernels, set once per device outside capture.
int floor_prepare(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MLA_ECUDA;
    }
    if (g_floor_ready[dev].load(std::memory_order_acquire)) return MLA_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ECUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return MLA_ENOTREADY;
    std::lock_guard<std::mutex> lock(g_floor_mutex);
    if (cudaFuncSetAttribute(mla_floor_empty_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(mla_floor_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kReadSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(mla_floor_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kReadSmem) !=
            cudaSuccess) {
        cudaGetLastError();
        return MLA_ECUDA;
    }
    g_floor_ready[dev].store(1, std::memory_order_release);
    return MLA_OK;
}

cudaLaunchConfig_t floor_config(int grid, int block, int smem, bool pdl, cudaStream_t stream,
                                cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

int launch_rc(cudaError_t e) {
    if (e == cudaSuccess) return MLA_OK;
    cudaGetLastError();
    return MLA_ECUDA;
}

bool valid_launch(int grid, int block, int smem) {
    return grid >= 1 && grid <= 65535 && block >= 32 && block <= 1024 && block % 32 == 0 && smem >= 0 &&
           smem <= kMaxSmem;
}

}  // namespace

extern "C" {

int mla_floor_empty_pair(int grid_a, int block_a, int smem_a, int grid_b, int block_b, int smem_b, int pdl,
                         void* stream) {
    if (!valid_launch(grid_a, block_a, smem_a) || !valid_launch(grid_b, block_b, smem_b) || (pdl != 0 && pdl != 1))
        return MLA_EINVAL;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int rc = floor_prepare(st);
    if (rc != MLA_OK) return rc;
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t a = floor_config(grid_a, block_a, smem_a, pdl != 0, st, &attr);
    cudaError_t e = cudaLaunchKernelEx(&a, mla_floor_empty_kernel);
    if (e != cudaSuccess) return launch_rc(e);
    cudaLaunchConfig_t b = floor_config(grid_b, block_b, smem_b, pdl != 0, st, &attr);
    return launch_rc(cudaLaunchKernelEx(&b, mla_floor_empty_kernel));
}

int mla_floor_read(const void* src, size_t bytes, int ctas, unsigned* sink, int* status, int pdl, void* stream) {
    if (!src || !sink || !status || bytes == 0 || ctas < 1 || ctas > 65535 || (pdl != 0 && pdl != 1))
        return MLA_EINVAL;
    if (bytes % 16 != 0 || reinterpret_cast<uintptr_t>(src) % 16 != 0 || reinterpret_cast<uintptr_t>(sink) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(status) % 4 != 0)
        return MLA_EALIGN;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int rc = floor_prepare(st);
    if (rc != MLA_OK) return rc;
    // equal pieces, 16-byte aligned (the last CTAs may get less, or nothing)
    const size_t per = (bytes / 16 + static_cast<size_t>(ctas) - 1) / static_cast<size_t>(ctas) * 16;
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = floor_config(ctas, 32, kReadSmem, pdl != 0, st, &attr);
    return launch_rc(cudaLaunchKernelEx(&cfg, mla_floor_read_kernel, static_cast<const uint8_t*>(src), bytes, per,
                                        sink, status));
}

int mla_floor_gather(const void* kv, long long kv_rows, long long row_stride, int row_bytes, const long long* rows,
                     long long n_rows, int ctas, unsigned* sink, int* status, int pdl, void* stream) {
    if (!kv || !rows || !sink || !status || kv_rows < 1 || n_rows < 1 || ctas < 1 || ctas > 65535 ||
        row_bytes < 16 || row_bytes > kGatherHalf || row_stride < row_bytes || (pdl != 0 && pdl != 1))
        return MLA_EINVAL;
    if (row_bytes % 16 != 0 || row_stride % 16 != 0 || reinterpret_cast<uintptr_t>(kv) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(rows) % 8 != 0 || reinterpret_cast<uintptr_t>(sink) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(status) % 4 != 0)
        return MLA_EALIGN;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int rc = floor_prepare(st);
    if (rc != MLA_OK) return rc;
    const long long per = (n_rows + ctas - 1) / ctas;     // list entries per CTA (the last CTAs may get fewer)
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = floor_config(ctas, 32, kReadSmem, pdl != 0, st, &attr);
    return launch_rc(cudaLaunchKernelEx(&cfg, mla_floor_gather_kernel, static_cast<const uint8_t*>(kv), row_stride,
                                        kv_rows, static_cast<uint32_t>(row_bytes), rows, n_rows, per, sink, status));
}

}  // extern "C"
