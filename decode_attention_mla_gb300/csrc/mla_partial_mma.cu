// mla_partial_mma.cu -- split-KV MLA decode partial, head-group-16 kernel.
//
// One CTA computes the online-softmax partial of one (request b, head group
// of 16 heads, context slice s) ("Launch Geometry", Lecture 04, s.1 and s.8:
// the context split is the axis manufactured for batch-1 decode; "Graph-
// resident decode", Lecture 08, s.6: per-slice partials merged afterwards).
//
// Data flow per 32-row stage:
//   producer warp : each lane moves one 1152-byte cache row into shared
//                   memory with a bulk copy (TMA engine), completion counted
//                   on the stage's mbarrier.  Dense rows are contiguous
//                   positions base + e; sparse rows are base + indices[b][e]
//                   (a gather, "The Commit That Changed Direction").  Rows
//                   that are past the slice or out of range are zero-filled
//                   and masked.
//   4 MMA warps   : scores S[16 heads x 32 rows] = Q . K^T with
//                   mma.m16n8k16 (bf16 in, fp32 accumulate); the 576-wide
//                   contraction is split across the warps (144 features
//                   each, Q fragments held in registers) and the four
//                   partial score tiles are summed in fixed warp order.
//                   Every warp then applies the same online-softmax update
//                   (base-2 exponent, quad shuffles for row max / row sum)
//                   and accumulates O[16 x 128 features of its own] += P . V
//                   with V = the latent c rows and P as a bf16 hi + lo pair
//                   (two MMAs), so P keeps ~16 significant bits.
// Epilogue: o_part = O / l (normalised) and lse_part = ln(sum exp(s)), or
// (0, -inf) for an empty slice.  No floating-point atomics: the result is a
// pure function of the inputs and the split count.
#include <cfloat>
#include <cmath>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kStages = 2;                                // pipeline depth (32-row stages)
constexpr int kComputeWarps = 4;
constexpr int kThreads = (kComputeWarps + 1) * 32;        // + one producer warp
constexpr int kSmemRow = kRowBytes + 16;                  // padding: 8 rows x 16 B hit 32 distinct banks
constexpr int kNT = kStageRows / 8;                       // score n-tiles of 8 rows
constexpr int kKSteps = kDRow / 16;                       // 36 k-steps over the 576 features
constexpr int kKStepsPerWarp = kKSteps / kComputeWarps;   // 9
constexpr int kFeatPerWarp = kDLatent / kComputeWarps;    // 128 output features per warp
constexpr int kPVTiles = kFeatPerWarp / 8;                // 16
constexpr int kPSteps = kStageRows / 16;                  // 2 k-steps of P . V per stage
constexpr float kLn2 = 0.6931471805599453f;

static_assert(kKSteps % kComputeWarps == 0, "feature split");
static_assert(kNT % 2 == 0 && kPVTiles % 2 == 0, "ldmatrix.x4 pairs");

struct __align__(128) SharedStorage {
    uint8_t kv[kStages][kStageRows][kSmemRow];
    float4 red[2][kComputeWarps][kNT][32];                // per-warp partial scores
    int valid[kStages][kStageRows];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t red_bar[2];
    int abort_flag;
};

__device__ __forceinline__ uint32_t ld_u32(const uint16_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ void raise_device_error(SharedStorage& sh, int* status) {
    sh.abort_flag = 1;
    if (status) atomicCAS(status, 0, static_cast<int>(MLA_EDEVICE));
}

__global__ void __launch_bounds__(kThreads, 2) mla_partial_mma_kernel(const PartialParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    SharedStorage& sh = *reinterpret_cast<SharedStorage*>(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hg = blockIdx.x;
    const int s = blockIdx.y;
    const int b = blockIdx.z;
    const int S = p.splits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], 32);
            mbar_init(&sh.empty[i], kComputeWarps);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&sh.red_bar[i], kComputeWarps * 32);
        sh.abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    // Inputs (d_pos, cache rows, indices) may be written by the kernel before
    // this one on the stream: wait for it before any global read.
    grid_dependency_wait();
    allow_dependent_launch();

    // ---- this CTA's slice of the context (or of the index list) ----------
    const long long base = p.row_offset ? p.row_offset[b] : 0;
    long long n_entries;
    if (!p.sparse) {
        long long n = static_cast<long long>(p.d_pos[b]) + 1;   // n_ctx = *d_pos + 1
        const long long cap = p.kv_rows - base;
        if (n > cap) n = cap;
        if (n < 0) n = 0;
        n_entries = n;
    } else {
        n_entries = p.topk;
    }
    long long per = (n_entries + S - 1) / S;
    per = (per + kStageRows - 1) / kStageRows * kStageRows;
    long long e0 = static_cast<long long>(s) * per;
    long long e1 = e0 + per;
    if (e1 > n_entries) e1 = n_entries;
    if (e0 > e1) e0 = e1;
    const int n_stages = static_cast<int>((e1 - e0 + kStageRows - 1) / kStageRows);

    if (warp == kComputeWarps) {
        // =========================== producer ===========================
        const int seg_len = p.sparse ? p.cache_len[b] : 0;
        const uint64_t policy = l2_policy_evict_first();
        int issued = 0;
        for (int it = 0; it < n_stages; ++it) {
            const int slot = it % kStages;
            if (it >= kStages) {
                if (!mbar_wait_bounded(&sh.empty[slot], ((it / kStages) - 1) & 1, &sh.abort_flag)) {
                    if (lane == 0) raise_device_error(sh, p.status);
                    break;
                }
            }
            const long long e = e0 + static_cast<long long>(it) * kStageRows + lane;
            bool valid = false;
            long long row = 0;
            if (e < e1) {
                if (!p.sparse) {
                    row = base + e;
                    valid = (row >= 0 && row < p.kv_rows);
                } else {
                    const int id = p.indices[static_cast<long long>(b) * p.topk + e];
                    if (id >= 0 && id < seg_len) {
                        row = base + id;
                        valid = (row >= 0 && row < p.kv_rows);
                    }
                }
            }
            uint8_t* dst = sh.kv[slot][lane];
            sh.valid[slot][lane] = valid ? 1 : 0;
            if (!valid) {
                // masked rows still feed P . V (with p = 0): keep them finite
                uint4* z = reinterpret_cast<uint4*>(dst);
#pragma unroll 8
                for (int i = 0; i < kRowBytes / 16; ++i) z[i] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sh.full[slot], valid ? static_cast<uint32_t>(kRowBytes) : 0u);
            if (valid) {
                bulk_copy_g2s(dst, p.kv + row * p.row_stride, kRowBytes, &sh.full[slot], policy);
            }
            issued = it + 1;
        }
        // Never retire the CTA with copies into its shared memory in flight.
        if (lane == 0) {
            for (int slot = 0; slot < kStages && slot < issued; ++slot) {
                const int last_use = (issued - 1 - slot) / kStages;
                volatile int never = 0;
                if (!mbar_wait_bounded(&sh.full[slot], last_use & 1, &never)) raise_device_error(sh, p.status);
            }
        }
        return;
    }

    // ============================ MMA warps ===============================
    const int w = warp;
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int h0 = hg * kHeadGroup;

    // Q fragments (rows = heads h0 + g and h0 + g + 8) for this warp's 9 k-steps
    uint32_t qa[kKStepsPerWarp][4];
    {
        const uint16_t* qb = p.q + (static_cast<long long>(b) * p.heads + h0) * kDRow;
#pragma unroll
        for (int kk = 0; kk < kKStepsPerWarp; ++kk) {
            const int col = (w * kKStepsPerWarp + kk) * 16 + 2 * tq;
            qa[kk][0] = ld_u32(qb + g * kDRow + col);
            qa[kk][1] = ld_u32(qb + (g + 8) * kDRow + col);
            qa[kk][2] = ld_u32(qb + g * kDRow + col + 8);
            qa[kk][3] = ld_u32(qb + (g + 8) * kDRow + col + 8);
        }
    }

    float o[kPVTiles][4];
#pragma unroll
    for (int i = 0; i < kPVTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};   // running max, base-2 units
    float l_run[2] = {0.f, 0.f};               // running sum of 2^(s - m_run)
    const int f_base = w * kFeatPerWarp;
    const int lrow = lane & 7;
    const int lmat = lane >> 3;

    for (int it = 0; it < n_stages; ++it) {
        const int slot = it % kStages;
        if (!mbar_wait_bounded(&sh.full[slot], (it / kStages) & 1, &sh.abort_flag)) {
            if (lane == 0) raise_device_error(sh, p.status);
            break;
        }
        const uint32_t kv_base = smem_u32(&sh.kv[slot][0][0]);

        // ---- partial scores over this warp's 144 features ----------------
        float acc[kNT][4];
#pragma unroll
        for (int j = 0; j < kNT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kKStepsPerWarp; ++kk) {
            const int col_bytes = (w * kKStepsPerWarp + kk) * 32;
#pragma unroll
            for (int j = 0; j < kNT; j += 2) {
                const int row = 8 * j + lrow + ((lmat >> 1) << 3);
                const uint32_t addr = kv_base + row * kSmemRow + col_bytes + ((lmat & 1) << 4);
                uint32_t bf[4];
                ldmatrix_x4(bf, addr);
                mma_bf16_16816(acc[j], qa[kk], bf[0], bf[1]);
                mma_bf16_16816(acc[j + 1], qa[kk], bf[2], bf[3]);
            }
        }

        // ---- sum the four warps' partial scores (fixed order) -------------
        const int rb = it & 1;
#pragma unroll
        for (int j = 0; j < kNT; ++j) sh.red[rb][w][j][lane] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
        mbar_arrive(&sh.red_bar[rb]);
        if (!mbar_wait_bounded(&sh.red_bar[rb], (it >> 1) & 1, &sh.abort_flag)) {
            if (lane == 0) raise_device_error(sh, p.status);
            break;
        }
        float sc[kNT][4];
#pragma unroll
        for (int j = 0; j < kNT; ++j) {
            const float4 v0 = sh.red[rb][0][j][lane];
            const float4 v1 = sh.red[rb][1][j][lane];
            const float4 v2 = sh.red[rb][2][j][lane];
            const float4 v3 = sh.red[rb][3][j][lane];
            sc[j][0] = ((v0.x + v1.x) + v2.x) + v3.x;
            sc[j][1] = ((v0.y + v1.y) + v2.y) + v3.y;
            sc[j][2] = ((v0.z + v1.z) + v2.z) + v3.z;
            sc[j][3] = ((v0.w + v1.w) + v2.w) + v3.w;
        }

        // ---- online softmax (identical in every MMA warp) -----------------
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < kNT; ++j) {
            const int c0 = 8 * j + 2 * tq;
            const bool v0 = sh.valid[slot][c0] != 0;
            const bool v1 = sh.valid[slot][c0 + 1] != 0;
            sc[j][0] = v0 ? sc[j][0] * p.scale_log2 : -INFINITY;
            sc[j][1] = v1 ? sc[j][1] * p.scale_log2 : -INFINITY;
            sc[j][2] = v0 ? sc[j][2] * p.scale_log2 : -INFINITY;
            sc[j][3] = v1 ? sc[j][3] * p.scale_log2 : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(sc[j][0], sc[j][1]));
            mx1 = fmaxf(mx1, fmaxf(sc[j][2], sc[j][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m_run[0], mx0);
        const float mn1 = fmaxf(m_run[1], mx1);
        const float ref0 = (mn0 == -INFINITY) ? 0.f : mn0;   // nothing attended yet: keep exponents finite
        const float ref1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float alpha0 = exp2f(m_run[0] - ref0);
        const float alpha1 = exp2f(m_run[1] - ref1);
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int j = 0; j < kNT; ++j) {
            sc[j][0] = exp2f(sc[j][0] - ref0);
            sc[j][1] = exp2f(sc[j][1] - ref0);
            sc[j][2] = exp2f(sc[j][2] - ref1);
            sc[j][3] = exp2f(sc[j][3] - ref1);
            ls0 += sc[j][0] + sc[j][1];
            ls1 += sc[j][2] + sc[j][3];
        }
        ls0 += __shfl_xor_sync(0xffffffffu, ls0, 1);
        ls0 += __shfl_xor_sync(0xffffffffu, ls0, 2);
        ls1 += __shfl_xor_sync(0xffffffffu, ls1, 1);
        ls1 += __shfl_xor_sync(0xffffffffu, ls1, 2);
        l_run[0] = l_run[0] * alpha0 + ls0;
        l_run[1] = l_run[1] * alpha1 + ls1;
        m_run[0] = mn0;
        m_run[1] = mn1;
#pragma unroll
        for (int i = 0; i < kPVTiles; ++i) {
            o[i][0] *= alpha0;
            o[i][1] *= alpha0;
            o[i][2] *= alpha1;
            o[i][3] *= alpha1;
        }

        // ---- P as the A operand of P . V, split P = P_hi + P_lo -------------
        // A single bf16 rounding of P (relative error up to 2^-8) moves the
        // output by ~3e-3 when a handful of rows carry the weight; the hi/lo
        // pair keeps ~16 significant bits of P at the cost of a second MMA.
        uint32_t pa_hi[kPSteps][4], pa_lo[kPSteps][4];
#pragma unroll
        for (int kp = 0; kp < kPSteps; ++kp) {
            split_bf16x2(sc[2 * kp][0], sc[2 * kp][1], pa_hi[kp][0], pa_lo[kp][0]);
            split_bf16x2(sc[2 * kp][2], sc[2 * kp][3], pa_hi[kp][1], pa_lo[kp][1]);
            split_bf16x2(sc[2 * kp + 1][0], sc[2 * kp + 1][1], pa_hi[kp][2], pa_lo[kp][2]);
            split_bf16x2(sc[2 * kp + 1][2], sc[2 * kp + 1][3], pa_hi[kp][3], pa_lo[kp][3]);
        }
        // ---- O[:, own 128 features] += P . V --------------------------------
#pragma unroll
        for (int nt = 0; nt < kPVTiles; nt += 2) {
#pragma unroll
            for (int kp = 0; kp < kPSteps; ++kp) {
                const int row = 16 * kp + lrow + ((lmat & 1) << 3);
                const int fbytes = (f_base + 8 * nt + ((lmat >> 1) << 3)) * 2;
                uint32_t vb[4];
                ldmatrix_x4_trans(vb, kv_base + row * kSmemRow + fbytes);
                mma_bf16_16816(o[nt], pa_lo[kp], vb[0], vb[1]);
                mma_bf16_16816(o[nt + 1], pa_lo[kp], vb[2], vb[3]);
                mma_bf16_16816(o[nt], pa_hi[kp], vb[0], vb[1]);
                mma_bf16_16816(o[nt + 1], pa_hi[kp], vb[2], vb[3]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
    }

    // ---- epilogue: normalised partial and its log-sum-exp -------------------
    const float inv0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
    const float inv1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
    const long long row0 = (static_cast<long long>(b) * p.heads + h0 + g) * S + s;
    const long long row1 = (static_cast<long long>(b) * p.heads + h0 + g + 8) * S + s;
    float* op0 = p.o_part + row0 * kDLatent + f_base + 2 * tq;
    float* op1 = p.o_part + row1 * kDLatent + f_base + 2 * tq;
#pragma unroll
    for (int nt = 0; nt < kPVTiles; ++nt) {
        *reinterpret_cast<float2*>(op0 + 8 * nt) = make_float2(o[nt][0] * inv0, o[nt][1] * inv0);
        *reinterpret_cast<float2*>(op1 + 8 * nt) = make_float2(o[nt][2] * inv1, o[nt][3] * inv1);
    }
    if (w == 0 && tq == 0) {
        p.lse_part[row0] = l_run[0] > 0.f ? (m_run[0] + log2f(l_run[0])) * kLn2 : -INFINITY;
        p.lse_part[row1] = l_run[1] > 0.f ? (m_run[1] + log2f(l_run[1])) * kLn2 : -INFINITY;
    }
}

}  // namespace

size_t partial_mma_smem_bytes() { return sizeof(SharedStorage); }
int partial_mma_block_threads() { return kThreads; }

cudaError_t partial_mma_prepare(int /*device*/) {
    return cudaFuncSetAttribute(mla_partial_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(sizeof(SharedStorage)));
}

cudaError_t partial_mma_occupancy(int* ctas_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, mla_partial_mma_kernel, kThreads,
                                                         sizeof(SharedStorage));
}

cudaError_t launch_partial_mma(const PartialParams& p, dim3 grid, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(SharedStorage);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mla_partial_mma_kernel, p);
}

}  // namespace mla
