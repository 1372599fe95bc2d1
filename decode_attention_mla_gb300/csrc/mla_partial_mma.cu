// mla_partial_mma.cu -- split-KV MLA decode partials, head-group-16 kernel.
//
// Work item = (request b, head group of 16 heads, context slice s); item i
// decodes as hg = i % G, s = (i / G) % S, b = i / (G * S), so the items that
// read the same cache rows for different head groups run side by side.  A
// persistent grid of at most one CTA per SM walks the items round-robin
// ("Launch Geometry", Lecture 04, s.1 and s.8: the context split is the axis
// manufactured for batch-1 decode; s.4: the grid is sized from the SM count).
// Each item yields one online-softmax partial: o_s (normalised) and lse_s
// ("Graph-resident decode", Lecture 08, s.6: per-slice partials, merged by a
// separate kernel).
//
// Warp roles:
//   producer warp : walks the same items and, per 32-row stage, moves one
//                   1152-byte cache row per lane into a 5-deep shared-memory
//                   ring with bulk copies (TMA engine); completion is counted
//                   on the stage's mbarrier.  Dense rows are base + e, sparse
//                   rows base + indices[b][e] (a gather, "The Commit That
//                   Changed Direction"); index loads are prefetched a few
//                   stages ahead.  Rows past the slice or out of range are
//                   zero-filled and masked.  It also stages the item's 16 query
//                   rows in shared memory when the (request, head group)
//                   changes.
//   8 MMA warps   : scores S[16 heads x 32 rows] = Q . K^T with mma.m16n8k16
//                   (bf16 in, fp32 accumulate).  Warp w takes k-steps
//                   9*(w%4) .. 9*(w%4)+8 of the 576-wide contraction for rows
//                   16*(w/4) .. +15; the four k-group partials are summed in
//                   fixed order through shared memory.  Every warp applies the
//                   same online-softmax update (base-2 exponent, quad shuffles
//                   for row max and row sum) and accumulates its own 64 output
//                   features: O += P . V with V = the latent c rows and P as a
//                   bf16 hi + lo pair (two MMAs, ~16 significant bits of P).
// No floating-point atomics: the result is a pure function of the inputs and
// the split count.  Every wait is bounded; a timeout raises MLA_EDEVICE in the
// status word and the CTA drains its copies before it exits.
#include <cfloat>
#include <cmath>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"
#include "slicing.cuh"
#include "tc_utils.cuh"

namespace mla {
namespace {

constexpr int kStages = 5;                                // ring depth (32-row stages)
constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;        // + one producer warp
constexpr int kProducerWarp = kComputeWarps;
constexpr int kSmemRow = kRowBytes + 16;                  // padding: 8 rows x 16 B hit 32 distinct banks
constexpr int kNT = kStageRows / 8;                       // 4 score n-tiles of 8 rows
constexpr int kKGroups = 4;                               // contraction split across warps
constexpr int kKStepsPerWarp = kDRow / 16 / kKGroups;     // 9
constexpr int kFeatPerWarp = kDLatent / kComputeWarps;    // 64 output features per warp
constexpr int kPVTiles = kFeatPerWarp / 8;                // 8
constexpr int kPSteps = kStageRows / 16;                  // 2
constexpr int kIdxPrefetch = 4;                           // sparse index prefetch depth (stages)
constexpr float kLn2 = 0.6931471805599453f;
// Cache rows arrive by one 1152-byte bulk copy per row into padded 1168-byte
// rows (8 consecutive rows hit 8 distinct 16-byte bank groups); the query tile
// is one TMA box [9 chunks][16 rows][64 bf16], 128-byte swizzled.  (A TMA box
// for whole dense stages was measured too: faster for single-stage slices,
// slower for two-stage ones and for the timed T = 8192 shape.)
constexpr int kChunks = kDRow / 64;                       // 9
constexpr int kQChunkBytes = kHeadGroup * 128;            // 2048

static_assert(kComputeWarps == 2 * kKGroups, "warp w: k-group w % 4, row half w / 4");
static_assert(kDRow / 16 % kKGroups == 0, "contraction split");

struct __align__(1024) SharedStorage {
    uint8_t q[kChunks * kQChunkBytes];                    // the item's 16 query rows (1024-byte aligned)
    uint8_t kv[kStages][kStageRows * kSmemRow];           // stage slots
    float4 red[2][kKGroups][kNT][32];                     // per-k-group partial scores
    int valid[kStages][kStageRows];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t red_bar[2];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t stall_bar;                                   // test hook: a barrier nothing arrives at
    int abort_flag;
};

// Byte offset of byte b of row r in a 128-byte-swizzled chunk-major tile whose
// 64-column chunks are chunk_bytes apart (b a multiple of 16 for ldmatrix rows).
__device__ __forceinline__ uint32_t sw_off(int r, int b, int chunk_bytes) {
    return static_cast<uint32_t>((b >> 7) * chunk_bytes + r * 128 + ((((b >> 4) & 7) ^ (r & 7)) << 4) + (b & 15));
}
__device__ __forceinline__ void raise_device_error(SharedStorage& sh, int* status) {
    sh.abort_flag = 1;
    if (status) atomicCAS(status, 0, static_cast<int>(MLA_EDEVICE));
}

struct Item {
    int b, hg, s, n_stages;
    long long base;
    uint32_t e0, e1;                      // entries [e0, e1) of the request
};

__device__ __forceinline__ Item decode_item(const PartialParams& p, int item) {
    Item it;
    const uint32_t ui = static_cast<uint32_t>(item);
    const uint32_t rest = ui / static_cast<uint32_t>(p.n_groups);
    it.hg = static_cast<int>(ui - rest * static_cast<uint32_t>(p.n_groups));
    const uint32_t b = rest / static_cast<uint32_t>(p.splits);
    it.s = static_cast<int>(rest - b * static_cast<uint32_t>(p.splits));
    it.b = static_cast<int>(b);
    // entry counts are below 2^31 (d_pos and the list length are int32), so
    // the slice arithmetic runs in 32 bits (64-bit division is slow)
    const uint32_t n = static_cast<uint32_t>(
        request_entries(p.sparse, p.topk, p.d_pos, p.row_offset, p.kv_rows, it.b, &it.base));
    const uint32_t per = slice_entries_u32(n, static_cast<uint32_t>(p.splits), kStageRows);
    uint32_t e0 = static_cast<uint32_t>(it.s) * per;
    uint32_t e1 = e0 + per;
    if (e1 > n) e1 = n;
    if (e0 > e1) e0 = e1;
    it.e0 = e0;
    it.e1 = e1;
    it.n_stages = static_cast<int>((e1 - e0 + kStageRows - 1) / kStageRows);
    return it;
}

// Query tile of the CTA's first item: known without the context length.
__device__ __forceinline__ int first_key(const PartialParams& p) {
    const int item = static_cast<int>(blockIdx.x);
    const int rest = item / p.n_groups;
    return (rest / p.splits) * p.n_groups + (item - rest * p.n_groups);
}

__device__ __forceinline__ void load_q(const TcMaps& maps, const PartialParams& p, SharedStorage& sh, int key,
                                       int lane) {
    if (lane == 0) {
        const int b = key / p.n_groups;
        const int hg = key - b * p.n_groups;
        mbar_arrive_expect_tx(&sh.q_full, kChunks * kQChunkBytes);
        tma_load_3d(sh.q, &maps.q, 0, b * p.heads + hg * kHeadGroup, 0, &sh.q_full, l2_policy_evict_normal());
    }
}

// ============================== producer ==================================
__device__ void producer(const TcMaps& maps, const PartialParams& p, SharedStorage& sh, int lane) {
    const uint64_t policy = l2_policy_evict_first();
    int stage = 0;            // stages issued so far (ring position)
    // the first query tile is requested before the context length is read; the
    // MMA warps follow the same sequence of keys (a new tile whenever a busy
    // item's key differs) and release a tile through q_empty, read or not
    int q_key = first_key(p);
    load_q(maps, p, sh, q_key, lane);
    int q_loads = 1;          // query tiles staged so far
    // test hook: a wait that runs out, so every role takes the abort path
    bool ok = !(p.stall_test && !mbar_wait_bounded(&sh.stall_bar, 0, &sh.abort_flag, kStallTestCycles));
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it = decode_item(p, item);
        if (it.n_stages == 0) continue;
        const int seg_len = p.sparse ? p.cache_len[it.b] : 0;
        const int key = it.b * p.n_groups + it.hg;
        if (key != q_key) {
            if (!mbar_wait_bounded(&sh.q_empty, (q_loads - 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            load_q(maps, p, sh, key, lane);
            q_key = key;
            ++q_loads;
        }
        // sparse: indices of the next few stages, loaded ahead of their use
        int idx_pf[kIdxPrefetch];
        const int* idx = p.sparse ? p.indices + static_cast<long long>(it.b) * p.topk : nullptr;
        if (p.sparse) {
#pragma unroll
            for (int k = 0; k < kIdxPrefetch; ++k) {
                const long long e = it.e0 + static_cast<long long>(k) * kStageRows + lane;
                idx_pf[k] = (e < it.e1) ? idx[e] : -1;
            }
        }
        for (int st = 0; st < it.n_stages; ++st, ++stage) {
            const int slot = stage % kStages;
            if (stage >= kStages &&
                !mbar_wait_bounded(&sh.empty[slot], ((stage / kStages) - 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            const long long e = it.e0 + static_cast<long long>(st) * kStageRows + lane;
            bool valid = false;
            long long row = 0;
            if (e < it.e1) {
                if (!p.sparse) {
                    row = it.base + e;
                    valid = (row >= 0 && row < p.kv_rows);
                } else {
                    const int id = idx_pf[0];
                    if (id >= 0 && id < seg_len) {
                        row = it.base + id;
                        valid = (row >= 0 && row < p.kv_rows);
                    }
                }
            }
            if (p.sparse) {
#pragma unroll
                for (int k = 0; k + 1 < kIdxPrefetch; ++k) idx_pf[k] = idx_pf[k + 1];
                const long long en = it.e0 + static_cast<long long>(st + kIdxPrefetch) * kStageRows + lane;
                idx_pf[kIdxPrefetch - 1] = (en < it.e1) ? idx[en] : -1;
            }
            uint8_t* dst = sh.kv[slot] + lane * kSmemRow;
            sh.valid[slot][lane] = valid ? 1 : 0;
            if (!valid) {
                // masked rows still feed P . V (with p = 0): keep them finite
                uint4* z = reinterpret_cast<uint4*>(dst);
#pragma unroll 8
                for (int i = 0; i < kRowBytes / 16; ++i) z[i] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sh.full[slot], valid ? static_cast<uint32_t>(kRowBytes) : 0u);
            if (valid) bulk_copy_g2s(dst, p.kv + row * p.row_stride, kRowBytes, &sh.full[slot], policy);
        }
    }
    if (!ok && lane == 0) raise_device_error(sh, p.status);
    // Never retire the CTA with copies into its shared memory in flight.
    if (lane == 0) {
        volatile int never = 0;
        for (int slot = 0; slot < kStages && slot < stage; ++slot) {
            const int last_use = (stage - 1 - slot) / kStages;
            if (!mbar_wait_bounded(&sh.full[slot], last_use & 1, &never)) raise_device_error(sh, p.status);
        }
        if (q_loads > 0 && !mbar_wait_bounded(&sh.q_full, (q_loads - 1) & 1, &never))
            raise_device_error(sh, p.status);
    }
}

// ============================== MMA warps =================================
__device__ void consumer(const PartialParams& p, SharedStorage& sh, int w, int lane) {
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int kg = w % kKGroups;           // contraction k-group
    const int rh = w / kKGroups;           // row half (n-tiles 2rh, 2rh+1) of the score tile
    const int f_base = w * kFeatPerWarp;   // own output features
    const int lrow = lane & 7;
    const int lmat = lane >> 3;
    const uint32_t q_base = smem_u32(sh.q);

    uint32_t qa[kKStepsPerWarp][4];
    int stage = 0;
    int red_round = 0;
    int q_phase = 0;                       // query tiles consumed (q_full phases)
    int q_key = first_key(p);              // key of the tile the producer loaded last
    bool q_in_regs = false;                // that tile is in registers (and released)
    bool ok = true;

    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it = decode_item(p, item);
        if (it.n_stages == 0) {
            write_empty_partial(p.o_part, p.lse_part,
                                (static_cast<long long>(it.b) * p.heads + it.hg * kHeadGroup) * p.splits + it.s,
                                p.splits, w * 32 + lane, kComputeWarps * 32);
            continue;
        }
        const int key = it.b * p.n_groups + it.hg;
        if (key != q_key) {
            // the producer loads another tile over this one: release it, read or
            // not (it must have landed first)
            if (!q_in_regs) {
                if (!mbar_wait_bounded(&sh.q_full, q_phase & 1, &sh.abort_flag)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.q_empty);
            }
            ++q_phase;
            q_key = key;
            q_in_regs = false;
        }
        if (!q_in_regs) {
            if (!mbar_wait_bounded(&sh.q_full, q_phase & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            // fragments of Q rows g, g+8 for this warp's 9 k-steps
#pragma unroll
            for (int kk = 0; kk < kKStepsPerWarp; ++kk) {
                const int cb = ((kg * kKStepsPerWarp + kk) * 16 + 2 * tq) * 2;
                qa[kk][0] = ld_shared_u32(q_base + sw_off(g, cb, kQChunkBytes));
                qa[kk][1] = ld_shared_u32(q_base + sw_off(g + 8, cb, kQChunkBytes));
                qa[kk][2] = ld_shared_u32(q_base + sw_off(g, cb + 16, kQChunkBytes));
                qa[kk][3] = ld_shared_u32(q_base + sw_off(g + 8, cb + 16, kQChunkBytes));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.q_empty);
            q_in_regs = true;
        }

        float o[kPVTiles][4];
#pragma unroll
        for (int i = 0; i < kPVTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};   // running max, base-2 units
        float l_run[2] = {0.f, 0.f};               // running sum of 2^(s - m_run)

        for (int st = 0; st < it.n_stages; ++st, ++stage) {
            const int slot = stage % kStages;
            if (!mbar_wait_bounded(&sh.full[slot], (stage / kStages) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t kv_base = smem_u32(sh.kv[slot]);

            // ---- partial scores: rows 16rh..16rh+15, this warp's 144 features
            float acc[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < kKStepsPerWarp; ++kk) {
                const int col_bytes = (kg * kKStepsPerWarp + kk) * 32;
                const int row = 16 * rh + lrow + ((lmat >> 1) << 3);
                uint32_t bf[4];
                ldmatrix_x4(bf, kv_base + row * kSmemRow + col_bytes + ((lmat & 1) << 4));
                mma_bf16_16816(acc[0], qa[kk], bf[0], bf[1]);
                mma_bf16_16816(acc[1], qa[kk], bf[2], bf[3]);
            }

            // ---- sum the four k-groups (fixed order) ------------------------
            const int rb = red_round & 1;
            sh.red[rb][kg][2 * rh][lane] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
            sh.red[rb][kg][2 * rh + 1][lane] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
            mbar_arrive(&sh.red_bar[rb]);
            if (!mbar_wait_bounded(&sh.red_bar[rb], (red_round >> 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            ++red_round;
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

            // ---- P as a bf16 hi + lo pair (A operand of P . V) ------------------
            uint32_t pa_hi[kPSteps][4], pa_lo[kPSteps][4];
#pragma unroll
            for (int kp = 0; kp < kPSteps; ++kp) {
                split_bf16x2(sc[2 * kp][0], sc[2 * kp][1], pa_hi[kp][0], pa_lo[kp][0]);
                split_bf16x2(sc[2 * kp][2], sc[2 * kp][3], pa_hi[kp][1], pa_lo[kp][1]);
                split_bf16x2(sc[2 * kp + 1][0], sc[2 * kp + 1][1], pa_hi[kp][2], pa_lo[kp][2]);
                split_bf16x2(sc[2 * kp + 1][2], sc[2 * kp + 1][3], pa_hi[kp][3], pa_lo[kp][3]);
            }
            // ---- O[:, own 64 features] += P . V ---------------------------------
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
        if (!ok) break;

        // ---- epilogue: normalised partial and its log-sum-exp -------------------
        const float inv0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
        const float inv1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
        const int h0 = it.hg * kHeadGroup;
        const long long row0 = (static_cast<long long>(it.b) * p.heads + h0 + g) * p.splits + it.s;
        const long long row1 = (static_cast<long long>(it.b) * p.heads + h0 + g + 8) * p.splits + it.s;
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
    if (!ok && lane == 0) raise_device_error(sh, p.status);
}

__global__ void __launch_bounds__(kThreads, 1) mla_partial_mma_kernel(const __grid_constant__ TcMaps maps,
                                                                       const PartialParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SharedStorage& sh =
        *reinterpret_cast<SharedStorage*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], 32);
            mbar_init(&sh.empty[i], kComputeWarps);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&sh.red_bar[i], kComputeWarps * 32);
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, kComputeWarps);
        mbar_init(&sh.stall_bar, 1);
        sh.abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    // Inputs (d_pos, cache rows, indices, q) may be written by the kernel
    // before this one on the stream: wait for it before any global read.
    grid_dependency_wait();
    allow_dependent_launch();
    if (warp == kProducerWarp)
        producer(maps, p, sh, lane);
    else
        consumer(p, sh, warp, lane);
}

}  // namespace

size_t partial_mma_smem_bytes() { return sizeof(SharedStorage) + 1024; }
int partial_mma_block_threads() { return kThreads; }

cudaError_t partial_mma_prepare(int /*device*/) {
    return cudaFuncSetAttribute(mla_partial_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(partial_mma_smem_bytes()));
}

cudaError_t partial_mma_occupancy(int* ctas_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, mla_partial_mma_kernel, kThreads,
                                                         partial_mma_smem_bytes());
}

cudaError_t launch_partial_mma(const TcMaps& maps, const PartialParams& p, dim3 grid, bool pdl,
                               cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = partial_mma_smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mla_partial_mma_kernel, maps, p);
}

}  // namespace mla
