// mla_partial_tc.cu -- split-KV MLA decode partials on the 5th-generation
// tensor cores (tcgen05 + tensor memory), head group of 16.
//
// Same work decomposition as the warp-MMA kernel: work item = (request b,
// head group hg of 16 heads, context slice s); a persistent grid of at most
// one CTA per SM walks the items round-robin ("Launch Geometry", Lecture 04,
// s.1, s.4, s.8); each item yields one online-softmax partial (o_s
// normalised, lse_s) that a separate kernel merges ("Graph-resident decode",
// Lecture 08, s.6).
//
// A slice is walked in tiles of 80 cache rows, double-buffered in shared
// memory as 9 column chunks of [80 rows x 64 bf16] in the 128-byte-swizzled
// layout the tensor cores read.  With the 16 heads of a group the products
// are taken "swapped", so the long axis (cache rows, or latent features)
// is the 128-wide M of the MMA and the 16 heads are N:
//   S^T[rows x 16]   = K_tile[rows x 576] . Q^T           36 MMAs, M=128 (80 valid rows), N=16
//   O^T[512 x 32]   += V_tile^T[512 x rows] . [P_hi | P_lo]^T
//                                                          4 x 5 MMAs, M=128 features, N=32
// P enters the second product as a bf16 pair P = P_hi + P_lo laid side by
// side along N (~16 significant bits of P in one MMA); O = O_hi + O_lo at the
// end.  Scores and O live in tensor memory (fp32).
//
// Warp roles (288 threads):
//   warps 0-3  producer: TMA tiled loads of the dense tile (9 boxes of 80 rows,
//              rows past the cache zero-filled by the TMA unit) or, for the
//              sparse top-k gather ("The Commit That Changed Direction"),
//              16-byte cp.async copies of the indexed rows straight into the
//              swizzled layout; also the item's 16 query rows (9 TMA boxes).
//   warps 4-7  softmax: thread t owns tile row t (TMEM lane t); per-head max
//              and sum by warp butterflies and a 4-warp exchange through shared
//              memory; online softmax in base 2 with a lazily moved reference
//              (the reference moves, and O and l are rescaled, only when a
//              head's max grows by more than 2^8, so p <= 256); writes P as
//              the bf16 pair; at the end of an item reads O from tensor memory
//              and writes the partial.
//   warp 8     MMA issue (one thread) and tensor-memory allocation.
// Every wait is bounded (MLA_EDEVICE in the status word on a timeout); the
// CTA drains its copies and its MMAs and frees its tensor memory before it
// exits.  No floating-point atomics: results are a pure function of the
// inputs and the split count.
#include <cfloat>
#include <cmath>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"
#include "slicing.cuh"
#include "tc_utils.cuh"

namespace mla {
namespace {

constexpr int kTileRows = kTcTileRows;                  // 80 cache rows per tile
constexpr int kChunks = kDRow / 64;                     // 9 column chunks of 64 bf16
constexpr int kChunkBytes = kTileRows * 128;            // 10240
constexpr int kTileBytes = kChunks * kChunkBytes;       // 92160
constexpr int kQChunkBytes = kHeadGroup * 128;          // 2048
constexpr int kPVHeads = 2 * kHeadGroup;                // [P_hi | P_lo] along N
constexpr int kPAtomBytes = kPVHeads * 128;             // one 64-row K atom of P^T
constexpr int kPBytes = 2 * kPAtomBytes;                // 80 rows need two K atoms
constexpr int kProducerThreads = 128;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kMmaWarp = 8;
constexpr int kThreads = 288;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemS = 0;                          // S^T[buf] at columns 16*buf
constexpr uint32_t kTmemO = 32;                         // O^T block j at 32 + 32j: hi 0..15, lo 16..31
constexpr float kRescaleLog2 = 8.0f;                    // move the reference when a max grows past 2^8
constexpr float kLn2 = 0.6931471805599453f;

static_assert(kTileRows % 16 == 0 && kTileRows <= 128, "tile rows: whole k-steps, at most M=128");
static_assert(kChunkBytes % 1024 == 0, "chunks stay 1024-byte aligned for the 128-byte swizzle");

struct __align__(1024) SharedStorage {
    uint8_t kv[2][kTileBytes];            // double-buffered tile (chunk c of buffer b at kv[b] + c*kChunkBytes)
    uint8_t q[kChunks * kQChunkBytes];    // Q^T: also absorbs the M=128 over-read of the last chunk
    uint8_t p[2][kPBytes];                // [P_hi | P_lo]^T, K-major, per tile buffer
    float red_max[2][4][16];
    float red_sum[2][4][16];
    int valid[2][kTileRows];
    uint64_t full[2], empty[2], s_full[2], p_full[2], o_done[2];
    uint64_t q_full, q_empty, o_free, bar_max[2], bar_sum[2], mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

struct Item {
    int b, hg, s, n_tiles;
    long long base, e0, e1;
};

__device__ __forceinline__ Item decode_item(const PartialParams& p, int item) {
    Item it;
    it.hg = item % p.n_groups;
    const int rest = item / p.n_groups;
    it.s = rest % p.splits;
    it.b = rest / p.splits;
    const long long n = request_entries(p.sparse, p.topk, p.d_pos, p.row_offset, p.kv_rows, it.b, &it.base);
    const long long per = slice_entries(n, p.splits, p.granule);
    long long e0 = static_cast<long long>(it.s) * per;
    long long e1 = e0 + per;
    if (e1 > n) e1 = n;
    if (e0 > e1) e0 = e1;
    it.e0 = e0;
    it.e1 = e1;
    it.n_tiles = static_cast<int>((e1 - e0 + kTileRows - 1) / kTileRows);
    return it;
}

__device__ __forceinline__ int rows_in_tile(const Item& it, int k) {
    const long long r0 = it.e0 + static_cast<long long>(k) * kTileRows;
    const long long left = it.e1 - r0;
    return static_cast<int>(left < kTileRows ? left : kTileRows);
}

// The next item of this CTA that has tiles, or -1.
__device__ __forceinline__ int next_busy_item(const PartialParams& p, int item, Item* out) {
    for (int i = item + static_cast<int>(gridDim.x); i < p.n_items; i += gridDim.x) {
        const Item it = decode_item(p, i);
        if (it.n_tiles > 0) {
            *out = it;
            return i;
        }
    }
    return -1;
}

__device__ __forceinline__ void raise_device_error(SharedStorage& sh, int* status) {
    sh.abort_flag = 1;
    if (status) atomicCAS(status, 0, static_cast<int>(MLA_EDEVICE));
}

// ============================== producer ==================================
__device__ void producer(const TcMaps& maps, const PartialParams& p, SharedStorage& sh, int t) {
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_normal();
    int g = 0;
    int q_loads = 0;
    int q_key = -1;
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it = decode_item(p, item);
        if (it.n_tiles == 0) continue;
        const int key = it.b * p.n_groups + it.hg;
        if (key != q_key) {
            if (q_loads > 0 && !mbar_wait_bounded(&sh.q_empty, (q_loads - 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            if (t == 0) {
                mbar_arrive_expect_tx(&sh.q_full, kChunks * kQChunkBytes);
                const int y = it.b * p.heads + it.hg * kHeadGroup;
#pragma unroll 1
                for (int c = 0; c < kChunks; ++c) tma_load_2d(sh.q + c * kQChunkBytes, &maps.q, 64 * c, y, &sh.q_full, pol_q);
            }
            q_key = key;
            ++q_loads;
        }
        const int seg_len = p.sparse ? p.cache_len[it.b] : 0;
        for (int k = 0; k < it.n_tiles; ++k, ++g) {
            const int buf = g & 1;
            if (g >= 2 && !mbar_wait_bounded(&sh.empty[buf], ((g >> 1) - 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            const long long r0 = it.e0 + static_cast<long long>(k) * kTileRows;
            const int rows = rows_in_tile(it, k);
            if (!p.sparse) {
                if (t < kTileRows) {
                    const long long row = it.base + r0 + t;
                    sh.valid[buf][t] = (t < rows && row >= 0 && row < p.kv_rows) ? 1 : 0;
                }
                if (t == 0) {
                    mbar_arrive_expect_tx(&sh.full[buf], kTileBytes);
                    const int y = static_cast<int>(it.base + r0);
#pragma unroll 1
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_2d(sh.kv[buf] + c * kChunkBytes, &maps.kv, 64 * c, y, &sh.full[buf], pol_kv);
                } else {
                    mbar_arrive(&sh.full[buf]);
                }
            } else {
                const int* idx = p.indices + static_cast<long long>(it.b) * p.topk + r0;
                if (t < kTileRows) {
                    bool v = false;
                    if (t < rows) {
                        const int id = idx[t];
                        v = id >= 0 && id < seg_len && it.base + id >= 0 && it.base + id < p.kv_rows;
                    }
                    sh.valid[buf][t] = v ? 1 : 0;
                }
                // rows past the tile's last k-step are never read by P . V; masked
                // rows inside it must hold zeros (they meet p = 0)
                const int rows_read = (rows + 15) & ~15;
                const uint32_t dst0 = smem_u32(sh.kv[buf]);
#pragma unroll 4
                for (int piece = t; piece < rows_read * 72; piece += kProducerThreads) {
                    const int r = piece / 72;
                    const int u = piece - r * 72;
                    const int c = u >> 3;
                    const uint32_t dst = dst0 + c * kChunkBytes + r * 128 + ((((u & 7) ^ (r & 7))) << 4);
                    bool v = false;
                    long long row = 0;
                    if (r < rows) {
                        const int id = idx[r];
                        row = it.base + id;
                        v = id >= 0 && id < seg_len && row >= 0 && row < p.kv_rows;
                    }
                    if (v)
                        cp_async_16(dst, reinterpret_cast<const uint8_t*>(p.kv + row * p.row_stride) + u * 16);
                    else
                        st_shared_v4_zero(dst);
                }
                cp_async_commit();
                cp_async_wait_group<0>();
                fence_proxy_async_smem();
                mbar_arrive(&sh.full[buf]);
            }
        }
    }
    if (!ok && t == 0) raise_device_error(sh, p.status);
    // Never retire the CTA with copies into its shared memory in flight.
    if (t == 0) {
        volatile int never = 0;
        for (int b = 0; b < 2 && b < g; ++b) {
            const int last = g - 1 - ((g - 1 - b) & 1);    // last tile number that used buffer b
            if (!mbar_wait_bounded(&sh.full[b], (last >> 1) & 1, &never)) raise_device_error(sh, p.status);
        }
        if (q_loads > 0 && !mbar_wait_bounded(&sh.q_full, (q_loads - 1) & 1, &never)) raise_device_error(sh, p.status);
    }
}

// ============================== MMA issue ==================================
__device__ void mma_issuer(const PartialParams& p, SharedStorage& sh, uint32_t tmem) {
    const uint32_t idesc_qk = make_idesc_bf16(128, kHeadGroup, 0, 0);
    const uint32_t idesc_pv = make_idesc_bf16(128, kPVHeads, 1, 0);
    const uint32_t kv0 = smem_u32(sh.kv[0]);
    const uint32_t q0 = smem_u32(sh.q);
    const uint32_t p0 = smem_u32(sh.p[0]);
    // K-major 128-byte-swizzled operands: 8-row groups 1024 bytes apart
    const uint64_t kv_desc0 = make_sdesc(kv0, 16, 1024, kLayoutSw128);
    const uint64_t q_desc0 = make_sdesc(q0, 16, 1024, kLayoutSw128);
    const uint64_t p_desc0 = make_sdesc(p0, 16, 1024, kLayoutSw128);
    // V^T is MN-major: 64-feature atoms one chunk apart, 8-row groups 1024 apart
    const uint64_t v_desc0 = make_sdesc(kv0, kChunkBytes, 1024, kLayoutSw128);
    int g = 0;
    int q_loads = 0;
    int items_done = 0;
    int cur_key = -1;
    bool ok = true;

    auto issue_pv = [&](int gg, const Item& it, int k, bool first_of_item) -> bool {
        const int buf = gg & 1;
        if (!mbar_wait_bounded(&sh.p_full[buf], (gg >> 1) & 1, &sh.abort_flag)) return false;
        if (first_of_item && items_done > 0 &&
            !mbar_wait_bounded(&sh.o_free, (items_done - 1) & 1, &sh.abort_flag))
            return false;
        tc_fence_after_sync();
        const int ksteps = (rows_in_tile(it, k) + 15) >> 4;
        const uint64_t vb = v_desc0 + ((static_cast<uint32_t>(buf) * kTileBytes) >> 4);
        const uint64_t pb = p_desc0 + ((static_cast<uint32_t>(buf) * kPBytes) >> 4);
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
#pragma unroll 1
            for (int kk = 0; kk < ksteps; ++kk) {
                const uint64_t a = vb + ((2u * j * kChunkBytes + kk * 2048u) >> 4);
                const uint64_t bd = pb + ((static_cast<uint32_t>(kk >> 2) * kPAtomBytes + (kk & 3) * 32u) >> 4);
                umma_bf16(tmem + kTmemO + 32 * j, a, bd, idesc_pv, (first_of_item && kk == 0) ? 0u : 1u);
            }
        }
        umma_commit(&sh.empty[buf]);
        umma_commit(&sh.o_done[buf]);
        return true;
    };

    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it = decode_item(p, item);
        if (it.n_tiles == 0) continue;
        const int key = it.b * p.n_groups + it.hg;
        if (key != cur_key) {
            if (!mbar_wait_bounded(&sh.q_full, q_loads & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            ++q_loads;
            cur_key = key;
        }
        const int first_g = g;
        for (int k = 0; k < it.n_tiles; ++k, ++g) {
            const int buf = g & 1;
            if (!mbar_wait_bounded(&sh.full[buf], (g >> 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint64_t kb = kv_desc0 + ((static_cast<uint32_t>(buf) * kTileBytes) >> 4);
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t off = (c * kChunkBytes + kk * 32u) >> 4;
                    const uint32_t qoff = (c * kQChunkBytes + kk * 32u) >> 4;
                    umma_bf16(tmem + kTmemS + 16 * buf, kb + off, q_desc0 + qoff, idesc_qk, (c | kk) ? 1u : 0u);
                }
            }
            umma_commit(&sh.s_full[buf]);
            if (k > 0 && !issue_pv(g - 1, it, k - 1, k - 1 == 0)) {
                ok = false;
                break;
            }
        }
        if (!ok) break;
        if (!issue_pv(g - 1, it, it.n_tiles - 1, it.n_tiles == 1)) {
            ok = false;
            break;
        }
        (void)first_g;
        ++items_done;
        // release the query tile once its last user has been issued, if the
        // next item of this CTA needs a different one
        Item nx;
        const int ni = next_busy_item(p, item, &nx);
        if (ni >= 0 && nx.b * p.n_groups + nx.hg != key) umma_commit(&sh.q_empty);
    }
    if (!ok) raise_device_error(sh, p.status);
    // all MMAs complete before the CTA frees its tensor memory
    umma_commit(&sh.mma_done);
    volatile int never = 0;
    if (!mbar_wait_bounded(&sh.mma_done, 0, &never)) raise_device_error(sh, p.status);
}

// ============================== softmax warps ==============================
__device__ __forceinline__ void warp_max16(float (&v)[16], int lane) {
    // After the halving steps lane L holds head (L >> 1); the last step joins the pair.
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const bool up = lane & 16;
        const float send = up ? v[k] : v[k + 8];
        const float keep = up ? v[k + 8] : v[k];
        v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool up = lane & 8;
        const float send = up ? v[k] : v[k + 4];
        const float keep = up ? v[k + 4] : v[k];
        v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool up = lane & 4;
        const float send = up ? v[k] : v[k + 2];
        const float keep = up ? v[k + 2] : v[k];
        v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
    {
        const bool up = lane & 2;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
    v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}
__device__ __forceinline__ void warp_sum16(float (&v)[16], int lane) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const bool up = lane & 16;
        const float send = up ? v[k] : v[k + 8];
        const float keep = up ? v[k + 8] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool up = lane & 8;
        const float send = up ? v[k] : v[k + 4];
        const float keep = up ? v[k + 4] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool up = lane & 4;
        const float send = up ? v[k] : v[k + 2];
        const float keep = up ? v[k + 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    {
        const bool up = lane & 2;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    v[0] = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__device__ void softmax_warps(const PartialParams& p, SharedStorage& sh, uint32_t tmem, int q, int lane) {
    const int t = q * 32 + lane;                     // tile row / TMEM lane of this thread
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    int g = 0;
    int items_done = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it = decode_item(p, item);
        if (it.n_tiles == 0) continue;
        float m_ref[16], l_run[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
            m_ref[h] = -INFINITY;
            l_run[h] = 0.f;
        }
        const int first_g = g;
        for (int k = 0; k < it.n_tiles; ++k, ++g) {
            const int buf = g & 1;
            const int rows = rows_in_tile(it, k);
            // the tile's row flags come from the producer: acquire its barrier too
            if (!mbar_wait_bounded(&sh.s_full[buf], (g >> 1) & 1, &sh.abort_flag) ||
                !mbar_wait_bounded(&sh.full[buf], (g >> 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float s[16];
            if (q * 32 < kTileRows) {
                tmem_ld16(tmem + lane_addr + kTmemS + 16 * buf, s);
            } else {
#pragma unroll
                for (int h = 0; h < 16; ++h) s[h] = 0.f;
            }
            const bool row_ok = t < rows && sh.valid[buf][t] != 0;
#pragma unroll
            for (int h = 0; h < 16; ++h) s[h] = row_ok ? s[h] * p.scale_log2 : -INFINITY;

            // ---- tile max per head (fixed butterfly + 4-warp exchange) ----------
            float red[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) red[h] = s[h];
            warp_max16(red, lane);
            if ((lane & 1) == 0) sh.red_max[buf][q][lane >> 1] = red[0];
            mbar_arrive(&sh.bar_max[buf]);
            if (!mbar_wait_bounded(&sh.bar_max[buf], (g >> 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            float alpha[16];
            bool rescale = false;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const float tmax = fmaxf(fmaxf(sh.red_max[buf][0][h], sh.red_max[buf][1][h]),
                                         fmaxf(sh.red_max[buf][2][h], sh.red_max[buf][3][h]));
                float ref = m_ref[h];
                alpha[h] = 1.f;
                if (tmax > -INFINITY && (ref == -INFINITY || tmax > ref + kRescaleLog2)) {
                    if (ref != -INFINITY && l_run[h] > 0.f) {
                        alpha[h] = exp2f(ref - tmax);
                        rescale = true;
                    }
                    ref = tmax;
                }
                m_ref[h] = ref;
            }

            // ---- probabilities, written as the bf16 pair [P_hi | P_lo]^T --------
            float pr[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) pr[h] = (row_ok && m_ref[h] > -INFINITY) ? exp2f(s[h] - m_ref[h]) : 0.f;
            if (g >= 2 && !mbar_wait_bounded(&sh.o_done[buf], ((g >> 1) - 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            if (t < kTileRows) {
                const uint32_t pbase = smem_u32(sh.p[buf]) + (t >> 6) * kPAtomBytes;
                const uint32_t byte = 2u * (t & 63);
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const __nv_bfloat16 hi = __float2bfloat16_rn(pr[h]);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(pr[h] - __bfloat162float(hi));
                    const int vh = h, vl = 16 + h;
                    st_shared_u16(pbase + (vh >> 3) * 1024 + sw128_offset(vh & 7, byte), __bfloat16_as_ushort(hi));
                    st_shared_u16(pbase + (vl >> 3) * 1024 + sw128_offset(vl & 7, byte), __bfloat16_as_ushort(lo));
                }
            }
            // ---- row sums -------------------------------------------------------
#pragma unroll
            for (int h = 0; h < 16; ++h) red[h] = pr[h];
            warp_sum16(red, lane);
            if ((lane & 1) == 0) sh.red_sum[buf][q][lane >> 1] = red[0];
            mbar_arrive(&sh.bar_sum[buf]);
            if (!mbar_wait_bounded(&sh.bar_sum[buf], (g >> 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const float ts = ((sh.red_sum[buf][0][h] + sh.red_sum[buf][1][h]) + sh.red_sum[buf][2][h]) +
                                 sh.red_sum[buf][3][h];
                l_run[h] = l_run[h] * alpha[h] + ts;
            }
            // ---- rare: move O to the new reference --------------------------------
            if (rescale && g > first_g) {
                const int gp = g - 1;
                if (!mbar_wait_bounded(&sh.o_done[gp & 1], (gp >> 1) & 1, &sh.abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        float o[16];
                        const uint32_t a = tmem + lane_addr + kTmemO + 32 * j + 16 * half;
                        tmem_ld16(a, o);
#pragma unroll
                        for (int h = 0; h < 16; ++h) o[h] *= alpha[h];
                        tmem_st16(a, o);
                    }
                }
            }
            // ---- dense: masked rows the P . V k-steps read must hold zeros -------
            if (!p.sparse && t < kTileRows && !row_ok && t < ((rows + 15) & ~15)) {
                const uint32_t row_base = smem_u32(sh.kv[buf]) + t * 128;
#pragma unroll 1
                for (int c = 0; c < 8; ++c)
#pragma unroll
                    for (int u = 0; u < 8; ++u) st_shared_v4_zero(row_base + c * kChunkBytes + u * 16);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&sh.p_full[buf]);
        }
        if (!ok) break;

        // ---- epilogue: O = (O_hi + O_lo) / l, lse = m + log2(l) (to natural log) ---
        const int gl = g - 1;
        if (!mbar_wait_bounded(&sh.o_done[gl & 1], (gl >> 1) & 1, &sh.abort_flag)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        float inv[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) inv[h] = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
        const long long row0 = (static_cast<long long>(it.b) * p.heads + it.hg * kHeadGroup) * p.splits + it.s;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            float hi[16], lo[16];
            tmem_ld16(tmem + lane_addr + kTmemO + 32 * j, hi);
            tmem_ld16(tmem + lane_addr + kTmemO + 32 * j + 16, lo);
            const int f = 128 * j + t;
#pragma unroll
            for (int h = 0; h < 16; ++h)
                p.o_part[(row0 + static_cast<long long>(h) * p.splits) * kDLatent + f] = (hi[h] + lo[h]) * inv[h];
        }
        if (t < 16) {
            float lv = 0.f, mv = 0.f;
#pragma unroll
            for (int h = 0; h < 16; ++h)
                if (h == t) {
                    lv = l_run[h];
                    mv = m_ref[h];
                }
            p.lse_part[row0 + static_cast<long long>(t) * p.splits] = lv > 0.f ? (mv + log2f(lv)) * kLn2 : -INFINITY;
        }
        tc_fence_before_sync();
        mbar_arrive(&sh.o_free);
        ++items_done;
    }
    if (!ok && lane == 0) raise_device_error(sh, p.status);
}

__global__ void __launch_bounds__(kThreads, 1) mla_partial_tc_kernel(const __grid_constant__ TcMaps maps,
                                                                      const PartialParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SharedStorage& sh =
        *reinterpret_cast<SharedStorage*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.full[i], kProducerThreads);
            mbar_init(&sh.empty[i], 1);
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.p_full[i], 128);
            mbar_init(&sh.o_done[i], 1);
            mbar_init(&sh.bar_max[i], 128);
            mbar_init(&sh.bar_sum[i], 128);
        }
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, 1);
        mbar_init(&sh.o_free, 128);
        mbar_init(&sh.mma_done, 1);
        sh.abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sh.tmem_base;
    // Inputs (d_pos, cache rows, indices, q) may be written by the kernel
    // before this one on the stream: wait for it before any global read.
    grid_dependency_wait();
    allow_dependent_launch();
    if (warp < 4) {
        producer(maps, p, sh, threadIdx.x);
    } else if (warp < kMmaWarp) {
        softmax_warps(p, sh, tmem, warp - kSoftmaxWarp0, lane);
    } else if (lane == 0) {
        mma_issuer(p, sh, tmem);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t partial_tc_smem_bytes() { return sizeof(SharedStorage) + 1024; }
int partial_tc_block_threads() { return kThreads; }

cudaError_t partial_tc_prepare(int /*device*/) {
    return cudaFuncSetAttribute(mla_partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(partial_tc_smem_bytes()));
}

cudaError_t launch_partial_tc(const TcMaps& maps, const PartialParams& p, dim3 grid, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = partial_tc_smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel, maps, p);
}

}  // namespace mla
