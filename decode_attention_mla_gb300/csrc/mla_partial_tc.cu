// mla_partial_tc.cu -- split-KV MLA decode partials on the 5th-generation
// tensor cores (tcgen05 + tensor memory), head groups of 16, 32 or 64.
//
// Same work decomposition as the warp-MMA kernel: work item = (request b,
// head group hg, context slice s); a persistent grid of at most one CTA per
// SM walks the items round-robin ("Launch Geometry", Lecture 04, s.1, s.4,
// s.8); each item yields one online-softmax partial per head (o_s
// normalised, lse_s) that a separate kernel merges ("Graph-resident decode",
// Lecture 08, s.6).
//
// A slice is walked in tiles of TR cache rows (80 for head groups of 16, 64
// for 32 and 64), double-buffered in shared memory as 9 column chunks of
// [TR rows x 64 bf16] in the 128-byte-swizzled layout the tensor cores read;
// a tile arrives as three TMA boxes of three chunks, each with its own
// barrier, so the score MMAs start on the first third while the rest is in
// flight.
//
// Head groups of 16 and 32: the products are taken "swapped", so the long
// axis (cache rows, or latent features) is the 128-wide M of the MMA and the
// HG heads are N:
//   S^T[rows x HG]   = K_tile[rows x 576] . Q^T         36 MMAs, M=128 (TR valid rows), N=HG
//   O^T[512 x 2HG]  += V_tile^T[512 x rows] . [P_hi | P_lo]^T
//                                                        4 x TR/16 MMAs, M=128 features, N=2HG
// P enters the second product as a bf16 pair P = P_hi + P_lo laid side by
// side along N (~16 significant bits of P in one MMA); O = O_hi + O_lo at the
// end.  Scores and O live in tensor memory (fp32).  The MMA cost is nearly
// flat in N up to 64, so 32 heads per CTA halve the instructions per head
// (and the re-reads of each cache row) of wide-head decode.
//
// Head group of 64 ("wide"): O^T with P_hi and P_lo side by side would fill
// all of tensor memory, so the pair is taken along K instead (two MMAs per
// k-step into one accumulator), and the scores are taken with the heads on M:
//   S[64 heads x rows]  = Q[64 x 576] . K_tile^T        36 MMAs, M=64, N=TR
//   O^T[512 x 64]      += V_tile^T . P_hi^T + V_tile^T . P_lo^T
//                                                        4 x 2 x TR/16 MMAs, M=128 features, N=64
// so the scores of one head lie in one tensor-memory lane: two threads own
// a head (32 rows each) and share nothing but the head's tile max.  P_hi^T of a tile is written
// over the tile's rope chunk (the scores are its only reader), which makes
// room in shared memory for the 64-head query tile.  Per cache row and head
// this issues 1.5x fewer MMAs than head groups of 32 and reads each row half
// as often.
//
// Online softmax in base 2 with a lazily moved reference m (per head, the
// same in every thread that sees the head): a tile whose scores all stay
// below m + 8 is turned into probabilities at once (one barrier that ORs
// "some score is above"); only otherwise (the first tile of a slice, or a max
// that grew by more than 2^8) the tile max becomes the reference and O is
// rescaled.  Head groups of 16 and 32 take the tile max with warp max
// instructions and a four-warp exchange through shared memory, and keep row
// sums per thread (one tile row each), added across the warpgroup once per
// slice in a fixed order; the wide group keeps one running sum per thread
// (32 rows of one head), the two of a head added once per slice.
//
// Warp roles, head group 16 (320 threads):
//   warps 0-3  producer.  Dense: one thread issues the TMA boxes (rows past
//              the cache are zero-filled by the TMA unit).  Sparse top-k
//              gather ("The Commit That Changed Direction"): 128 threads
//              copy the indexed rows with 16-byte cp.async straight into the
//              swizzled layout, one commit group per third of the tile.
//              Also the item's query rows (one TMA box).
//   warps 4-7  softmax: thread t owns tile row t (tensor-memory lane t);
//              writes P as the bf16 pair; at the end of an item reads O from
//              tensor memory and writes the partial.
//   warp 8     score MMA issue and tensor-memory allocation; warp 9 P . V
//              MMA issue.
// Head group 32 (384 threads, dense only): warp 0 producer, warp 1 score
// MMAs and allocation, warp 2 P . V MMAs, warps 4-7 and 8-11 softmax for
// heads 0-15 and 16-31 of the group (each warpgroup covers the tile's rows).
// Head group 64 (256 threads, dense only): warps 0-2 as for 32; warps 4-7
// own 16 heads each, two threads per head, and write the partial (O^T lane
// = feature).
// Every wait is bounded (MLA_EDEVICE in the status word on a timeout); the
// threads of a hardware barrier leave a loop together (the decision to leave
// is the barrier's own OR-reduction); the CTA drains its copies and its MMAs
// and frees its tensor memory before it exits.  No floating-point atomics:
// results are a pure function of the inputs and the split count.
#include <cfloat>
#include <cmath>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"
#include "slicing.cuh"
#include "tc_utils.cuh"

namespace mla {
namespace {

constexpr int kChunks = kDRow / 64;                     // 9 column chunks of 64 bf16
constexpr int kGroups = kChunks / kTcBoxChunks;         // TMA boxes (and barriers) per tile
constexpr int kGatherBatches = 3;                       // sparse: cp.async commit groups per tile
constexpr int kGroupsPerBatch = kGroups / kGatherBatches;
constexpr int kProducerThreads = 128;                   // sparse gather threads (head group 16)
constexpr int kSoftmaxThreads = 128;                    // one warpgroup per 16 heads
constexpr int kSoftmaxWarp0 = 4;
constexpr int kBarProducer = 1;                         // hardware barrier ids (0 is __syncthreads)
constexpr int kBarTmem = 2;                             // softmax + MMA warps: tensor memory allocated
constexpr int kBarSoftmax0 = 3;                         // + softmax warpgroup
constexpr float kRescaleLog2 = 8.0f;                    // move the reference when a max grows past 2^8
constexpr float kLn2 = 0.6931471805599453f;

static_assert(kChunks % kTcBoxChunks == 0, "a tile is a whole number of TMA boxes");
static_assert(kGroups % kGatherBatches == 0, "gather batches cover whole boxes");
static_assert((kTcGranule & (kTcGranule - 1)) == 0, "power-of-two granule");

// Everything that follows from the head group HG (16, 32 or 64).
template <int HG>
struct Cfg {
    static constexpr bool kWide = HG == 64;                        // heads on M for the scores, P pair along K
    static constexpr int kTileRows = HG == 16 ? kTcTileRows : kTcTileRows32;
    static constexpr int kChunkBytes = kTileRows * 128;
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kGroupBytes = kTcBoxChunks * kChunkBytes;
    static constexpr int kQChunkBytes = HG * 128;
    static constexpr int kQBytes = kChunks * kQChunkBytes;
    static constexpr int kPVHeads = kWide ? HG : 2 * HG;           // N of P . V: [P_hi | P_lo], or one of them
    static constexpr int kPAtomBytes = kPVHeads * 128;             // one 64-row K atom of P^T
    static constexpr int kPAtoms = (kTileRows + 63) / 64;
    static constexpr int kPBytes = kPAtoms * kPAtomBytes;
    static constexpr int kWGs = kWide ? 1 : HG / 16;               // softmax warpgroups
    static constexpr int kSoftmaxWarps = 4 * kWGs;
    static constexpr int kMmaWarp = HG == 16 ? 8 : 1;              // QK issue + TMEM allocation
    static constexpr int kPvWarp = HG == 16 ? 9 : 2;               // P . V issue (its own warp)
    static constexpr int kThreads = HG == 16 ? 320 : HG == 32 ? 384 : 256;
    static constexpr int kSCols = kWide ? kTileRows : HG;          // columns of one score buffer
    static constexpr uint32_t kTmemS = 0;                          // scores [buf] at columns kSCols*buf
    static constexpr uint32_t kTmemO = 2 * kSCols;                 // O^T block j at kTmemO + kPVHeads*j
    static constexpr uint32_t kTmemCols = HG == 16 ? 256 : 512;
    static_assert(kTileRows % 16 == 0 && kTileRows <= 128, "tile rows: whole k-steps, at most M=128");
    static_assert(kChunkBytes % 1024 == 0, "chunks stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(kTmemO + 4 * kPVHeads <= kTmemCols, "tensor memory holds S and O");
    static_assert(!kWide || (kTileRows == 64 && kPBytes == kChunkBytes),
                  "wide: a tile's P_hi^T (64 head lines of 64 rows) fits its rope chunk exactly");
};

template <int HG>
struct __align__(1024) SharedStorage {
    using C = Cfg<HG>;
    uint8_t kv[2][C::kTileBytes];         // double-buffered tile (chunk c of buffer b at kv[b] + c*kChunkBytes)
    uint8_t q[C::kQBytes];                // Q^T: also absorbs the M=128 over-read of the last chunk
    uint8_t p[2][C::kPBytes];             // [P_hi | P_lo]^T, K-major, per tile buffer
    alignas(16) float red_max[C::kWGs][2][4][16];
    alignas(16) float red_sum[C::kWGs][4][16];
    int valid[2][C::kTileRows];
    long long rowid[2][C::kTileRows];     // sparse: the tile's absolute cache rows (-1 = masked)
    uint64_t full[2][kGroups], empty[2], s_full[2], p_full[2], o_done[2];
    uint64_t q_full, q_empty, o_free, mma_done[2];
    uint64_t stall_bar;                   // test hook: a barrier nothing arrives at
    uint64_t patch_bar;                   // fused append: the tile holding the new row landed
    uint32_t tmem_base;
    int abort_flag;
};

// Wide head group: the rope chunk of each tile buffer takes the tile's P_hi^T
// once its scores are taken; P_lo^T has one buffer of its own.
template <>
struct __align__(1024) SharedStorage<64> {
    using C = Cfg<64>;
    uint8_t kv[2][C::kTileBytes];         // chunk c of buffer b at kv[b] + c*kChunkBytes; chunk 8 -> P_hi^T
    uint8_t q[C::kQBytes];                // Q, K-major: head lines of 128 bytes per 64-column chunk
    uint8_t p_lo[C::kPBytes];             // P_lo^T
    alignas(16) float alpha[64];          // per-head factors of a rescale of O
    alignas(16) float inv_l[64];          // 1 / row sum per head, for the partial
    uint64_t p_hi_full[2];                // P_hi^T of the tile written (its P . V MMAs may start)
    uint64_t full[2][kGroups], empty[2], s_full[2], p_full[2], o_done[2];
    uint64_t q_full, q_empty, o_free, mma_done[2];
    uint64_t stall_bar;
    uint64_t patch_bar;
    uint32_t tmem_base;
    int abort_flag;
};

// 227 KB of dynamic shared memory per CTA, 1 KB of it kept for aligning the window
constexpr size_t kMaxDynamicSmem = 227 * 1024;
static_assert(sizeof(SharedStorage<16>) + 1024 <= kMaxDynamicSmem, "head group 16 fits shared memory");
static_assert(sizeof(SharedStorage<32>) + 1024 <= kMaxDynamicSmem, "head group 32 fits shared memory");
static_assert(sizeof(SharedStorage<64>) + 1024 <= kMaxDynamicSmem, "head group 64 fits shared memory");

struct Item {
    int b, hg, s, n_tiles;
    int e0, e1;                           // entries [e0, e1) of the request
    long long base;                       // first cache row of the request
};

template <int HG>
__device__ __forceinline__ Item decode_item(const PartialParams& p, int item) {
    Item it;
    const uint32_t ui = static_cast<uint32_t>(item);
    const uint32_t rest = ui / static_cast<uint32_t>(p.n_groups);
    it.hg = static_cast<int>(ui - rest * static_cast<uint32_t>(p.n_groups));
    const uint32_t b = rest / static_cast<uint32_t>(p.splits);
    it.s = static_cast<int>(rest - b * static_cast<uint32_t>(p.splits));
    it.b = static_cast<int>(b);
    // the kernel runs only on caches below 2^31 rows, so counts fit 32 bits
    const uint32_t n = static_cast<uint32_t>(
        request_entries(p.sparse, p.topk, p.d_pos, p.row_offset, p.kv_rows, it.b, &it.base));
    const uint32_t per = slice_entries_u32(n, static_cast<uint32_t>(p.splits), kTcGranule);
    uint32_t e0 = static_cast<uint32_t>(it.s) * per;
    uint32_t e1 = e0 + per;
    if (e1 > n) e1 = n;
    if (e0 > e1) e0 = e1;
    it.e0 = static_cast<int>(e0);
    it.e1 = static_cast<int>(e1);
    it.n_tiles = static_cast<int>((e1 - e0 + Cfg<HG>::kTileRows - 1) / Cfg<HG>::kTileRows);
    return it;
}

template <int HG>
__device__ __forceinline__ int rows_in_tile(const Item& it, int k) {
    constexpr int TR = Cfg<HG>::kTileRows;
    const int left = it.e1 - (it.e0 + k * TR);
    return left < TR ? left : TR;
}

__device__ __forceinline__ int item_key(const PartialParams& p, const Item& it) { return it.b * p.n_groups + it.hg; }

// Query tile of the CTA's first item: known without the context length.
__device__ __forceinline__ int first_key(const PartialParams& p) {
    const int item = static_cast<int>(blockIdx.x);
    const int rest = item / p.n_groups;
    return (rest / p.splits) * p.n_groups + (item - rest * p.n_groups);
}

__device__ __forceinline__ void raise_device_error(int* abort_flag, int* status) {
    *abort_flag = 1;
    if (status) atomicCAS(status, 0, static_cast<int>(MLA_EDEVICE));
}

// A cursor over this CTA's tiles in order: (item, tile k within it, global
// tile number g).
struct Cursor {
    int item, k, g;
    bool valid;
    Item it;
};

template <int HG>
__device__ __forceinline__ void cursor_next_item(const PartialParams& p, Cursor& c) {
    for (int i = c.item + static_cast<int>(gridDim.x); i < p.n_items; i += gridDim.x) {
        const Item it = decode_item<HG>(p, i);
        if (it.n_tiles > 0) {
            c.item = i;
            c.it = it;
            c.k = 0;
            c.valid = true;
            return;
        }
    }
    c.valid = false;
}
template <int HG>
__device__ __forceinline__ void cursor_init(const PartialParams& p, Cursor& c) {
    c.item = static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x);
    c.g = 0;
    c.k = 0;
    cursor_next_item<HG>(p, c);
}
template <int HG>
__device__ __forceinline__ void cursor_step(const PartialParams& p, Cursor& c) {
    ++c.g;
    if (++c.k == c.it.n_tiles) cursor_next_item<HG>(p, c);
}
template <int HG>
__device__ __forceinline__ int cursor_row(const Cursor& c) {
    return static_cast<int>(c.it.base) + c.it.e0 + c.k * Cfg<HG>::kTileRows;
}

// Sparse: the request-local id of row t of a tile (or -1 past its rows),
// with what it is checked against; fetched a tile ahead of its use so the
// index load is off the gather's critical path.
struct IdSlot {
    int id, seg, rows;
    long long base;
    bool valid;
};
template <int HG>
__device__ __forceinline__ IdSlot fetch_id(const PartialParams& p, const Cursor& c, int seg, int t) {
    IdSlot s;
    s.valid = c.valid;
    s.id = -1;
    s.seg = seg;
    s.rows = 0;
    s.base = 0;
    if (c.valid) {
        s.rows = rows_in_tile<HG>(c.it, c.k);
        s.base = c.it.base;
        if (t < s.rows)
            s.id = p.indices[static_cast<long long>(c.it.b) * p.topk + c.it.e0 + c.k * Cfg<HG>::kTileRows + t];
    }
    return s;
}
// The absolute cache row of a fetched id, or -1 when the id is masked.
__device__ __forceinline__ long long id_row(const PartialParams& p, const IdSlot& s) {
    const long long row = s.base + s.id;
    return (s.id >= 0 && s.id < s.seg && row >= 0 && row < p.kv_rows) ? row : -1;
}

template <int HG>
__device__ __forceinline__ void load_q(const TcMaps& maps, const PartialParams& p, SharedStorage<HG>& sh, int key,
                                       uint64_t policy) {
    const int b = key / p.n_groups;
    const int hg = key - b * p.n_groups;
    mbar_arrive_expect_tx(&sh.q_full, Cfg<HG>::kQBytes);
    tma_load_3d(sh.q, &maps.q, 0, b * p.heads + hg * HG, 0, &sh.q_full, policy);
}

// ============================== producer ==================================
// Query tiles: the first one is requested by a thread of the P . V warp at
// kernel start (before the context length is known, and off the producer's
// path); the producer and the score-MMA thread follow the same sequence of
// keys (a new load whenever the next busy item's key differs), and the MMA
// thread releases a tile through q_empty before the next one is loaded over it.
template <int HG>
__device__ void producer(const TcMaps& maps, const PartialParams& p, SharedStorage<HG>& sh, int t) {
    using C = Cfg<HG>;
    constexpr int TR = C::kTileRows;
    if (!p.sparse && t != 0) return;
    const uint64_t pol_q = l2_policy_evict_normal();
    int q_key = first_key(p);
    const uint64_t pol_kv = l2_policy_evict_first();
    int q_loads = 1;
    int patch_uses = 0;                                  // fused append: tiles patched so far
    Cursor cur;
    cursor_init<HG>(p, cur);
    // L2 prefetch runs two tiles ahead of the shared-memory loads (dense); the
    // sparse gather prefetches the next tile's rows
    Cursor nx = cur;
    if (nx.valid) cursor_step<HG>(p, nx);
    Cursor pf = nx;
    if (pf.valid) cursor_step<HG>(p, pf);
    // sparse: ids of this tile and the next, the segment length of the item the
    // prefetch cursor is in
    IdSlot id_cur{}, id_nx{};
    int pf_seg = 0;
    if (p.sparse && t < TR) {
        const int seg0 = cur.valid ? p.cache_len[cur.it.b] : 0;
        const int seg1 = nx.valid ? (nx.it.b == cur.it.b ? seg0 : p.cache_len[nx.it.b]) : 0;
        pf_seg = pf.valid ? (pf.it.b == nx.it.b ? seg1 : p.cache_len[pf.it.b]) : 0;
        id_cur = fetch_id<HG>(p, cur, seg0, t);
        id_nx = fetch_id<HG>(p, nx, seg1, t);
    }
    // `stop` is uniform over the producer threads (sparse: agreed at a barrier)
    bool stop = false;
    while (cur.valid && !stop) {
        const Item& it = cur.it;
        const int g = cur.g;
        const int k = cur.k;
        if (k == 0) {
            const int key = item_key(p, it);
            if (key != q_key) {
                if (t == 0) {
                    if (!mbar_wait_bounded(&sh.q_empty, (q_loads - 1) & 1, &sh.abort_flag))
                        raise_device_error(&sh.abort_flag, p.status);
                    else
                        load_q<HG>(maps, p, sh, key, pol_q);
                }
                q_key = key;
                ++q_loads;
            }
        }
        const int buf = g & 1;
        if (t == 0 && g >= 2 && !mbar_wait_bounded(&sh.empty[buf], ((g >> 1) - 1) & 1, &sh.abort_flag))
            raise_device_error(&sh.abort_flag, p.status);
        const int r0 = it.e0 + k * TR;
        if (!p.sparse) {
            stop = sh.abort_flag != 0;
            if (stop) break;
            const int y = static_cast<int>(it.base) + r0;
            // fused append: the tile holding entry d_pos[b] of the request lands on
            // the patch barrier; that row is then overwritten with the new row and
            // the tile handed on through its three barriers
            int patch_r = -1;
            if (p.new_rows) {
                const long long dp = p.d_pos[it.b];
                if (dp >= r0 && dp < r0 + rows_in_tile<HG>(it, k)) patch_r = static_cast<int>(dp - r0);
            }
            if (patch_r < 0) {
#pragma unroll
                for (int grp = 0; grp < kGroups; ++grp) {
                    mbar_arrive_expect_tx(&sh.full[buf][grp], C::kGroupBytes);
                    tma_load_3d(sh.kv[buf] + grp * C::kGroupBytes, &maps.kv, 0, y, grp * kTcBoxChunks,
                                &sh.full[buf][grp], pol_kv);
                }
            } else {
                mbar_arrive_expect_tx(&sh.patch_bar, C::kTileBytes);
#pragma unroll
                for (int grp = 0; grp < kGroups; ++grp)
                    tma_load_3d(sh.kv[buf] + grp * C::kGroupBytes, &maps.kv, 0, y, grp * kTcBoxChunks, &sh.patch_bar,
                                pol_kv);
                volatile int never = 0;
                const bool landed = mbar_wait_bounded(&sh.patch_bar, patch_uses & 1, &never);
                ++patch_uses;
                if (!landed) {
                    raise_device_error(&sh.abort_flag, p.status);
                    break;
                }
                const uint4* src = reinterpret_cast<const uint4*>(p.new_rows + static_cast<long long>(it.b) * kDRow);
                const uint32_t row = smem_u32(sh.kv[buf]) + patch_r * 128;
                for (int u = 0; u < kRowBytes / 16; ++u) {
                    const uint4 v = src[u];
                    st_shared_v4(row + (u >> 3) * C::kChunkBytes + (((u & 7) ^ (patch_r & 7)) << 4), v.x, v.y, v.z,
                                 v.w);
                }
                fence_proxy_async_smem();            // the tensor cores read it next
#pragma unroll
                for (int grp = 0; grp < kGroups; ++grp) mbar_arrive(&sh.full[buf][grp]);
            }
            if (pf.valid) {
                const int yp = cursor_row<HG>(pf);
#pragma unroll
                for (int grp = 0; grp < kGroups; ++grp) tma_prefetch_3d(&maps.kv, 0, yp, grp * kTcBoxChunks);
            }
        } else if constexpr (HG == 16) {
            const int rows = rows_in_tile<HG>(it, k);
            // the buffer is free, or some thread saw the CTA abort
            stop = named_barrier_or(kBarProducer, kProducerThreads, sh.abort_flag != 0);
            if (stop) break;
            // the tile's row ids (fetched a tile ago), resolved once into shared memory
            if (t < TR) {
                const long long row = id_row(p, id_cur);
                sh.rowid[buf][t] = row;
                sh.valid[buf][t] = row >= 0 ? 1 : 0;
            }
            named_barrier_sync(kBarProducer, kProducerThreads);      // row ids ready
            // rows past the tile's last k-step are never read by P . V; masked
            // rows inside it must hold zeros (they meet p = 0)
            const int rows_read = (rows + 15) & ~15;
            const uint32_t dst0 = smem_u32(sh.kv[buf]);
            const uint8_t* kvb = reinterpret_cast<const uint8_t*>(p.kv);
            const long long stride_bytes = p.row_stride * 2;
            constexpr int kUnits = kGroupsPerBatch * kTcBoxChunks * 8;  // 16-byte units of a row per batch
#pragma unroll
            for (int bt = 0; bt < kGatherBatches; ++bt) {
#pragma unroll 4
                for (int piece = t; piece < rows_read * kUnits; piece += kProducerThreads) {
                    const int r = piece / kUnits;
                    const int u = bt * kUnits + (piece - r * kUnits);
                    const int c = u >> 3;
                    const uint32_t dst = dst0 + c * C::kChunkBytes + r * 128 + ((((u & 7) ^ (r & 7))) << 4);
                    const long long row = sh.rowid[buf][r];
                    if (row >= 0)
                        cp_async_16(dst, kvb + row * stride_bytes + u * 16);
                    else
                        st_shared_v4_zero(dst);
                }
                cp_async_commit();
            }
            if (t < TR) {
                // the next tile's rows into L2 while this tile's copies land, and
                // the ids of the tile after it
                const long long nrow = id_nx.valid ? id_row(p, id_nx) : -1;
                if (nrow >= 0) bulk_prefetch_l2(kvb + nrow * stride_bytes, kRowBytes);
                id_cur = id_nx;
                id_nx = fetch_id<HG>(p, pf, pf_seg, t);
            }
            static_assert(kGatherBatches == 3, "three commit groups per tile");
            cp_async_wait_group<2>();
            fence_proxy_async_smem();
#pragma unroll
            for (int i = 0; i < kGroupsPerBatch; ++i) mbar_arrive(&sh.full[buf][i]);
            cp_async_wait_group<1>();
            fence_proxy_async_smem();
#pragma unroll
            for (int i = 0; i < kGroupsPerBatch; ++i) mbar_arrive(&sh.full[buf][kGroupsPerBatch + i]);
            cp_async_wait_group<0>();
            fence_proxy_async_smem();
#pragma unroll
            for (int i = 0; i < kGroupsPerBatch; ++i) mbar_arrive(&sh.full[buf][2 * kGroupsPerBatch + i]);
        }
        if (pf.valid) {
            const int b_before = pf.it.b;
            cursor_step<HG>(p, pf);
            if (p.sparse && t < TR && pf.valid && pf.it.b != b_before) pf_seg = p.cache_len[pf.it.b];
        }
        if (nx.valid) cursor_step<HG>(p, nx);
        cursor_step<HG>(p, cur);
    }
    // Never retire the CTA with copies into its shared memory in flight.
    if (t == 0) {
        volatile int never = 0;
        const int g = cur.g;                             // tiles issued
        for (int b = 0; b < 2 && b < g; ++b) {
            const int last = g - 1 - ((g - 1 - b) & 1);    // last tile number that used buffer b
            for (int grp = 0; grp < kGroups; ++grp)
                if (!mbar_wait_bounded(&sh.full[b][grp], (last >> 1) & 1, &never))
                    raise_device_error(&sh.abort_flag, p.status);
        }
        if (!mbar_wait_bounded(&sh.q_full, (q_loads - 1) & 1, &never)) raise_device_error(&sh.abort_flag, p.status);
    }
}

// ============================== MMA issue ==================================
// Two threads in two warps issue the MMAs (the tensor pipe overlaps
// instructions from different issuers, and a waiting issuer does not stall
// the other): the scores of each tile, and the P . V products.  QK of tile g
// waits for each third of its tile and for the softmax of tile g-2 (the
// owner of its score buffer); P . V of tile g waits for the softmax of tile
// g (wide: its P_hi products for P_hi, its P_lo products for P_lo), and the
// first one of an item for the previous item's epilogue.
template <int HG>
__device__ void mma_issue_qk(const PartialParams& p, SharedStorage<HG>& sh, uint32_t tmem) {
    using C = Cfg<HG>;
    // swapped: M = 128 cache rows, N = HG heads; wide: M = 64 heads, N = TR rows
    const uint32_t idesc_qk = C::kWide ? make_idesc_bf16(64, C::kTileRows, 0, 0) : make_idesc_bf16(128, HG, 0, 0);
    // K-major 128-byte-swizzled operands: 8-row groups 1024 bytes apart
    const uint64_t kv_desc0 = make_sdesc(smem_u32(sh.kv[0]), 16, 1024, kLayoutSw128);
    const uint64_t q_desc0 = make_sdesc(smem_u32(sh.q), 16, 1024, kLayoutSw128);
    Cursor qc;
    cursor_init<HG>(p, qc);
    int q_key = first_key(p);
    int q_phase = 0;
    bool q_ready = false;
    // test hook: a wait that runs out, so every role takes the abort path
    bool ok = !(p.stall_test && !mbar_wait_bounded(&sh.stall_bar, 0, &sh.abort_flag, kStallTestCycles));
    while (qc.valid && ok) {
        const int key = item_key(p, qc.it);
        const int buf = qc.g & 1;
        if (key != q_key) {
            // the producer loads the next query tile over this one: it must have
            // landed (never read, possibly) and its MMAs must be complete
            if (!q_ready && !mbar_wait_bounded(&sh.q_full, q_phase & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            umma_commit(&sh.q_empty);
            ++q_phase;
            q_key = key;
            q_ready = false;
        }
        if (!q_ready) {
            if (!mbar_wait_bounded(&sh.q_full, q_phase & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            q_ready = true;
        }
        if (qc.g >= 2 && !mbar_wait_bounded(&sh.p_full[buf], ((qc.g >> 1) - 1) & 1, &sh.abort_flag)) {
            ok = false;
            break;
        }
        const uint64_t kb = kv_desc0 + ((static_cast<uint32_t>(buf) * C::kTileBytes) >> 4);
        // fully unrolled: every descriptor is a constant offset from kb / q_desc0,
        // so the issuing thread keeps pace with the tensor pipe
#pragma unroll
        for (int grp = 0; grp < kGroups; ++grp) {
            if (!mbar_wait_bounded(&sh.full[buf][grp], (qc.g >> 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
#pragma unroll
            for (int cc = 0; cc < kTcBoxChunks; ++cc) {
                const int c = grp * kTcBoxChunks + cc;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t off = (c * C::kChunkBytes + kk * 32u) >> 4;
                    const uint32_t qoff = (c * C::kQChunkBytes + kk * 32u) >> 4;
                    if constexpr (C::kWide) {
                        // S[heads x rows]: A = the 64 query lines, B = the tile's rows
                        umma_bf16(tmem + C::kTmemS + C::kSCols * buf, q_desc0 + qoff, kb + off, idesc_qk,
                                  (c | kk) ? 1u : 0u);
                    } else {
                        umma_bf16(tmem + C::kTmemS + C::kSCols * buf, kb + off, q_desc0 + qoff, idesc_qk,
                                  (c | kk) ? 1u : 0u);
                    }
                }
            }
        }
        if (!ok) break;
        umma_commit(&sh.s_full[buf]);
        cursor_step<HG>(p, qc);
    }
    if (!ok) raise_device_error(&sh.abort_flag, p.status);
    umma_commit(&sh.mma_done[0]);
    volatile int never = 0;
    if (!mbar_wait_bounded(&sh.mma_done[0], 0, &never)) raise_device_error(&sh.abort_flag, p.status);
}

template <int HG>
__device__ void mma_issue_pv(const PartialParams& p, SharedStorage<HG>& sh, uint32_t tmem) {
    using C = Cfg<HG>;
    constexpr int TR = C::kTileRows;
    const uint32_t idesc_pv = make_idesc_bf16(128, C::kPVHeads, 1, 0);
    // P^T, K-major: head lines of 128 bytes (64 rows), 8-line groups 1024 apart
    uint64_t p_desc0, plo_desc = 0;
    if constexpr (C::kWide) {
        p_desc0 = make_sdesc(smem_u32(sh.kv[0] + (kChunks - 1) * C::kChunkBytes), 16, 1024, kLayoutSw128);
        plo_desc = make_sdesc(smem_u32(sh.p_lo), 16, 1024, kLayoutSw128);
    } else {
        p_desc0 = make_sdesc(smem_u32(sh.p[0]), 16, 1024, kLayoutSw128);
    }
    // V^T is MN-major: 64-feature atoms one chunk apart, 8-row groups 1024 apart
    const uint64_t v_desc0 = make_sdesc(smem_u32(sh.kv[0]), C::kChunkBytes, 1024, kLayoutSw128);
    Cursor pc;
    cursor_init<HG>(p, pc);
    int items_done = 0;
    bool ok = true;
    while (pc.valid && ok) {
        const int buf = pc.g & 1;
        const bool first = pc.k == 0;
        uint64_t* p_ready;                   // wide: P_hi first (P_lo is waited for below)
        if constexpr (C::kWide)
            p_ready = &sh.p_hi_full[buf];
        else
            p_ready = &sh.p_full[buf];
        if (!mbar_wait_bounded(p_ready, (pc.g >> 1) & 1, &sh.abort_flag) ||
            (first && items_done > 0 && !mbar_wait_bounded(&sh.o_free, (items_done - 1) & 1, &sh.abort_flag))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const int ksteps = (rows_in_tile<HG>(pc.it, pc.k) + 15) >> 4;
        const uint64_t vb = v_desc0 + ((static_cast<uint32_t>(buf) * C::kTileBytes) >> 4);
        [[maybe_unused]] const uint64_t pb = p_desc0 + ((static_cast<uint32_t>(buf) * C::kPBytes) >> 4);
        const uint32_t acc0 = first ? 0u : 1u;
        if constexpr (C::kWide) {
            // P_hi^T (over the tile's rope chunk) into every block, then P_lo^T (its
            // own buffer, written once the previous tile's products are done)
            const uint64_t phi = p_desc0 + ((static_cast<uint32_t>(buf) * C::kTileBytes) >> 4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int kk = 0; kk < TR / 16; ++kk) {
                    if (kk < ksteps) {
                        const uint64_t a = vb + ((2u * j * C::kChunkBytes + kk * 2048u) >> 4);
                        umma_bf16(tmem + C::kTmemO + C::kPVHeads * j, a, phi + ((kk * 32u) >> 4), idesc_pv,
                                  kk == 0 ? acc0 : 1u);
                    }
                }
            }
            if (!mbar_wait_bounded(&sh.p_full[buf], (pc.g >> 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int kk = 0; kk < TR / 16; ++kk) {
                    if (kk < ksteps) {
                        const uint64_t a = vb + ((2u * j * C::kChunkBytes + kk * 2048u) >> 4);
                        umma_bf16(tmem + C::kTmemO + C::kPVHeads * j, a, plo_desc + ((kk * 32u) >> 4), idesc_pv, 1u);
                    }
                }
            }
        } else if (ksteps == TR / 16) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int kk = 0; kk < TR / 16; ++kk) {
                    const uint64_t a = vb + ((2u * j * C::kChunkBytes + kk * 2048u) >> 4);
                    const uint64_t bd =
                        pb + ((static_cast<uint32_t>(kk >> 2) * C::kPAtomBytes + (kk & 3) * 32u) >> 4);
                    umma_bf16(tmem + C::kTmemO + C::kPVHeads * j, a, bd, idesc_pv, kk == 0 ? acc0 : 1u);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int kk = 0; kk < TR / 16; ++kk) {
                    if (kk < ksteps) {
                        const uint64_t a = vb + ((2u * j * C::kChunkBytes + kk * 2048u) >> 4);
                        const uint64_t bd =
                            pb + ((static_cast<uint32_t>(kk >> 2) * C::kPAtomBytes + (kk & 3) * 32u) >> 4);
                        umma_bf16(tmem + C::kTmemO + C::kPVHeads * j, a, bd, idesc_pv, kk == 0 ? acc0 : 1u);
                    }
                }
            }
        }
        umma_commit(&sh.empty[buf]);
        umma_commit(&sh.o_done[buf]);
        if (pc.k == pc.it.n_tiles - 1) ++items_done;
        cursor_step<HG>(p, pc);
    }
    if (!ok) raise_device_error(&sh.abort_flag, p.status);
    umma_commit(&sh.mma_done[1]);
    volatile int never = 0;
    if (!mbar_wait_bounded(&sh.mma_done[1], 0, &never)) raise_device_error(&sh.abort_flag, p.status);
}

// ============================== softmax warps ==============================
__device__ __forceinline__ void warp_sum16(float (&v)[16], int lane) {
    // After the halving steps lane L holds head (L >> 1); the last step joins the pair.
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

// The four warps of a softmax warpgroup meet at their own hardware barrier; a
// bounded wait that ran out in any of them turns the barrier's OR true, and
// then all 128 threads leave together (a thread that left alone would strand
// the others).
__device__ __forceinline__ bool softmax_barrier_or(int wg, bool pred) {
    return named_barrier_or(kBarSoftmax0 + wg, kSoftmaxThreads, pred);
}

// Warpgroup wg handles heads 16 wg .. 16 wg + 15 of the group; warp q of it
// owns tile rows 32 q .. 32 q + 31 (tensor-memory lanes of warp q mod 4).
template <int HG>
__device__ void softmax_warps(const PartialParams& p, SharedStorage<HG>& sh, uint32_t tmem, int wg, int q, int lane) {
    using C = Cfg<HG>;
    constexpr int TR = C::kTileRows;
    const int t = q * 32 + lane;                     // tile row / TMEM lane of this thread
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const bool has_rows = q * 32 < TR;               // warp-uniform
    const int h_off = 16 * wg;                       // this warpgroup's heads within the group
    int g = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it = decode_item<HG>(p, item);
        const long long row0 = (static_cast<long long>(it.b) * p.heads + it.hg * HG + h_off) * p.splits + it.s;
        if (it.n_tiles == 0) {
            write_empty_partial(p.o_part, p.lse_part, row0, p.splits, t, kSoftmaxThreads);
            continue;
        }
        float m_ref[16], l_part[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
            m_ref[h] = -INFINITY;
            l_part[h] = 0.f;
        }
        const int first_g = g;
        for (int k = 0; k < it.n_tiles; ++k, ++g) {
            const int buf = g & 1;
            const int rows = rows_in_tile<HG>(it, k);
            // scores of tile g; sparse: the producer's row flags; P buffer free (P . V of g-2 done)
            bool w = mbar_wait_bounded(&sh.s_full[buf], (g >> 1) & 1, &sh.abort_flag);
            if (p.sparse) w = w && mbar_wait_bounded(&sh.full[buf][0], (g >> 1) & 1, &sh.abort_flag);
            if (g >= 2) w = w && mbar_wait_bounded(&sh.o_done[buf], ((g >> 1) - 1) & 1, &sh.abort_flag);
            w = __all_sync(0xffffffffu, w);
            tc_fence_after_sync();
            float s[16];
            if (w && has_rows) {
                tmem_ld16(tmem + lane_addr + C::kTmemS + C::kSCols * buf + h_off, s);
            } else {
#pragma unroll
                for (int h = 0; h < 16; ++h) s[h] = 0.f;
            }
            bool row_ok;
            if (p.sparse) {
                row_ok = t < rows && sh.valid[buf][t] != 0;
            } else {
                const long long row = it.base + it.e0 + k * TR + t;
                row_ok = t < rows && row >= 0 && row < p.kv_rows;
            }
            bool need = !w;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                s[h] = row_ok ? s[h] * p.scale_log2 : -INFINITY;
                need |= s[h] > m_ref[h] + kRescaleLog2;             // false for masked rows and -inf refs alike
            }
            float alpha[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) alpha[h] = 1.f;
            if (softmax_barrier_or(wg, need)) {
                // ---- tile max per head: warp max, then the four warps through shared memory
                float mine = -INFINITY;
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const float r = warp_max_f32(s[h]);
                    if (lane == h) mine = r;
                }
                if (lane < 16) sh.red_max[wg][buf][q][lane] = mine;
                if (softmax_barrier_or(wg, !w)) {
                    ok = false;
                    break;
                }
                bool rescale = false;
                const float4* rm = reinterpret_cast<const float4*>(&sh.red_max[wg][buf][0][0]);
#pragma unroll
                for (int h4 = 0; h4 < 4; ++h4) {
                    const float4 a = rm[h4], b = rm[4 + h4], c = rm[8 + h4], d = rm[12 + h4];
                    const float tm[4] = {fmaxf(fmaxf(a.x, b.x), fmaxf(c.x, d.x)), fmaxf(fmaxf(a.y, b.y), fmaxf(c.y, d.y)),
                                         fmaxf(fmaxf(a.z, b.z), fmaxf(c.z, d.z)), fmaxf(fmaxf(a.w, b.w), fmaxf(c.w, d.w))};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        // the reference moves to the tile max when that exceeds it by
                        // more than 2^8 (or nothing was referenced yet); sums and O taken
                        // against a finite old reference are scaled to the new one
                        const int h = 4 * h4 + i;
                        const float ref = m_ref[h];
                        const bool move = tm[i] > ref + kRescaleLog2;     // false while the tile max is -inf
                        const float nref = move ? tm[i] : ref;
                        const bool scale = move && ref > -INFINITY;
                        alpha[h] = scale ? ex2_approx(ref - nref) : 1.f;
                        rescale |= scale;
                        m_ref[h] = nref;
                    }
                }
                if (rescale && g > first_g) {
                    // ---- rare: O holds earlier tiles of this slice; move it to the new reference
                    const int gp = g - 1;
                    bool w2 = mbar_wait_bounded(&sh.o_done[gp & 1], (gp >> 1) & 1, &sh.abort_flag);
                    w2 = __all_sync(0xffffffffu, w2);
                    if (softmax_barrier_or(wg, !w2)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t a = tmem + lane_addr + C::kTmemO + C::kPVHeads * j + h_off;
                        float hi[16], lo[16];
                        tmem_ld16(a, hi);
                        tmem_ld16(a + HG, lo);
#pragma unroll
                        for (int h = 0; h < 16; ++h) {
                            hi[h] *= alpha[h];
                            lo[h] *= alpha[h];
                        }
                        tmem_st16(a, hi);
                        tmem_st16(a + HG, lo);
                    }
                }
            }

            // ---- probabilities, written as the bf16 pair [P_hi | P_lo]^T ----------
            float pr[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) pr[h] = (row_ok && m_ref[h] > -INFINITY) ? ex2_approx(s[h] - m_ref[h]) : 0.f;
            if (t < TR) {
                // row t of head h: line h_off + h (hi) / HG + h_off + h (lo) of the K atom
                // t / 64, byte 2 * (t % 64); lines are 128 bytes, 8-line groups 1024 apart
                const uint32_t pbase = smem_u32(sh.p[buf]) + (t >> 6) * C::kPAtomBytes + h_off * 128 + 2u * (t & 7);
                const uint32_t unit = static_cast<uint32_t>((t & 63) >> 3);
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const __nv_bfloat16 hi = __float2bfloat16_rn(pr[h]);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(pr[h] - __bfloat162float(hi));
                    const uint32_t a = pbase + (h >> 3) * 1024 + (h & 7) * 128 + ((unit ^ (h & 7)) << 4);
                    st_shared_u16(a, __bfloat16_as_ushort(hi));
                    st_shared_u16(a + HG * 128, __bfloat16_as_ushort(lo));
                }
            }
#pragma unroll
            for (int h = 0; h < 16; ++h) l_part[h] = l_part[h] * alpha[h] + pr[h];
            // ---- dense: masked rows the P . V k-steps read must hold zeros ---------
            if (!p.sparse && wg == 0 && t < TR && !row_ok && t < ((rows + 15) & ~15)) {
                const uint32_t row_base = smem_u32(sh.kv[buf]) + t * 128;
#pragma unroll 1
                for (int c = 0; c < 8; ++c)
#pragma unroll
                    for (int u = 0; u < 8; ++u) st_shared_v4_zero(row_base + c * C::kChunkBytes + u * 16);
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&sh.p_full[buf]);
        }
        if (!ok) break;

        // ---- epilogue: l = sum of the rows' sums (fixed order), O = (O_hi + O_lo) / l,
        //      lse = m + log2(l) (to natural log).  The sums and lse do not need
        //      the last P . V, so they are formed while it runs. -----------------
        {
            float red[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) red[h] = l_part[h];
            warp_sum16(red, lane);
            if ((lane & 1) == 0) sh.red_sum[wg][q][lane >> 1] = red[0];
        }
        named_barrier_sync(kBarSoftmax0 + wg, kSoftmaxThreads);
        float l_run[16];
        {
            const float4* rs = reinterpret_cast<const float4*>(&sh.red_sum[wg][0][0]);
#pragma unroll
            for (int h4 = 0; h4 < 4; ++h4) {
                const float4 a = rs[h4], b = rs[4 + h4], c = rs[8 + h4], d = rs[12 + h4];
                l_run[4 * h4 + 0] = ((a.x + b.x) + c.x) + d.x;
                l_run[4 * h4 + 1] = ((a.y + b.y) + c.y) + d.y;
                l_run[4 * h4 + 2] = ((a.z + b.z) + c.z) + d.z;
                l_run[4 * h4 + 3] = ((a.w + b.w) + c.w) + d.w;
            }
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
        float inv[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) inv[h] = l_run[h] > 0.f ? __frcp_rn(l_run[h]) : 0.f;
        const int gl = g - 1;
        bool w = mbar_wait_bounded(&sh.o_done[gl & 1], (gl >> 1) & 1, &sh.abort_flag);
        w = __all_sync(0xffffffffu, w);
        if (softmax_barrier_or(wg, !w)) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        float* o_row = p.o_part + row0 * kDLatent + t;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            float hi[16], lo[16];                         // features 128 j + t of the 16 heads
            const uint32_t a = tmem + lane_addr + C::kTmemO + C::kPVHeads * j + h_off;
            if constexpr (HG == 16) {
                float o[32];
                tmem_ld32(a, o);
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    hi[h] = o[h];
                    lo[h] = o[16 + h];
                }
            } else {
                tmem_ld16(a, hi);
                tmem_ld16(a + HG, lo);
            }
#pragma unroll
            for (int h = 0; h < 16; ++h)
                o_row[static_cast<long long>(h) * p.splits * kDLatent + 128 * j] = (hi[h] + lo[h]) * inv[h];
        }
        tc_fence_before_sync();
        mbar_arrive(&sh.o_free);
    }
    if (!ok && lane == 0) raise_device_error(&sh.abort_flag, p.status);
}

// ---- wide head group (64 heads): two softmax threads per head -------------
// The scores come from an M = 64 product, which places head 16i + j in
// tensor-memory lane 32i + j (i = 0..3, j = 0..15): warp i of the warpgroup
// reads heads 16i .. 16i + 15 in its lanes 0-15 and hands the tile's rows
// 32-63 of each head to lane j + 16 (shuffles), so every thread works on 32
// rows of one head.  The head's reference m is the same in both threads (the
// tile max is exchanged); each keeps the sum of its own rows, and the two
// sums are added once per slice.  For the rescales of O and the partial
// writes, tensor-memory lane 32i + lane is latent feature 128j + 32i + lane
// of block j.
__device__ __forceinline__ uint32_t bf16_rn_bits(float x) {
    // round-to-nearest-even to bf16 for finite x (the upper 16 bits of the result)
    const uint32_t b = __float_as_uint(x);
    return (b + 0x7fffu + ((b >> 16) & 1u)) >> 16;
}

__device__ void softmax_wide(const PartialParams& p, SharedStorage<64>& sh, uint32_t tmem, int q, int lane) {
    using C = Cfg<64>;
    constexpr int TR = C::kTileRows;
    constexpr int HG = 64;
    constexpr int RH = TR / 2;                       // rows of a tile per thread
    const int t = q * 32 + lane;                     // thread of the warpgroup (O^T lane in the epilogue)
    const int half = lane >> 4;                      // rows 32 * half .. 32 * half + 31 of the tile
    const int head = 16 * q + (lane & 15);           // head of this thread's scores
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t line = (static_cast<uint32_t>(head) >> 3) * 1024u + (static_cast<uint32_t>(head) & 7u) * 128u;
    const uint32_t swz = static_cast<uint32_t>(head) & 7u;
    int g = 0;
    bool ok = true;
    bool lo_wait_failed = false;                     // a P_lo wait that ran out, reported at the next barrier
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it = decode_item<HG>(p, item);
        const long long row0 = (static_cast<long long>(it.b) * p.heads + it.hg * HG) * p.splits + it.s;
        if (it.n_tiles == 0) {
            for (int k = 0; k < HG / kHeadGroup; ++k)
                write_empty_partial(p.o_part, p.lse_part, row0 + static_cast<long long>(k) * kHeadGroup * p.splits,
                                    p.splits, t, kSoftmaxThreads);
            continue;
        }
        float m_ref = -INFINITY;
        float l = 0.f;                               // sum over this thread's rows
        const int first_g = g;
        for (int k = 0; k < it.n_tiles; ++k, ++g) {
            const int buf = g & 1;
            const int rows = rows_in_tile<HG>(it, k);
            // rows at or past the end of the cache were zero-filled by the TMA unit and are masked
            const long long row_first = it.base + it.e0 + static_cast<long long>(k) * TR;
            const long long in_cache = p.kv_rows - row_first;
            const int valid = in_cache < rows ? static_cast<int>(in_cache > 0 ? in_cache : 0) : rows;
            bool w = mbar_wait_bounded(&sh.s_full[buf], (g >> 1) & 1, &sh.abort_flag) && !lo_wait_failed;
            w = __all_sync(0xffffffffu, w);
            tc_fence_after_sync();
            // raw scores of rows 32 * half + i (lanes 16-31 take theirs from lane - 16)
            float s[RH];
            {
                float v[RH], u[RH];                  // rows 0-31 / 32-63 of the lane's head (lanes 0-15)
                const uint32_t sa = tmem + lane_addr + C::kTmemS + C::kSCols * buf;
                if (w) {                             // warp-uniform (the loads are .sync.aligned)
                    tmem_ld32(sa, v);
                    tmem_ld32(sa + RH, u);
                }
#pragma unroll
                for (int i = 0; i < RH; ++i) {
                    const float x = __shfl_sync(0xffffffffu, u[i], lane & 15);
                    s[i] = (w && RH * half + i < valid) ? (half ? x : v[i]) : -INFINITY;
                }
            }
            float tmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < RH; ++i) tmax = fmaxf(tmax, s[i]);
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16)) * p.scale_log2;   // base-2 units (scale > 0)
            // false while the tile max is -inf (nothing attended yet, or all masked)
            const bool need = tmax > m_ref + kRescaleLog2;
            if (softmax_barrier_or(0, need || !w)) {
                if (softmax_barrier_or(0, sh.abort_flag != 0 || !w)) {
                    ok = false;
                    break;
                }
                // the reference of the head moves to its tile max; the row sums and O
                // (if it holds earlier tiles of this slice) are scaled to it
                float alpha = 1.f;
                if (need) {
                    alpha = m_ref > -INFINITY ? ex2_approx(m_ref - tmax) : 1.f;
                    m_ref = tmax;
                    l *= alpha;
                }
                if (softmax_barrier_or(0, alpha != 1.f && g > first_g)) {
                    if (half == 0) sh.alpha[head] = alpha;
                    const int gp = g - 1;
                    bool w2 = mbar_wait_bounded(&sh.o_done[gp & 1], (gp >> 1) & 1, &sh.abort_flag);
                    w2 = __all_sync(0xffffffffu, w2);
                    // (the barrier also publishes the factors)
                    if (softmax_barrier_or(0, !w2)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int j = 0; j < 4; ++j) {
#pragma unroll 1
                        for (int c = 0; c < HG; c += 16) {
                            const uint32_t a = tmem + lane_addr + C::kTmemO + C::kPVHeads * j + c;
                            float o[16];
                            tmem_ld16(a, o);
#pragma unroll
                            for (int h = 0; h < 16; ++h) o[h] *= sh.alpha[c + h];
                            tmem_st16(a, o);
                        }
                    }
                }
            }

            // ---- probabilities as the bf16 pair: P_hi^T into the tile's rope chunk
            //      (line = head, 64 rows x 2 bytes; this thread: units 4 half .. +3),
            //      P_lo^T into its buffer ---------------------------------------------
            uint32_t lo[RH / 2];
            {
                const float neg_m = m_ref > -INFINITY ? -m_ref : 0.f;    // m = -inf: every score is -inf
                const uint32_t hi_base = smem_u32(sh.kv[buf] + (kChunks - 1) * C::kChunkBytes) + line;
#pragma unroll
                for (int u = 0; u < RH / 8; ++u) {
                    uint32_t hi[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = 8 * u + 2 * i;
                        const float p0 = ex2_approx(fmaf(s[r], p.scale_log2, neg_m));   // masked: 2^-inf = 0
                        const float p1 = ex2_approx(fmaf(s[r + 1], p.scale_log2, neg_m));
                        l += p0;
                        l += p1;
                        hi[i] = pack_bf16x2(p0, p1);
                        const float r0 = p0 - __uint_as_float(hi[i] << 16);          // exact
                        const float r1 = p1 - __uint_as_float(hi[i] & 0xffff0000u);
                        lo[4 * u + i] = bf16_rn_bits(r0) | (bf16_rn_bits(r1) << 16);
                    }
                    const uint32_t unit = static_cast<uint32_t>(4 * half + u);
                    st_shared_v4(hi_base + ((unit ^ swz) << 4), hi[0], hi[1], hi[2], hi[3]);
                }
            }
            // ---- dense: masked rows inside the last k-step must hold zeros in V
            //      (they meet p = 0, and 0 * NaN would not vanish) --------------------
            {
                const int rows_read = (rows + 15) & ~15;
                const uint32_t base = smem_u32(sh.kv[buf]);
                for (int i = t; i < (rows_read - rows) * 64; i += kSoftmaxThreads) {
                    const int r = rows + (i >> 6);
                    const int c = (i >> 3) & 7;
                    st_shared_v4_zero(base + c * C::kChunkBytes + r * 128 + (i & 7) * 16);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&sh.p_hi_full[buf]);
            // P_lo^T has one buffer: the P . V of the previous tile must be done with it
            if (g > 0) {
                const int gp = g - 1;
                lo_wait_failed = !mbar_wait_bounded(&sh.o_done[gp & 1], (gp >> 1) & 1, &sh.abort_flag);
            }
            if (!lo_wait_failed) {
                const uint32_t lo_base = smem_u32(sh.p_lo) + line;
#pragma unroll
                for (int u = 0; u < RH / 8; ++u) {
                    const uint32_t unit = static_cast<uint32_t>(4 * half + u);
                    st_shared_v4(lo_base + ((unit ^ swz) << 4), lo[4 * u], lo[4 * u + 1], lo[4 * u + 2], lo[4 * u + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(&sh.p_full[buf]);
        }
        if (!ok) break;

        // ---- epilogue: lse = m + log2(l) (to natural log) per head, then every
        //      thread writes its latent feature of the 64 partials, O / l ------------
        const float l_head = l + __shfl_xor_sync(0xffffffffu, l, 16);   // the same sum in both threads
        if (half == 0) {
            p.lse_part[row0 + static_cast<long long>(head) * p.splits] =
                l_head > 0.f ? (m_ref + log2f(l_head)) * kLn2 : -INFINITY;
            sh.inv_l[head] = l_head > 0.f ? __frcp_rn(l_head) : 0.f;
        }
        const int gl = g - 1;
        bool w = mbar_wait_bounded(&sh.o_done[gl & 1], (gl >> 1) & 1, &sh.abort_flag) && !lo_wait_failed;
        w = __all_sync(0xffffffffu, w);
        if (softmax_barrier_or(0, !w)) {                 // (also publishes 1 / l)
            ok = false;
            break;
        }
        tc_fence_after_sync();
        {
            float* o_row = p.o_part + row0 * kDLatent + t;
            const long long head_stride = static_cast<long long>(p.splits) * kDLatent;
            // eight pieces (block j, heads c .. c + 31) of feature 128 j + t; the next
            // piece's tensor-memory load is in flight while this one is stored
            uint32_t ob[2][32];
            tmem_ld32_async(tmem + lane_addr + C::kTmemO, ob[0]);
            tmem_wait_ld32(ob[0]);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = i >> 1, c = 32 * (i & 1);
                if (i + 1 < 8)
                    tmem_ld32_async(tmem + lane_addr + C::kTmemO + C::kPVHeads * ((i + 1) >> 1) + 32 * ((i + 1) & 1),
                                    ob[(i + 1) & 1]);
                // the piece's 32 factors in registers (eight 16-byte loads, not one
                // shared-memory load per stored value: measured 40.3 -> 36.7 us per
                // call at H = 128, T = 32832)
                float il[32];
                const float4* ils = reinterpret_cast<const float4*>(sh.inv_l + c);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float4 f = ils[k];
                    il[4 * k] = f.x;
                    il[4 * k + 1] = f.y;
                    il[4 * k + 2] = f.z;
                    il[4 * k + 3] = f.w;
                }
#pragma unroll
                for (int h = 0; h < 32; ++h)
                    o_row[(c + h) * head_stride + 128 * j] = __uint_as_float(ob[i & 1][h]) * il[h];
                if (i + 1 < 8) tmem_wait_ld32(ob[(i + 1) & 1]);
            }
        }
        tc_fence_before_sync();
        mbar_arrive(&sh.o_free);
    }
    if (!ok && lane == 0) raise_device_error(&sh.abort_flag, p.status);
}

template <int HG>
__global__ void __launch_bounds__(Cfg<HG>::kThreads, 1) mla_partial_tc_kernel(const __grid_constant__ TcMaps maps,
                                                                               const PartialParams p) {
    using C = Cfg<HG>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SharedStorage<HG>& sh = *reinterpret_cast<SharedStorage<HG>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&maps.kv);
        prefetch_tensormap(&maps.q);
        for (int i = 0; i < 2; ++i) {
            for (int grp = 0; grp < kGroups; ++grp) mbar_init(&sh.full[i][grp], p.sparse ? kProducerThreads : 1);
            mbar_init(&sh.empty[i], 1);
            mbar_init(&sh.s_full[i], 1);
            mbar_init(&sh.p_full[i], kSoftmaxThreads * C::kWGs);
            if constexpr (C::kWide) mbar_init(&sh.p_hi_full[i], kSoftmaxThreads);
            mbar_init(&sh.o_done[i], 1);
        }
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, 1);
        mbar_init(&sh.o_free, kSoftmaxThreads * C::kWGs);
        mbar_init(&sh.mma_done[0], 1);
        mbar_init(&sh.mma_done[1], 1);
        mbar_init(&sh.stall_bar, 1);
        mbar_init(&sh.patch_bar, 1);
        sh.abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();                                     // barriers initialised
    // Inputs (d_pos, cache rows, indices, q) may be written by the kernel
    // before this one on the stream: wait for it before any global read.
    grid_dependency_wait();
    allow_dependent_launch();
    if (warp == C::kPvWarp && lane == 1) load_q<HG>(maps, p, sh, first_key(p), l2_policy_evict_normal());
    const bool softmax = warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + C::kSoftmaxWarps;
    const bool mma = warp == C::kMmaWarp || warp == C::kPvWarp;
    uint32_t tmem = 0;
    if (softmax || mma) {
        // the tensor-memory users wait for the allocation; the producer does not
        if (warp == C::kMmaWarp) {
            tmem_alloc(&sh.tmem_base, C::kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before_sync();
        named_barrier_sync(kBarTmem, 32 * (C::kSoftmaxWarps + 2));
        tc_fence_after_sync();
        tmem = sh.tmem_base;
    }
    if (HG == 16 ? warp < 4 : warp == 0) {
        producer<HG>(maps, p, sh, threadIdx.x);
    } else if (softmax) {
        const int sw = warp - kSoftmaxWarp0;
        if constexpr (C::kWide)
            softmax_wide(p, sh, tmem, sw, lane);
        else
            softmax_warps<HG>(p, sh, tmem, sw >> 2, sw & 3, lane);
    } else if (warp == C::kMmaWarp) {
        if (lane == 0) mma_issue_qk<HG>(p, sh, tmem);
    } else if (warp == C::kPvWarp && lane == 0) {
        mma_issue_pv<HG>(p, sh, tmem);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace

size_t partial_tc_smem_bytes(int head_group) {
    const size_t storage = head_group == 64   ? sizeof(SharedStorage<64>)
                           : head_group == 32 ? sizeof(SharedStorage<32>)
                                              : sizeof(SharedStorage<16>);
    return storage + 1024;                               // + the alignment of the dynamic window
}
int partial_tc_block_threads(int head_group) {
    return head_group == 64 ? Cfg<64>::kThreads : head_group == 32 ? Cfg<32>::kThreads : Cfg<16>::kThreads;
}

cudaError_t partial_tc_prepare(int /*device*/) {
    cudaError_t e = cudaFuncSetAttribute(mla_partial_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(partial_tc_smem_bytes(16)));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mla_partial_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(partial_tc_smem_bytes(32)));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mla_partial_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(partial_tc_smem_bytes(64)));
    return e;
}

cudaError_t launch_partial_tc(const TcMaps& maps, const PartialParams& p, int head_group, dim3 grid, bool pdl,
                              cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(partial_tc_block_threads(head_group), 1, 1);
    cfg.dynamicSmemBytes = partial_tc_smem_bytes(head_group);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (head_group == 64) return cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<64>, maps, p);
    return head_group == 32 ? cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<32>, maps, p)
                            : cudaLaunchKernelEx(&cfg, mla_partial_tc_kernel<16>, maps, p);
}

}  // namespace mla
