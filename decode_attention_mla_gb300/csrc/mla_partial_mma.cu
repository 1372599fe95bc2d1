// mla_partial_mma.cu -- split-KV MLA decode partials, head-group-16 kernel on
// warp-level tensor-core MMA (mma.sync m16n8k16, bf16 in, fp32 accumulate).
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
//   producer warp : (one warp of a warpgroup that hands its registers to the
//                   MMA warps) fills a 4-deep ring of 32-row slots.  Dense slices: one
//                   TMA box {64, 32 rows, 9 chunks} per slot, landing as
//                   [chunk][row][128 B], 128-byte swizzled (rows past the end
//                   of the cache read as zeros).  Sparse lists: all four warps
//                   of the group, eight rows of a slot each, one 1152-byte
//                   bulk copy per row into padded 1168-byte rows, rows taken
//                   from indices[b][e] (a gather, "The Commit That Changed
//                   Direction"); masked entries are zero-filled.  It also
//                   stages the item's 16 query rows (one TMA box) whenever the
//                   (request, head group) changes.
//   8 MMA warps   : two groups of four (one warp of each group on every SM
//                   sub-partition) take alternate 32-row slots of an item, each
//                   group with its own online softmax, so one group's
//                   exchanges, barriers and softmax overlap the other's MMAs.
//                   Scores: in a group, warp pair p takes rows 16p .. +15 of
//                   the slot and each warp half of the 576-wide contraction
//                   (k-steps 4c + 2h + {0, 1} of each 64-column chunk c, its
//                   query fragments held in registers); the halves meet
//                   through shared memory, each warp finishing one 8-row
//                   tile.  Softmax keeps one base-2 reference per head for the
//                   group and moves it only when a score exceeds it by more
//                   than 8 (one OR-barrier per slot decides); each warp turns
//                   its 8 rows into P = 2^(s - ref) as a bf16 hi + lo pair
//                   (about 16 significant bits) and publishes them.  P . V:
//                   warp w of a group owns output features 128w .. 128w+127
//                   for all 16 heads and all 32 rows of the slot.  At the end
//                   of an item group 1 stages its O, reference and row sums in
//                   its last slot and group 0 merges the two states.
// No floating-point atomics: the result is a pure function of the inputs and
// the split count.  Every wait is bounded; a timeout raises MLA_EDEVICE in the
// status word, every warp leaves through the same barrier, and the CTA drains
// its copies before it exits.
#include <cfloat>
#include <cmath>
#include <cstddef>
#include <type_traits>

#include "device_utils.cuh"
#include "mla_decode.h"
#include "mla_internal.h"
#include "slicing.cuh"
#include "tc_utils.cuh"

namespace mla {
namespace {

constexpr int kSlots = 4;                                  // ring depth (32-row slots)
constexpr int kComputeWarps = 8;                           // two groups of four MMA warps
constexpr int kGroups = 2;
constexpr int kGroupWarps = kComputeWarps / kGroups;       // 4: one per SM sub-partition
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kThreads = (kComputeWarps + 4) * 32;         // + a producer warpgroup (one working warp)
constexpr int kProducerWarp = kComputeWarps;
// Sparse rows are copied by all four warps of the producer warpgroup, eight
// rows of a slot each: one warp issuing 32 row copies caps a CTA at ~27 GB/s
// (measured), four warps of 8 at ~56 GB/s.  Each producer warp signals its
// own full barrier per slot, so that it can drain its own copies.
constexpr int kProdWarps = 4;
constexpr int kRowsPerProd = 32 / kProdWarps;
// Register split: the CTA is launched with kLaunchRegs per thread; the
// producer warpgroup drops to RegSplit::kProducer and the two MMA warpgroups
// rise to RegSplit::kMma (the query fragments of a contraction half alone take 72).
constexpr int kLaunchRegs = 168;
// The E4M3 instantiation's producer warpgroup widens bytes in registers and
// takes a larger share: ptxas spills 120 bytes at 56 and 48 at 104.  At T =
// 131072 the E4M3 call then takes 37.9 us, against 43.4 us with (56, 224)
// and 38.9 us with (88, 208).
template <bool kFp8>
struct RegSplit {
    static constexpr int kProducer = kFp8 ? 104 : 56;
    static constexpr int kMma = kFp8 ? 200 : 224;
};
static_assert(128 * RegSplit<false>::kProducer + kComputeWarps * 32 * RegSplit<false>::kMma <= kThreads * kLaunchRegs,
              "register split");
static_assert(128 * RegSplit<true>::kProducer + kComputeWarps * 32 * RegSplit<true>::kMma <= kThreads * kLaunchRegs,
              "register split (E4M3)");
constexpr int kChunks = kDRow / 64;                        // 9 column chunks of 64 bf16
constexpr int kKSteps = kDRow / 16;                        // 36 k-steps of the score contraction
constexpr int kKHalf = kKSteps / 2;                        // 18 per warp
constexpr int kFeatPerWarp = kDLatent / kGroupWarps;       // 128 output features per warp
constexpr int kPVTiles = kFeatPerWarp / 8;                 // 16 n-tiles of P . V per warp
constexpr int kSlotTiles = kStageRows / 8;                 // 4 score tiles of 8 rows per slot
constexpr int kIdxPrefetch = 4;                            // sparse index prefetch depth (slots)
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;                   // log2 units: P stays <= 256
// dense slot: [9 chunks][32 rows][128 B], swizzled; sparse slot: 32 padded rows
constexpr int kDenseChunkBytes = kStageRows * 128;         // 4096
constexpr int kDenseSlotBytes = kChunks * kDenseChunkBytes;  // 36,864
constexpr int kSmemRow = kRowBytes + 16;                   // 8 consecutive rows hit 8 distinct 16-byte groups
constexpr int kSparseSlotBytes = kStageRows * kSmemRow;    // 37,376
constexpr int kQChunkBytes = kHeadGroup * 128;             // 2048
constexpr int kStagePitch = kDLatent + 4;                  // floats per staged row of group 1's O (2064 B)
// named barriers: 0 is __syncthreads, 1..4 the warp pairs (two per group),
// 5 and 6 the groups, 7 all MMA warps
constexpr int kBarPair0 = 1;
constexpr int kBarGroup0 = 5;
constexpr int kBarMma = 7;
constexpr int kBarConvert = 8;                             // E4M3 cache: the converting producer warps
constexpr int kMmaThreads = kComputeWarps * 32;
// E4M3 cache: a slot's bytes, [9 chunks][32 rows][64 bytes] (one TMA box,
// unswizzled), land in the upper part of the slot and are widened to f16 in
// place
constexpr int kFp8ChunkBytes = kStageRows * 64;            // 2048
constexpr int kFp8SlotBytes = kChunks * kFp8ChunkBytes;    // 18,432
constexpr int kFp8StageOffset = kDenseSlotBytes - kFp8SlotBytes;   // 18,432: the slot's upper half
constexpr int kFp8DirectChunks = 4;                        // chunks 0-3 widen straight into [0, 16 KB)
constexpr int kConvertThreads = 128;                       // the producer warpgroup
constexpr int kConvertUnits = kFp8SlotBytes / 8;           // 8 E4M3 bytes -> 16 f16 bytes each
constexpr float kFp8PScale = 128.f;                        // P enters the f16 products as P * 2^7

static_assert(kDenseSlotBytes % 1024 == 0, "swizzled slots stay 1024-byte aligned");
static_assert(kKHalf == 2 * kChunks && kGroupWarps == 2 * (kStageRows / 16),
              "a group's warp pairs cover a slot 16 rows each, a contraction half per warp");
static_assert(kHeadGroup * kStagePitch * 4 <= kDenseSlotBytes, "group 1's O fits in one slot");

struct Fp8Stage {
    uint64_t full[kSlots];                                 // a slot's E4M3 bytes landed (upper part of the slot)
};
struct NoFp8Stage {};

// P . V on the 5th-generation tensor cores (dense bf16 cache): per group, P^T
// of its slot as the K-major B operand ([P_hi | P_lo]: 32 lines of 128 bytes,
// line h = P_hi of head h, line 16 + h = P_lo; the two P buffers of a group
// are K positions 0-31 and 32-63 of the same lines, 128-byte swizzled), and
// the tensor-memory bookkeeping.  O^T of group g, feature block j (features
// 128j .. 128j+127 = tensor-memory lanes 0-127) is columns 128g + 32j ..
// +31: [O_hi | O_lo] of the 16 heads.
constexpr int kPtBytes = 32 * 128;
constexpr uint32_t kTmemCols = 256;
struct __align__(1024) TcPvStage {
    uint8_t pt[kGroups][kPtBytes];                         // P^T per group (1024-byte aligned)
    uint64_t pv_done[kGroups][2];                          // a group's P . V MMAs of P buffer b completed
    uint64_t drain[kGroups];                               // every MMA of the group completed (exit)
    float merge_m[kGroups][kHeadGroup];                    // each group's reference and row sum, per head
    float merge_l[kGroups][kHeadGroup];
    uint32_t tmem_base;
};
struct NoTcPvStage {};

template <bool kDense, bool kFp8 = false, bool kTcPv = false>
struct __align__(1024) SharedStorage {
    static constexpr int kSlotBytes = kDense ? kDenseSlotBytes : kSparseSlotBytes;
    uint8_t q[kChunks * kQChunkBytes];                     // the item's 16 query rows (1024-byte aligned)
    uint8_t kv[kSlots][kSlotBytes];                        // ring of 32-row slots
    std::conditional_t<kTcPv, TcPvStage, NoTcPvStage> tc;  // dense bf16 cache, P . V on tcgen05
    uint4 p[kGroups][2][kSlotTiles][32];                   // P of a group's slot as mma A fragments, double-buffered
    float4 red[kGroups][2][2][32];                         // half-contraction scores exchanged in each pair
    float mx[kGroups][kGroupWarps][kHeadGroup];            // per-warp head maxima (reference moves)
    float lsum[kGroups][kGroupWarps][kHeadGroup];          // per-warp row sums (epilogue)
    float merge_m[kHeadGroup];                             // group 1's reference and row sum, for the merge
    float merge_l[kHeadGroup];
    int valid[kSlots][kStageRows];                         // sparse: row holds an attended entry
    uint64_t full[kSlots][kDense ? 1 : kProdWarps];        // per slot, one per producer warp (dense: one)
    uint64_t empty[kSlots];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t stall_bar;                                    // test hook: a barrier nothing arrives at
    uint64_t patch_bar;                                    // fused append: the slot holding the new row landed
    int abort_flag;
    std::conditional_t<kFp8, Fp8Stage, NoFp8Stage> fp8;    // dense E4M3 cache only
};

// Byte offset of byte b of row r in a 128-byte-swizzled chunk-major tile whose
// 64-column chunks are chunk_bytes apart (b a multiple of 16 for ldmatrix rows).
__device__ __forceinline__ uint32_t sw_off(int r, int b, int chunk_bytes) {
    return static_cast<uint32_t>((b >> 7) * chunk_bytes + r * 128 + ((((b >> 4) & 7) ^ (r & 7)) << 4) + (b & 15));
}
// Lane offsets of the ldmatrix rows inside a slot.  Score operand: row r of
// the slot (0..31), k-step 4c + 2*kh + j of chunk c; the part that varies with
// c is added as a constant (c * chunk stride).  P . V operand: row r, features
// 128gw + 16i + 8*hi .. +7 (chunk 2gw + i/4).
template <bool kDense>
__device__ __forceinline__ uint32_t qk_lane_off(int r, int kh, int j, int lmat) {
    if constexpr (kDense)
        return static_cast<uint32_t>(r * 128 + ((((4 * kh + 2 * j + (lmat & 1)) ^ (r & 7))) << 4));
    else
        return static_cast<uint32_t>(r * kSmemRow + (2 * kh + j) * 32 + (lmat & 1) * 16);
}
template <bool kDense>
__device__ __forceinline__ uint32_t qk_chunk_stride() {
    return kDense ? kDenseChunkBytes : 128;
}
template <bool kDense>
__device__ __forceinline__ uint32_t pv_lane_off(int r, int gw, int i, int hi) {
    if constexpr (kDense)
        return static_cast<uint32_t>((2 * gw + (i >> 2)) * kDenseChunkBytes + r * 128 +
                                     (((2 * (i & 3) + hi) ^ (r & 7)) << 4));
    else
        return static_cast<uint32_t>(r * kSmemRow + gw * 256 + (2 * i + hi) * 16);
}
template <bool kDense>
__host__ __device__ constexpr uint32_t row_pitch() {
    return kDense ? 128 : kSmemRow;
}

template <class S>
__device__ __forceinline__ void raise_device_error(S& sh, int* status) {
    sh.abort_flag = 1;
    if (status) atomicCAS(status, 0, static_cast<int>(MLA_EDEVICE));
}

struct Item {
    int b, hg, s, n_slots;
    long long base;
    uint32_t e0, e1;                       // entries [e0, e1) of the request
    bool skip;                             // flat split: no such piece (nothing to write)
    bool last_piece;                       // flat split: holds the request's last entry
};

// Where an item sits, from the split alone (no device reads): request b, head
// group hg, slice s and, for the flat split, the piece's entries [e0, e1)
// (exists = false for the second piece of a range that holds one request).
// The flat split is sparse only: the dense instantiations compile without it.
struct ItemCoords {
    int b, hg, s;
    uint32_t e0, e1;
    bool exists, last_piece;
};
template <bool kDense>
__device__ __forceinline__ ItemCoords item_coords(const PartialParams& p, int item) {
    ItemCoords c;
    const uint32_t ui = static_cast<uint32_t>(item);
    const uint32_t rest = ui / static_cast<uint32_t>(p.n_groups);
    c.hg = static_cast<int>(ui - rest * static_cast<uint32_t>(p.n_groups));
    c.e0 = c.e1 = 0;
    c.exists = true;
    c.last_piece = false;
    if (kDense || p.flat_ranges == 0) {
        const uint32_t b = rest / static_cast<uint32_t>(p.splits);
        c.s = static_cast<int>(rest - b * static_cast<uint32_t>(p.splits));
        c.b = static_cast<int>(b);
        return c;
    }
    // flat: item = (part, range, head group); the range's entries in the
    // concatenated lists, and the request(s) they belong to
    const uint32_t G = static_cast<uint32_t>(p.flat_ranges);
    const uint32_t part = rest / G;
    const uint32_t r = rest - part * G;
    const uint32_t k = static_cast<uint32_t>(p.topk), P = static_cast<uint32_t>(p.flat_per);
    const uint32_t total = static_cast<uint32_t>(p.batch) * k;
    const uint32_t start = r * P;
    const uint32_t end = start + P < total ? start + P : total;
    uint32_t b = start / k;
    if (part == 1) ++b;
    const uint32_t lo = b * k, hi = lo + k;
    c.b = static_cast<int>(b);
    if (start >= total || b >= static_cast<uint32_t>(p.batch) || end <= lo) {
        c.exists = false;
        c.s = 0;
        c.b = 0;
        return c;
    }
    c.e0 = (start > lo ? start : lo) - lo;
    c.e1 = (end < hi ? end : hi) - lo;
    c.s = static_cast<int>(r - lo / P);
    c.last_piece = end >= hi;
    return c;
}

// The request fields an item's slice depends on (dense: d_pos[b] and the
// segment's first row), read ahead of their use by the caller.
struct RequestRead {
    int d_pos;
    long long base;
};
template <bool kDense>
__device__ __forceinline__ RequestRead read_request(const PartialParams& p, int b) {
    RequestRead r;
    r.d_pos = kDense ? p.d_pos[b] : 0;
    r.base = p.row_offset ? p.row_offset[b] : 0;
    return r;
}
template <bool kDense>
__device__ __forceinline__ int request_of(const PartialParams& p, int item) {
    return item_coords<kDense>(p, item).b;
}

template <bool kDense>
__device__ __forceinline__ Item decode_item(const PartialParams& p, int item, const RequestRead* pre = nullptr) {
    Item it;
    const ItemCoords c = item_coords<kDense>(p, item);
    it.hg = c.hg;
    it.s = c.s;
    it.b = c.b;
    it.skip = !c.exists;
    it.last_piece = c.last_piece;
    if (!kDense && p.flat_ranges > 0) {
        // flat split (sparse only): the piece's entries are known without reads
        it.base = pre ? pre->base : (c.exists && p.row_offset ? p.row_offset[c.b] : 0);
        it.e0 = c.e0;
        it.e1 = c.e1;
        it.n_slots = c.exists ? static_cast<int>((c.e1 - c.e0 + kStageRows - 1) / kStageRows) : 0;
        return it;
    }
    // entry counts are below 2^31 (d_pos and the list length are int32), so
    // the slice arithmetic runs in 32 bits (64-bit division is slow); dense
    // entries are already clamped to the rows that exist in the cache
    uint32_t n;
    if (pre) {
        // the same count as request_entries, from values read earlier
        it.base = pre->base;
        long long m = kDense ? static_cast<long long>(pre->d_pos) + 1 : p.topk;
        if (kDense) {
            const long long cap = p.kv_rows - it.base;
            if (m > cap) m = cap;
            if (m < 0) m = 0;
        }
        n = static_cast<uint32_t>(m);
    } else {
        n = static_cast<uint32_t>(request_entries(!kDense, p.topk, p.d_pos, p.row_offset, p.kv_rows, it.b, &it.base));
    }
    const uint32_t per = slice_entries_u32(n, static_cast<uint32_t>(p.splits), kStageRows);
    uint32_t e0 = static_cast<uint32_t>(it.s) * per;
    uint32_t e1 = e0 + per;
    if (e1 > n) e1 = n;
    if (e0 > e1) e0 = e1;
    it.e0 = e0;
    it.e1 = e1;
    it.n_slots = static_cast<int>((e1 - e0 + kStageRows - 1) / kStageRows);
    return it;
}

// Query tile of the CTA's first item: known without the context length.
template <bool kDense>
__device__ __forceinline__ int first_key(const PartialParams& p) {
    const ItemCoords c = item_coords<kDense>(p, static_cast<int>(blockIdx.x));
    return c.b * p.n_groups + c.hg;
}

template <class S>
__device__ __forceinline__ void load_q(const TcMaps& maps, const PartialParams& p, S& sh, int key, int lane) {
    if (lane == 0) {
        const int b = key / p.n_groups;
        const int hg = key - b * p.n_groups;
        mbar_arrive_expect_tx(&sh.q_full, kChunks * kQChunkBytes);
        tma_load_3d(sh.q, &maps.q, 0, b * p.heads + hg * kHeadGroup, 0, &sh.q_full, l2_policy_evict_normal());
    }
}

// ============================== producer ==================================
// While the preceding kernel still runs: the first item's query tile, its
// request fields and the first row of its partial output into L2 (with their
// address translations).  Hints only: everything is read again after the
// grid dependency.
template <bool kDense>
__device__ void prefetch_first_inputs(const TcMaps& maps, const PartialParams& p) {
    const int item = static_cast<int>(blockIdx.x);
    if (item >= p.n_items) return;
    const ItemCoords c = item_coords<kDense>(p, item);
    const int hg = c.hg, b = c.b, s = c.s;
    tma_prefetch_3d(&maps.q, 0, b * p.heads + hg * kHeadGroup, 0);
    if (kDense) prefetch_l2(p.d_pos + b);
    if (p.row_offset) prefetch_l2(p.row_offset + b);
    if (!kDense) {
        prefetch_l2(p.cache_len + b);
        prefetch_l2(p.indices + static_cast<long long>(b) * p.topk);
    }
    const long long row0 = (static_cast<long long>(b) * p.heads + hg * kHeadGroup) * p.splits + s;
    prefetch_l2(p.o_part + row0 * kDLatent);
    prefetch_l2(p.lse_part + row0);
}

// Dense: while the preceding kernel still runs, bring the first slots of the
// CTA's first item into L2.  The context length read here may be stale (that
// kernel may be advancing it): it only aims the prefetch, and every row the
// kernel uses is loaded again after the grid dependency.
__device__ void prefetch_first_slots(const TcMaps& maps, const PartialParams& p) {
    const int item = static_cast<int>(blockIdx.x);
    if (item >= p.n_items) return;
    const int rest = item / p.n_groups;
    const int b = rest / p.splits;
    const int s = rest - b * p.splits;
    const long long base = p.row_offset ? ld_relaxed_s64(p.row_offset + b) : 0;
    if (base < 0 || base >= p.kv_rows) return;
    long long n = static_cast<long long>(ld_relaxed_s32(p.d_pos + b)) + 1;
    if (n > p.kv_rows - base) n = p.kv_rows - base;
    if (n <= 0) return;
    const long long per = slice_entries(n, p.splits, kStageRows);
    const long long e0 = static_cast<long long>(s) * per;
    long long e1 = e0 + per;
    if (e1 > n) e1 = n;
    for (long long e = e0, k = 0; e < e1 && k < kSlots; e += kStageRows, ++k)
        tma_prefetch_3d(&maps.kv, 0, static_cast<int>(base + e), 0);
}

// wp: producer warp (0 .. kProdWarps-1); dense slices use warp 0 alone, which
// also stages the query tiles.
template <bool kDense, class S>
__device__ void producer(const TcMaps& maps, const PartialParams& p, S& sh, int wp, int lane) {
    const uint64_t policy = l2_policy_evict_first();
    int stage = 0;            // slots issued so far (ring position)
    // the first query tile is requested before the item is decoded (its key
    // needs no context length); the MMA warps follow the same sequence of keys
    // (a new tile whenever a busy item's key differs) and release a tile
    // through q_empty, read or not
    int q_key = first_key<kDense>(p);
    int q_loads = 0;          // query tiles staged so far
    int patch_uses = 0;       // fused append: slots patched so far (phase of patch_bar)
    // the first item's request fields are read before the query tile is
    // requested, so that the two latencies overlap
    RequestRead first{0, 0};
    if (wp == 0) {
        first = read_request<kDense>(p, blockIdx.x < p.n_items ? request_of<kDense>(p, blockIdx.x) : 0);
        load_q(maps, p, sh, q_key, lane);
        q_loads = 1;
    }
    // test hook: a wait that runs out, so every role takes the abort path
    bool ok = !(wp == 0 && p.stall_test && !mbar_wait_bounded(&sh.stall_bar, 0, &sh.abort_flag, kStallTestCycles));
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it =
            decode_item<kDense>(p, item, (wp == 0 && item == static_cast<int>(blockIdx.x)) ? &first : nullptr);
        if (it.n_slots == 0) continue;
        const int key = it.b * p.n_groups + it.hg;
        if (wp == 0 && key != q_key) {
            if (!mbar_wait_bounded(&sh.q_empty, (q_loads - 1) & 1, &sh.abort_flag)) {
                ok = false;
                break;
            }
            load_q(maps, p, sh, key, lane);
            q_key = key;
            ++q_loads;
        }
        if constexpr (kDense) {
            // fused append: entry d_pos[b] of the request is the new row; it lies
            // in this item when the slice holds it (then it is the item's last
            // entry, in its last slot)
            int patch_r = -1;
            if (p.new_rows) {
                const long long dp = p.d_pos[it.b];
                if (dp >= static_cast<long long>(it.e0) && dp < static_cast<long long>(it.e1))
                    patch_r = static_cast<int>(dp - it.e0) - (it.n_slots - 1) * kStageRows;
            }
            // one TMA box per slot from lane 0; rows before the cache (a
            // negative first row) and past its end read as zeros
            bool patch_issued = false;
            if (lane == 0) {
                for (int st = 0; st < it.n_slots; ++st, ++stage) {
                    const int slot = stage % kSlots;
                    if (stage >= kSlots &&
                        !mbar_wait_bounded(&sh.empty[slot], ((stage / kSlots) - 1) & 1, &sh.abort_flag)) {
                        ok = false;
                        break;
                    }
                    long long y = it.base + it.e0 + static_cast<long long>(st) * kStageRows;
                    if (y < -2 * kStageRows) y = -2 * kStageRows;   // a box wholly before row 0 either way
                    // the slot that takes the new row lands on the patch barrier first
                    const bool patched = patch_r >= 0 && st == it.n_slots - 1;
                    uint64_t* bar = patched ? &sh.patch_bar : &sh.full[slot][0];
                    patch_issued = patched;
                    mbar_arrive_expect_tx(bar, kDenseSlotBytes);
                    tma_load_3d(sh.kv[slot], &maps.kv, 0, static_cast<int>(y), 0, bar, policy);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            stage = __shfl_sync(0xffffffffu, stage, 0);
            if (__shfl_sync(0xffffffffu, patch_issued ? 1 : 0, 0)) {
                // once the slot's rows are in, row patch_r is overwritten with the new
                // row (same swizzled layout), then the slot is handed to the MMA warps
                volatile int never = 0;
                bool w = mbar_wait_bounded(&sh.patch_bar, patch_uses & 1, &never);
                w = __all_sync(0xffffffffu, w);
                ++patch_uses;
                const int slot = (stage - 1) % kSlots;
                if (w && ok) {
                    const uint4* src = reinterpret_cast<const uint4*>(p.new_rows + static_cast<long long>(it.b) * kDRow);
                    const uint32_t row = smem_u32(sh.kv[slot]) + patch_r * 128;
                    for (int u = lane; u < kRowBytes / 16; u += 32) {
                        const uint4 v = src[u];
                        st_shared_v4(row + (u >> 3) * kDenseChunkBytes + (((u & 7) ^ (patch_r & 7)) << 4), v.x, v.y,
                                     v.z, v.w);
                    }
                    fence_proxy_async_smem();   // the tensor cores may read the slot next
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.full[slot][0]);
                } else {
                    ok = false;
                }
            }
        } else {
            // rows 8*wp .. 8*wp+7 of each slot, one per lane 0..7; indices
            // of the next few slots are loaded ahead of their use
            const int r_slot = kRowsPerProd * wp + lane;    // row of the slot this lane copies (lane < 8)
            const bool mine = lane < kRowsPerProd;
            const int seg_len = p.cache_len[it.b];
            const int* idx = p.indices + static_cast<long long>(it.b) * p.topk;
            int idx_pf[kIdxPrefetch];
#pragma unroll
            for (int k = 0; k < kIdxPrefetch; ++k) {
                const uint32_t e = it.e0 + static_cast<uint32_t>(k * kStageRows + r_slot);
                idx_pf[k] = (mine && e < it.e1) ? idx[e] : -1;
            }
            for (int st = 0; st < it.n_slots; ++st, ++stage) {
                const int slot = stage % kSlots;
                if (stage >= kSlots &&
                    !mbar_wait_bounded(&sh.empty[slot], ((stage / kSlots) - 1) & 1, &sh.abort_flag)) {
                    ok = false;
                    break;
                }
                const int id = idx_pf[0];
                long long row = 0;
                bool valid = false;
                if (id >= 0 && id < seg_len) {
                    row = it.base + id;
                    valid = (row >= 0 && row < p.kv_rows);
                }
#pragma unroll
                for (int k = 0; k + 1 < kIdxPrefetch; ++k) idx_pf[k] = idx_pf[k + 1];
                const uint32_t en = it.e0 + static_cast<uint32_t>((st + kIdxPrefetch) * kStageRows + r_slot);
                idx_pf[kIdxPrefetch - 1] = (mine && en < it.e1) ? idx[en] : -1;

                uint8_t* dst = sh.kv[slot] + r_slot * kSmemRow;
                if (mine) sh.valid[slot][r_slot] = valid ? 1 : 0;
                if (mine && !valid) {
                    // masked rows still feed P . V (with p = 0): keep them finite
                    uint4* z = reinterpret_cast<uint4*>(dst);
#pragma unroll 8
                    for (int i = 0; i < kRowBytes / 16; ++i) z[i] = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();   // before a later copy lands on these bytes
                }
                const uint32_t n_valid = __popc(__ballot_sync(0xffffffffu, valid));
                __syncwarp();                   // zero rows and flags before the arrival that publishes them
                if (lane == 0)
                    mbar_arrive_expect_tx(&sh.full[slot][wp], n_valid * static_cast<uint32_t>(kRowBytes));
                __syncwarp();                   // the byte count is registered before any copy lands
                if (valid) bulk_copy_g2s(dst, p.kv + row * p.row_stride, kRowBytes, &sh.full[slot][wp], policy);
            }
        }
    }
    if (!ok && lane == 0) raise_device_error(sh, p.status);
    // Never retire the CTA with copies into its shared memory in flight: each
    // producer warp waits for the last phase it armed on its own barriers.
    if (lane == 0) {
        volatile int never = 0;
        for (int slot = 0; slot < kSlots && slot < stage; ++slot) {
            const int last_use = (stage - 1 - slot) / kSlots;
            if (!mbar_wait_bounded(&sh.full[slot][wp], last_use & 1, &never)) raise_device_error(sh, p.status);
        }
        if (q_loads > 0 && !mbar_wait_bounded(&sh.q_full, (q_loads - 1) & 1, &never))
            raise_device_error(sh, p.status);
    }
}

// ---- dense E4M3 cache ------------------------------------------------------
// A slot's E4M3 bytes (one TMA box {64 bytes, 32 rows, 9 chunks}, no
// swizzle, 18,432 bytes) land in the upper half of the slot they become, so
// the ring is as deep as for bf16 rows (four slots in flight), and the four
// producer warps widen them in place to f16 (one cvt per pair, exact: an
// E4M3 value has 4 significant bits and an exponent inside f16's normal
// range; NaN stays NaN), in the 128-byte-swizzled chunk-major layout a bf16
// cache lands in.  The MMA warps take the f16 forms of their products (query
// fragments rounded to f16 once per tile, P as f16 pairs).  In place: the f16
// chunks 0-3 fill [0, 16 KB), below the staged bytes, and are written at
// once; chunks 4-8 overwrite staged bytes, so every thread first reads its
// share of them into registers, and writes only after a barrier.  One thread
// also issues the loads (a slot's load as soon as the MMA warps free it,
// checked without waiting between slots, waited for only when the slot about
// to be widened has not been issued yet) and prefetches six slots ahead into
// L2.  Rows before the cache or past its end read as zero bytes (the TMA
// fill), i.e. 0.0.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two)));
    return h2;
}

// The (item, slot) sequence of this CTA, walked ahead of the conversions by
// the thread that issues the loads and L2 prefetches.
struct SlotCursor {
    int item, st, n_slots;
    long long row0;                               // first cache row of the item's slice
    bool valid;
};
__device__ __forceinline__ void slot_cursor_next_item(const PartialParams& p, SlotCursor& c, int from) {
    for (int i = from; i < p.n_items; i += gridDim.x) {
        const Item it = decode_item<true>(p, i);
        if (it.n_slots > 0) {
            c.item = i;
            c.st = 0;
            c.n_slots = it.n_slots;
            c.row0 = it.base + it.e0;
            c.valid = true;
            return;
        }
    }
    c.valid = false;
}
__device__ __forceinline__ void slot_cursor_step(const PartialParams& p, SlotCursor& c) {
    if (++c.st == c.n_slots) slot_cursor_next_item(p, c, c.item + static_cast<int>(gridDim.x));
}
__device__ __forceinline__ int slot_cursor_row(const SlotCursor& c) {
    long long y = c.row0 + static_cast<long long>(c.st) * kStageRows;
    if (y < -2 * kStageRows) y = -2 * kStageRows;   // a box wholly before row 0 either way
    return static_cast<int>(y);
}

// Unit i of a slot (8 E4M3 bytes -> 16 f16 bytes): chunk c, row r, 8-byte group u.
__device__ __forceinline__ uint32_t fp8_src(uint32_t slot, int i) {
    return slot + kFp8StageOffset + (i >> 8) * kFp8ChunkBytes + ((i >> 3) & (kStageRows - 1)) * 64 + (i & 7) * 8;
}
__device__ __forceinline__ uint32_t fp8_dst(uint32_t slot, int i) {
    const int r = (i >> 3) & (kStageRows - 1);
    return slot + (i >> 8) * kDenseChunkBytes + r * 128 + (((i & 7) ^ (r & 7)) << 4);
}
__device__ __forceinline__ void fp8_store(uint32_t dst, uint32_t w0, uint32_t w1) {
    st_shared_v4(dst, e4m3x2_to_f16x2(w0), e4m3x2_to_f16x2(w0 >> 16), e4m3x2_to_f16x2(w1),
                 e4m3x2_to_f16x2(w1 >> 16));
}

template <class S>
__device__ void producer_fp8(const TcMaps& maps, const PartialParams& p, S& sh, int wp, int lane) {
    constexpr int kDirectUnits = kFp8DirectChunks * 256;             // units of chunks 0-3
    constexpr int kHeldPerThread = (kConvertUnits - kDirectUnits) / kConvertThreads;   // 10
    static_assert(kConvertUnits % 256 == 0 && kStageRows == 32, "unit decomposition: 256 units per chunk");
    static_assert((kConvertUnits - kDirectUnits) % kConvertThreads == 0 && kDirectUnits % kConvertThreads == 0,
                  "whole units per thread");
    static_assert(kFp8DirectChunks * kDenseChunkBytes <= kFp8StageOffset, "chunks 0-3 lie below the staged bytes");
    const uint64_t policy = l2_policy_evict_first();
    const int ct = wp * 32 + lane;                // converting thread (all four producer warps)
    const bool issuer = ct == 0;                  // issues the loads, prefetches ahead, loads the query tiles
    constexpr int kPrefetchAhead = 6;             // slots of L2 prefetch ahead of the loads
    volatile int never = 0;
    int q_key = first_key<true>(p);
    int q_loads = 0;
    int issued = 0;                               // slot loads issued (issuer)
    SlotCursor ic{}, pc{};                        // issue and prefetch cursors (issuer)
    if (wp == 0) {
        load_q(maps, p, sh, q_key, lane);
        q_loads = 1;
    }
    bool ok = !(wp == 0 && p.stall_test && !mbar_wait_bounded(&sh.stall_bar, 0, &sh.abort_flag, kStallTestCycles));
    ok = !named_barrier_or(kBarConvert, kConvertThreads, !ok);
    if (issuer && ok) {
        slot_cursor_next_item(p, ic, blockIdx.x);
        pc = ic;
        for (int k = 0; k < kPrefetchAhead && pc.valid; ++k) {
            tma_prefetch_3d(&maps.kv, 0, slot_cursor_row(pc), 0);
            slot_cursor_step(p, pc);
        }
    }
    int stage = 0;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        const Item it = decode_item<true>(p, item);
        if (it.n_slots == 0) continue;
        bool qw = true;                            // the query tile's buffer was free (warp 0)
        if (wp == 0) {
            const int key = it.b * p.n_groups + it.hg;
            if (key != q_key) {
                qw = mbar_wait_bounded(&sh.q_empty, (q_loads - 1) & 1, &sh.abort_flag);
                if (qw) load_q(maps, p, sh, key, lane);
                q_key = key;
                ++q_loads;
            }
        }
        for (int st = 0; st < it.n_slots; ++st, ++stage) {
            const int slot = stage % kSlots;
            // loads: this slot's for certain (waiting for its previous use to be
            // released), later ones while their slots are already free
            bool w = st > 0 || qw;
            if (issuer) {
                while (w && ic.valid && issued < stage + kSlots) {
                    const int js = issued % kSlots;
                    if (issued >= kSlots) {
                        const uint32_t par = ((issued / kSlots) - 1) & 1;
                        if (issued > stage) {
                            if (!mbar_test(&sh.empty[js], par)) break;
                        } else if (!mbar_wait_bounded(&sh.empty[js], par, &sh.abort_flag)) {
                            w = false;
                            break;
                        }
                    }
                    mbar_arrive_expect_tx(&sh.fp8.full[js], kFp8SlotBytes);
                    tma_load_3d(sh.kv[js] + kFp8StageOffset, &maps.kv, 0, slot_cursor_row(ic), 0, &sh.fp8.full[js],
                                policy);
                    slot_cursor_step(p, ic);
                    ++issued;
                    if (pc.valid) {
                        tma_prefetch_3d(&maps.kv, 0, slot_cursor_row(pc), 0);
                        slot_cursor_step(p, pc);
                    }
                }
            }
            w = w && mbar_wait_bounded(&sh.fp8.full[slot], (stage / kSlots) & 1, &sh.abort_flag);
            if (named_barrier_or(kBarConvert, kConvertThreads, !w)) {   // (the threads decide together)
                ok = false;
                break;
            }
            const uint32_t sb = smem_u32(sh.kv[slot]);
            // chunks 0-3: straight into the lower part, which holds no staged
            // bytes (all loads first: the widening is bound by shared-memory
            // latency, not by its arithmetic)
            {
                constexpr int kDirectPerThread = kDirectUnits / kConvertThreads;   // 8
                uint32_t d[kDirectPerThread][2];
#pragma unroll
                for (int k = 0; k < kDirectPerThread; ++k)
                    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                                 : "=r"(d[k][0]), "=r"(d[k][1])
                                 : "r"(fp8_src(sb, ct + k * kConvertThreads)));
#pragma unroll
                for (int k = 0; k < kDirectPerThread; ++k)
                    fp8_store(fp8_dst(sb, ct + k * kConvertThreads), d[k][0], d[k][1]);
            }
            // chunks 4-8: read this thread's units before anything overwrites them
            uint32_t held[kHeldPerThread][2];
#pragma unroll
            for (int k = 0; k < kHeldPerThread; ++k) {
                const int i = kDirectUnits + ct + k * kConvertThreads;
                asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(held[k][0]), "=r"(held[k][1]) : "r"(fp8_src(sb, i)));
            }
            named_barrier_sync(kBarConvert, kConvertThreads);   // every staged byte has been read
#pragma unroll
            for (int k = 0; k < kHeldPerThread; ++k) {
                const int i = kDirectUnits + ct + k * kConvertThreads;
                fp8_store(fp8_dst(sb, i), held[k][0], held[k][1]);
            }
            fence_proxy_async_smem();                           // the tensor cores may read it
            named_barrier_sync(kBarConvert, kConvertThreads);   // the slot is complete
            if (issuer) mbar_arrive(&sh.full[slot][0]);
        }
    }
    if (!ok && lane == 0) raise_device_error(sh, p.status);
    // never retire with copies in flight: the issuer waits for the last phase
    // armed on each slot, and for the query tile
    if (issuer) {
        for (int s = 0; s < kSlots && s < issued; ++s) {
            const int last_use = (issued - 1 - s) / kSlots;
            if (!mbar_wait_bounded(&sh.fp8.full[s], last_use & 1, &never)) raise_device_error(sh, p.status);
        }
        if (q_loads > 0 && !mbar_wait_bounded(&sh.q_full, (q_loads - 1) & 1, &never))
            raise_device_error(sh, p.status);
    }
}

// ============================== MMA warps =================================
// Two groups of four warps (one warp of each on every SM sub-partition) take
// alternate 32-row slots of an item: group 0 slots 0, 2, 4, ..., group 1
// slots 1, 3, 5, ...  Each group runs its own online softmax (its own
// reference, row sums and O), so one group's exchanges, barriers and softmax
// overlap the other group's MMAs; the two partials meet once per item, in
// shared memory, before the normalised partial is stored.
//
// Bounded wait whose answer is the same on every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort_flag));
}
__device__ __forceinline__ float4 as_float4(const float (&v)[4]) { return make_float4(v[0], v[1], v[2], v[3]); }

// This warp's half of the score contraction for its pair's 16 rows of a slot
// (two 8-row tiles), in two accumulation chains per tile (even / odd k-steps)
// added once; zeros when `run` is false.
template <bool kDense, bool kF16 = false>
__device__ __forceinline__ void qk_scores(float (&acc)[2][4], const uint32_t (&qa)[kKHalf][4], uint32_t sbase,
                                          const uint32_t (&qk_off)[2], bool run) {
#pragma unroll
    for (int j = 0; j < 2; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    if (!run) return;
    float acc2[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) acc2[j][0] = acc2[j][1] = acc2[j][2] = acc2[j][3] = 0.f;
    const uint32_t a0 = sbase + qk_off[0];
    const uint32_t a1 = sbase + qk_off[1];
#pragma unroll
    for (int kk = 0; kk < kKHalf; ++kk) {
        uint32_t bf[4];
        ldmatrix_x4(bf, ((kk & 1) ? a1 : a0) + (kk >> 1) * qk_chunk_stride<kDense>());
        if (kk & 1) {
            mma_16816<kF16>(acc2[0], qa[kk], bf[0], bf[1]);
            mma_16816<kF16>(acc2[1], qa[kk], bf[2], bf[3]);
        } else {
            mma_16816<kF16>(acc[0], qa[kk], bf[0], bf[1]);
            mma_16816<kF16>(acc[1], qa[kk], bf[2], bf[3]);
        }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[j][c] += acc2[j][c];
}

// One k-step (16 rows of a slot) of O += P . V for this warp's 128 features:
// P as the A fragments of the group's published hi / lo pairs, V by
// transposing ldmatrix, in two halves of eight n-tiles (low-part MMAs first,
// then the high parts: each accumulator's two MMAs eight instructions apart).
template <bool kDense, bool kF16 = false>
__device__ __forceinline__ void pv_kstep(float (&o)[kPVTiles][4], const uint4* pt, int kp, uint32_t vbase,
                                         const uint32_t (&pv_off)[kPVTiles / 2], int v_hi, int tq, int lane) {
    const uint4 t0 = pt[(2 * kp) * 32 + lane];
    const uint4 t1 = pt[(2 * kp + 1) * 32 + lane];
    const uint32_t a_hi[4] = {t0.x, t0.y, t1.x, t1.y};
    const uint32_t a_lo[4] = {t0.z, t0.w, t1.z, t1.w};
    // dense rows past the slice may hold anything (even NaN): zero their V so
    // that p = 0 really contributes nothing
    uint32_t m_lo = 0xffffffffu, m_hi = 0xffffffffu;
    if (kDense && v_hi < 16 * (kp + 1)) {
        const int k0 = 16 * kp + 2 * tq;
        m_lo = (k0 < v_hi ? 0x0000ffffu : 0u) | (k0 + 1 < v_hi ? 0xffff0000u : 0u);
        m_hi = (k0 + 8 < v_hi ? 0x0000ffffu : 0u) | (k0 + 9 < v_hi ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        uint32_t v[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ldmatrix_x4_trans(v[i], vbase + pv_off[4 * hh + i]);
            v[i][0] &= m_lo;
            v[i][1] &= m_hi;
            v[i][2] &= m_lo;
            v[i][3] &= m_hi;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            mma_16816<kF16>(o[8 * hh + 2 * i], a_lo, v[i][0], v[i][1]);
            mma_16816<kF16>(o[8 * hh + 2 * i + 1], a_lo, v[i][2], v[i][3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            mma_16816<kF16>(o[8 * hh + 2 * i], a_hi, v[i][0], v[i][1]);
            mma_16816<kF16>(o[8 * hh + 2 * i + 1], a_hi, v[i][2], v[i][3]);
        }
    }
}

template <bool kDense, bool kFp8 = false>
__device__ void consumer(const PartialParams& p, SharedStorage<kDense, kFp8>& sh, int w, int lane) {
    constexpr uint32_t kSlotBytes = SharedStorage<kDense, kFp8>::kSlotBytes;
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int grp = w / kGroupWarps;        // group: the item's slots grp, grp + 2, ...
    const int gw = w % kGroupWarps;         // warp within the group
    const int pr = gw >> 1;                 // warp pair: rows 16*pr .. +15 of a slot
    const int kh = gw & 1;                  // contraction half, and the pair's 8-row tile this warp finishes
    const int my_tile = 2 * pr + kh;        // score tile of 8 rows (slot rows 8*my_tile ..)
    const int r_own = 8 * my_tile + 2 * tq; // slot rows of this lane's scores: r_own, r_own + 1
    const int f_base = gw * kFeatPerWarp;   // own output features
    const int lrow = lane & 7;
    const int lmat = lane >> 3;
    const int bar_pair = kBarPair0 + 2 * grp + pr;
    const int bar_group = kBarGroup0 + grp;
    const uint32_t q_base = smem_u32(sh.q);
    const uint32_t kv_base = smem_u32(sh.kv[0]);
    // ldmatrix lane offsets: score rows 16*pr + lrow + 8*(lmat/2) of the slot;
    // P . V rows lrow + 8*(lmat%2) (+16 for the second k-step)
    const int qk_row = 16 * pr + lrow + ((lmat >> 1) << 3);
    const uint32_t qk_off[2] = {qk_lane_off<kDense>(qk_row, kh, 0, lmat), qk_lane_off<kDense>(qk_row, kh, 1, lmat)};
    const int pv_row = lrow + ((lmat & 1) << 3);
    uint32_t pv_off[kPVTiles / 2];
#pragma unroll
    for (int i = 0; i < kPVTiles / 2; ++i) pv_off[i] = pv_lane_off<kDense>(pv_row, gw, i, lmat >> 1);

    uint32_t qa[kKHalf][4];                 // query fragments of this warp's contraction half
    int stage = 0;                          // slots of earlier items (ring position of this item's slot 0)
    int pbuf = 0;                           // this group's P buffer for its next slot
    int q_phase = 0;                        // query tiles consumed (q_full phases)
    int q_key = first_key<kDense>(p);               // key of the tile the producer loaded last
    bool q_in_regs = false;                 // that tile is in registers (and released)
    bool failed = false;                    // a wait of this warp ran out
    bool stop = false;                      // every MMA warp saw a failure at the same barrier: leave

    for (int item = blockIdx.x; item < p.n_items && !stop; item += gridDim.x) {
        const Item it = decode_item<kDense>(p, item);
        const long long row_b = (static_cast<long long>(it.b) * p.heads + it.hg * kHeadGroup) * p.splits;
        if (!kDense && it.last_piece) {
            // flat split: the request has no pieces past this one; its remaining
            // slices are written empty so that the merge can read every slice
            for (int s2 = it.s + 1; s2 < p.splits; ++s2)
                write_empty_partial(p.o_part, p.lse_part, row_b + s2, p.splits, w * 32 + lane, kMmaThreads);
        }
        if (it.n_slots == 0) {
            if (kDense || !it.skip) write_empty_partial(p.o_part, p.lse_part, row_b + it.s, p.splits, w * 32 + lane, kMmaThreads);
            continue;
        }
        const int key = it.b * p.n_groups + it.hg;
        if (key != q_key) {
            // the producer loads another tile over this one: release it, read
            // or not (it must have landed first)
            if (!q_in_regs && !failed) {
                if (warp_wait(&sh.q_full, q_phase & 1, &sh.abort_flag)) {
                    if (lane == 0) mbar_arrive(&sh.q_empty);
                } else {
                    failed = true;
                }
            }
            ++q_phase;
            q_key = key;
            q_in_regs = false;
        }
        if (!q_in_regs && !failed) {
            if (warp_wait(&sh.q_full, q_phase & 1, &sh.abort_flag)) {
#pragma unroll
                for (int kk = 0; kk < kKHalf; ++kk)
                    ldmatrix_x4(qa[kk], q_base + sw_off(lrow + ((lmat & 1) << 3),
                                                         (4 * (kk >> 1) + 2 * kh + (kk & 1)) * 32 + ((lmat >> 1) << 4),
                                                         kQChunkBytes));
                if constexpr (kFp8) {
                    // the E4M3 path multiplies in f16: the query fragments once per tile
#pragma unroll
                    for (int kk = 0; kk < kKHalf; ++kk)
#pragma unroll
                        for (int r = 0; r < 4; ++r) qa[kk][r] = bf16x2_to_f16x2(qa[kk][r]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.q_empty);
                q_in_regs = true;
            } else {
                failed = true;
            }
        }

        float o[kPVTiles][4];
#pragma unroll
        for (int i = 0; i < kPVTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_ref[2] = {-INFINITY, -INFINITY};   // heads g, g+8: base-2 reference shared by the group
        float l_own[2] = {0.f, 0.f};               // sums of 2^(s - ref) over this lane's rows
        const int my_slots = it.n_slots > grp ? (it.n_slots - grp + 1) / 2 : 0;
        // the group holding the item's last slot finishes last and merges; the
        // other stages its state while that slot is still being worked on
        const int last_grp = (it.n_slots - 1) & 1;
        const int stage_grp = 1 - last_grp;
        bool gstop = false;                        // the group saw a failure at one of its barriers
        for (int k = 0; k < my_slots && !gstop; ++k) {
            const int j = grp + 2 * k;                      // slot of the item
            const int st = stage + j;                       // its ring position
            const int slot = st % kSlots;
            // dense: one TMA box per slot; sparse: each producer warp's rows
#pragma unroll
            for (int q = 0; q < (kDense ? 1 : kProdWarps); ++q)
                if (!failed && !warp_wait(&sh.full[slot][q], (st / kSlots) & 1, &sh.abort_flag)) failed = true;
            // slot rows [v_lo, v_hi) are attended (dense); sparse rows carry flags
            const uint32_t e_slot = it.e0 + static_cast<uint32_t>(j * kStageRows);
            const int v_hi = static_cast<int>(min(it.e1 - e_slot, static_cast<uint32_t>(kStageRows)));
            const long long first_row = it.base + e_slot;
            const int v_lo =
                first_row >= 0 ? 0 : first_row <= -kStageRows ? kStageRows : static_cast<int>(-first_row);
            const uint32_t sbase = kv_base + static_cast<uint32_t>(slot) * kSlotBytes;

            // ---- scores of this warp's 8-row tile: two contraction halves ------
            float acc[2][4];
            qk_scores<kDense, kFp8>(acc, qa, sbase, qk_off, !failed);
            sh.red[grp][pr][1 - kh][lane] = kh ? as_float4(acc[0]) : as_float4(acc[1]);
            named_barrier_sync(bar_pair, 64);
            const float4 other = sh.red[grp][pr][kh][lane];
            const float4 mine = kh ? as_float4(acc[1]) : as_float4(acc[0]);
            bool v0, v1;
            if constexpr (kDense) {
                v0 = r_own >= v_lo && r_own < v_hi;
                v1 = r_own + 1 >= v_lo && r_own + 1 < v_hi;
            } else {
                v0 = sh.valid[slot][r_own] != 0;
                v1 = sh.valid[slot][r_own + 1] != 0;
            }
            float sc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (!failed) {
                sc[0] = v0 ? (mine.x + other.x) * p.scale_log2 : -INFINITY;
                sc[1] = v1 ? (mine.y + other.y) * p.scale_log2 : -INFINITY;
                sc[2] = v0 ? (mine.z + other.z) * p.scale_log2 : -INFINITY;
                sc[3] = v1 ? (mine.w + other.w) * p.scale_log2 : -INFINITY;
            }
            float mx0 = fmaxf(sc[0], sc[1]);   // head g over this lane's two rows
            float mx1 = fmaxf(sc[2], sc[3]);   // head g + 8

            // ---- P against the group's reference; move it only when needed ----
            float pv[4];
            bool need = true;                  // the group's first slot of an item sets the reference
            if (k > 0) {
                const float ref0 = m_ref[0] == -INFINITY ? 0.f : m_ref[0];
                const float ref1 = m_ref[1] == -INFINITY ? 0.f : m_ref[1];
                pv[0] = ex2_approx(sc[0] - ref0);
                pv[1] = ex2_approx(sc[1] - ref0);
                pv[2] = ex2_approx(sc[2] - ref1);
                pv[3] = ex2_approx(sc[3] - ref1);
                uint4 pk;
                if constexpr (kFp8) {
                    // f16 pairs of P * 2^7 (small probabilities stay clear of f16
                    // subnormals; the epilogue takes the 2^-7 back)
                    split_f16x2(pv[0] * kFp8PScale, pv[1] * kFp8PScale, pk.x, pk.z);
                    split_f16x2(pv[2] * kFp8PScale, pv[3] * kFp8PScale, pk.y, pk.w);
                } else {
                    split_bf16x2(pv[0], pv[1], pk.x, pk.z);
                    split_bf16x2(pv[2], pv[3], pk.y, pk.w);
                }
                sh.p[grp][pbuf][my_tile][lane] = pk;
                const bool over = mx0 > m_ref[0] + kRescaleThreshold || mx1 > m_ref[1] + kRescaleThreshold;
                need = named_barrier_or(bar_group, kGroupThreads, over || failed);
            }
            if (need) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                if (tq == 0) {
                    sh.mx[grp][gw][g] = mx0;
                    sh.mx[grp][gw][g + 8] = mx1;
                }
                if (named_barrier_or(bar_group, kGroupThreads, failed)) {
                    gstop = true;
                    break;
                }
                float n0 = m_ref[0], n1 = m_ref[1];
#pragma unroll
                for (int v = 0; v < kGroupWarps; ++v) {
                    n0 = fmaxf(n0, sh.mx[grp][v][g]);
                    n1 = fmaxf(n1, sh.mx[grp][v][g + 8]);
                }
                if (k > 0) {
                    // what was accumulated against the old reference, scaled to the new one
                    const float a0 = m_ref[0] == -INFINITY ? 0.f : ex2_approx(m_ref[0] - n0);
                    const float a1 = m_ref[1] == -INFINITY ? 0.f : ex2_approx(m_ref[1] - n1);
#pragma unroll
                    for (int i = 0; i < kPVTiles; ++i) {
                        o[i][0] *= a0;
                        o[i][1] *= a0;
                        o[i][2] *= a1;
                        o[i][3] *= a1;
                    }
                    l_own[0] *= a0;
                    l_own[1] *= a1;
                }
                m_ref[0] = n0;
                m_ref[1] = n1;
                const float ref0 = n0 == -INFINITY ? 0.f : n0;   // nothing attended yet: keep exponents finite
                const float ref1 = n1 == -INFINITY ? 0.f : n1;
                pv[0] = ex2_approx(sc[0] - ref0);
                pv[1] = ex2_approx(sc[1] - ref0);
                pv[2] = ex2_approx(sc[2] - ref1);
                pv[3] = ex2_approx(sc[3] - ref1);
                uint4 pk;
                if constexpr (kFp8) {
                    // f16 pairs of P * 2^7 (small probabilities stay clear of f16
                    // subnormals; the epilogue takes the 2^-7 back)
                    split_f16x2(pv[0] * kFp8PScale, pv[1] * kFp8PScale, pk.x, pk.z);
                    split_f16x2(pv[2] * kFp8PScale, pv[3] * kFp8PScale, pk.y, pk.w);
                } else {
                    split_bf16x2(pv[0], pv[1], pk.x, pk.z);
                    split_bf16x2(pv[2], pv[3], pk.y, pk.w);
                }
                sh.p[grp][pbuf][my_tile][lane] = pk;
                named_barrier_sync(bar_group, kGroupThreads);
            }
            l_own[0] += pv[0] + pv[1];
            l_own[1] += pv[2] + pv[3];

            // ---- O[:, own 128 features] += P . V over the slot's 32 rows --------
            const uint4* pt = &sh.p[grp][pbuf][0][0];
            pv_kstep<kDense, kFp8>(o, pt, 0, sbase, pv_off, v_hi, tq, lane);
            pv_kstep<kDense, kFp8>(o, pt, 1, sbase + 16 * row_pitch<kDense>(), pv_off, v_hi, tq, lane);
            __syncwarp();
            // the group without the item's last slot keeps its own last slot:
            // its O is staged there for the other group to merge
            const bool keep = it.n_slots > 1 && grp == stage_grp && k + 1 == my_slots;
            if (lane == 0 && !keep) mbar_arrive(&sh.empty[slot]);
            pbuf ^= 1;
        }

        // ---- epilogue --------------------------------------------------------
        float l0 = l_own[0], l1 = l_own[1];
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        if (tq == 0) {
            sh.lsum[grp][gw][g] = l0;
            sh.lsum[grp][gw][g + 8] = l1;
        }
        // the staging group's O (against its own reference), reference and row
        // sums go to its kept slot as soon as its own slots are done
        const int stg_slot = it.n_slots > 1 ? (stage + it.n_slots - 2) % kSlots : 0;
        float* stage_o = reinterpret_cast<float*>(sh.kv[stg_slot]);   // [16][kStagePitch]
        if (it.n_slots > 1 && grp == stage_grp) {
            named_barrier_sync(bar_group, kGroupThreads);   // the group's row sums are written
            float S0 = 0.f, S1 = 0.f;
#pragma unroll
            for (int v = 0; v < kGroupWarps; ++v) {
                S0 += sh.lsum[grp][v][g];
                S1 += sh.lsum[grp][v][g + 8];
            }
#pragma unroll
            for (int nt = 0; nt < kPVTiles; ++nt) {
                const int f = f_base + 8 * nt + 2 * tq;
                *reinterpret_cast<float2*>(stage_o + g * kStagePitch + f) = make_float2(o[nt][0], o[nt][1]);
                *reinterpret_cast<float2*>(stage_o + (g + 8) * kStagePitch + f) = make_float2(o[nt][2], o[nt][3]);
            }
            fence_proxy_async_smem();   // these bytes are a slot the producer refills later
            if (gw == 0 && tq == 0) {
                sh.merge_m[g] = m_ref[0];
                sh.merge_m[g + 8] = m_ref[1];
                sh.merge_l[g] = S0;
                sh.merge_l[g + 8] = S1;
            }
        }
        // every MMA warp learns whether to go on (and the merging group waits
        // for the staged state)
        if (named_barrier_or(kBarMma, kMmaThreads, failed || gstop)) {
            stop = true;
            break;
        }
        const long long row_h0 = (static_cast<long long>(it.b) * p.heads + it.hg * kHeadGroup) * p.splits + it.s;
        float* op0 = p.o_part + (row_h0 + static_cast<long long>(g) * p.splits) * kDLatent + f_base + 2 * tq;
        float* op1 = p.o_part + (row_h0 + static_cast<long long>(g + 8) * p.splits) * kDLatent + f_base + 2 * tq;
        // (v_scale: the E4M3 cache's scale, 1 for bf16; oscale adds the 2^-7 of P)
        const float oscale = kFp8 ? p.v_scale * (1.f / kFp8PScale) : p.v_scale;
        if (it.n_slots == 1) {
            // one slot: group 0 alone attended rows
            if (grp == 0) {
                float L0 = 0.f, L1 = 0.f;
#pragma unroll
                for (int v = 0; v < kGroupWarps; ++v) {
                    L0 += sh.lsum[0][v][g];
                    L1 += sh.lsum[0][v][g + 8];
                }
                const float inv0 = L0 > 0.f ? rcp_approx(L0) * oscale : 0.f;
                const float inv1 = L1 > 0.f ? rcp_approx(L1) * oscale : 0.f;
#pragma unroll
                for (int nt = 0; nt < kPVTiles; ++nt) {
                    *reinterpret_cast<float2*>(op0 + 8 * nt) = make_float2(o[nt][0] * inv0, o[nt][1] * inv0);
                    *reinterpret_cast<float2*>(op1 + 8 * nt) = make_float2(o[nt][2] * inv1, o[nt][3] * inv1);
                }
                if (gw == 0 && tq == 0) {
                    p.lse_part[row_h0 + static_cast<long long>(g) * p.splits] =
                        L0 > 0.f ? (m_ref[0] + lg2_approx(L0)) * kLn2 : -INFINITY;
                    p.lse_part[row_h0 + static_cast<long long>(g + 8) * p.splits] =
                        L1 > 0.f ? (m_ref[1] + lg2_approx(L1)) * kLn2 : -INFINITY;
                }
            }
        } else if (grp == last_grp) {
            // merge the two online-softmax states, group 0's terms first (the
            // same arithmetic whichever group merges), and store the partial
            float L0 = 0.f, L1 = 0.f;
#pragma unroll
            for (int v = 0; v < kGroupWarps; ++v) {
                L0 += sh.lsum[grp][v][g];
                L1 += sh.lsum[grp][v][g + 8];
            }
            const bool g0 = grp == 0;
            const float ms_a = sh.merge_m[g], ms_b = sh.merge_m[g + 8];
            const float Ls_a = sh.merge_l[g], Ls_b = sh.merge_l[g + 8];
            // (reference, row sum) of group 0 and group 1, per head g and g + 8
            const float m0a = g0 ? m_ref[0] : ms_a, m1a = g0 ? ms_a : m_ref[0];
            const float m0b = g0 ? m_ref[1] : ms_b, m1b = g0 ? ms_b : m_ref[1];
            const float L0a = g0 ? L0 : Ls_a, L1a = g0 ? Ls_a : L0;
            const float L0b = g0 ? L1 : Ls_b, L1b = g0 ? Ls_b : L1;
            const float ma = fmaxf(m0a, m1a);
            const float mb = fmaxf(m0b, m1b);
            const float s0a = m0a == -INFINITY ? 0.f : ex2_approx(m0a - ma);
            const float s1a = m1a == -INFINITY ? 0.f : ex2_approx(m1a - ma);
            const float s0b = m0b == -INFINITY ? 0.f : ex2_approx(m0b - mb);
            const float s1b = m1b == -INFINITY ? 0.f : ex2_approx(m1b - mb);
            const float La = L0a * s0a + L1a * s1a;
            const float Lb = L0b * s0b + L1b * s1b;
            const float inva = La > 0.f ? rcp_approx(La) * oscale : 0.f;
            const float invb = Lb > 0.f ? rcp_approx(Lb) * oscale : 0.f;
            const float c0a = s0a * inva, c1a = s1a * inva, c0b = s0b * invb, c1b = s1b * invb;
#pragma unroll
            for (int nt = 0; nt < kPVTiles; ++nt) {
                const int f = f_base + 8 * nt + 2 * tq;
                const float2 ua = *reinterpret_cast<const float2*>(stage_o + g * kStagePitch + f);
                const float2 ub = *reinterpret_cast<const float2*>(stage_o + (g + 8) * kStagePitch + f);
                const float2 x0a = g0 ? make_float2(o[nt][0], o[nt][1]) : ua;   // group 0's O, head g
                const float2 x1a = g0 ? ua : make_float2(o[nt][0], o[nt][1]);   // group 1's O, head g
                const float2 x0b = g0 ? make_float2(o[nt][2], o[nt][3]) : ub;
                const float2 x1b = g0 ? ub : make_float2(o[nt][2], o[nt][3]);
                *reinterpret_cast<float2*>(op0 + 8 * nt) =
                    make_float2(x0a.x * c0a + x1a.x * c1a, x0a.y * c0a + x1a.y * c1a);
                *reinterpret_cast<float2*>(op1 + 8 * nt) =
                    make_float2(x0b.x * c0b + x1b.x * c1b, x0b.y * c0b + x1b.y * c1b);
            }
            if (gw == 0 && tq == 0) {
                p.lse_part[row_h0 + static_cast<long long>(g) * p.splits] =
                    La > 0.f ? (ma + lg2_approx(La)) * kLn2 : -INFINITY;
                p.lse_part[row_h0 + static_cast<long long>(g + 8) * p.splits] =
                    Lb > 0.f ? (mb + lg2_approx(Lb)) * kLn2 : -INFINITY;
            }
        }
        if (it.n_slots > 1) {
            named_barrier_sync(kBarMma, kMmaThreads);   // the staged state has been read
            if (grp == stage_grp && lane == 0) mbar_arrive(&sh.empty[stg_slot]);
        }
        stage += it.n_slots;
    }
    if ((stop || failed) && lane == 0) raise_device_error(sh, p.status);
}

// ---- dense bf16 cache: scores on the warps, P . V on tcgen05 ---------------
// The MMA warps compute the scores and the softmax exactly as above, write P
// of their slot as the bf16 pair [P_hi | P_lo]^T into the group's P^T buffer,
// and one thread of the group issues the slot's P . V on the tensor cores:
//   O^T[512 x 32] += V_slot^T[512 x 32 rows] . [P_hi | P_lo]^T
// as 4 feature blocks (M = 128) x 2 k-steps of 16 rows (N = 32), V read in
// place from the slot (MN-major: 64-feature atoms one 4096-byte chunk apart),
// O in tensor memory.  The MMAs' completion releases the slot to the
// producer and the P buffer to the group, so the warps never wait for P . V
// within an item.  At the end of an item every MMA warp merges both groups'
// O straight from tensor memory (its own lane quarter, two feature blocks).
// P of this lane's four scores as the pair the tensor cores take: bf16 hi/lo,
// or (E4M3 cache) f16 hi/lo of P * 2^7.
template <bool kFp8>
__device__ __forceinline__ void split_pair(const float (&pv)[4], uint32_t& hi0, uint32_t& lo0, uint32_t& hi1,
                                           uint32_t& lo1) {
    if constexpr (kFp8) {
        split_f16x2(pv[0] * kFp8PScale, pv[1] * kFp8PScale, hi0, lo0);
        split_f16x2(pv[2] * kFp8PScale, pv[3] * kFp8PScale, hi1, lo1);
    } else {
        split_bf16x2(pv[0], pv[1], hi0, lo0);
        split_bf16x2(pv[2], pv[3], hi1, lo1);
    }
}
__device__ __forceinline__ uint32_t pt_off(int n, int k) {
    return static_cast<uint32_t>((n >> 3) * 1024 + (n & 7) * 128 + ((((k >> 3) ^ (n & 7))) << 4) + (k & 7) * 2);
}
__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// E4M3 cache (kFp8): the widened slot holds f16, the scores run in f16 and P
// enters the tensor cores as an f16 pair of P * 2^7 (the 2^-7 returns in the
// merge weights), as on the warp path.
template <bool kFp8, class S>
__device__ void consumer_tcpv(const PartialParams& p, S& sh, int w, int lane) {
    constexpr uint32_t kSlotBytes = kDenseSlotBytes;
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int grp = w / kGroupWarps;
    const int gw = w % kGroupWarps;          // also this warp's tensor-memory lane quarter (w % 4)
    const int pr = gw >> 1;
    const int kh = gw & 1;
    const int my_tile = 2 * pr + kh;
    const int r_own = 8 * my_tile + 2 * tq;
    const int lrow = lane & 7;
    const int lmat = lane >> 3;
    const int bar_pair = kBarPair0 + 2 * grp + pr;
    const int bar_group = kBarGroup0 + grp;
    const uint32_t q_base = smem_u32(sh.q);
    const uint32_t kv_base = smem_u32(sh.kv[0]);
    const int qk_row = 16 * pr + lrow + ((lmat >> 1) << 3);
    const uint32_t qk_off[2] = {qk_lane_off<true>(qk_row, kh, 0, lmat), qk_lane_off<true>(qk_row, kh, 1, lmat)};
    const bool issuer = gw == 0 && lane == 0;   // issues the group's P . V

    // tensor memory: kTmemCols columns for the CTA (one CTA per SM)
    if (w == 0) {
        tmem_alloc(&sh.tc.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    named_barrier_sync(kBarMma, kMmaThreads);
    tc_fence_after_sync();
    const uint32_t tmem = sh.tc.tmem_base;
    const uint32_t tmem_lane = static_cast<uint32_t>(32 * gw) << 16;
    const uint32_t tmem_grp = tmem + 128u * static_cast<uint32_t>(grp);

    const uint32_t pt_base = smem_u32(sh.tc.pt[grp]);
    // lines g, 8 + g, 16 + g, 24 + g (P_hi of heads g and g + 8, then P_lo) share
    // a swizzle and lie 1024 bytes apart; K position 32 * buffer + r_own
    const uint32_t pt_lane0 = pt_base + pt_off(g, r_own);
    const uint32_t pt_lane1 = pt_base + pt_off(g, 32 + r_own);
    const uint32_t idesc = kFp8 ? make_idesc_f16(128, 32, 1, 0) : make_idesc_bf16(128, 32, 1, 0);
    const uint64_t v_desc0 = make_sdesc(kv_base, kDenseChunkBytes, 1024, kLayoutSw128);
    const uint64_t p_desc0 = make_sdesc(pt_base, 16, 1024, kLayoutSw128);

    uint32_t qa[kKHalf][4];
    int stage = 0;
    int q_phase = 0;
    int q_key = first_key<true>(p);
    bool q_in_regs = false;
    bool failed = false;
    bool stop = false;
    int issued = 0;                         // P . V batches this warp's group issued so far
    int issued_other = 0;                   // ... and the other group

    for (int item = blockIdx.x; item < p.n_items && !stop; item += gridDim.x) {
        const Item it = decode_item<true>(p, item);
        const long long row_b = (static_cast<long long>(it.b) * p.heads + it.hg * kHeadGroup) * p.splits;
        if (it.n_slots == 0) {
            write_empty_partial(p.o_part, p.lse_part, row_b + it.s, p.splits, w * 32 + lane, kMmaThreads);
            continue;
        }
        const int key = it.b * p.n_groups + it.hg;
        if (key != q_key) {
            if (!q_in_regs && !failed) {
                if (warp_wait(&sh.q_full, q_phase & 1, &sh.abort_flag)) {
                    if (lane == 0) mbar_arrive(&sh.q_empty);
                } else {
                    failed = true;
                }
            }
            ++q_phase;
            q_key = key;
            q_in_regs = false;
        }
        if (!q_in_regs && !failed) {
            if (warp_wait(&sh.q_full, q_phase & 1, &sh.abort_flag)) {
#pragma unroll
                for (int kk = 0; kk < kKHalf; ++kk)
                    ldmatrix_x4(qa[kk], q_base + sw_off(lrow + ((lmat & 1) << 3),
                                                         (4 * (kk >> 1) + 2 * kh + (kk & 1)) * 32 + ((lmat >> 1) << 4),
                                                         kQChunkBytes));
                if constexpr (kFp8) {
                    // the E4M3 path multiplies in f16: the query fragments once per tile
#pragma unroll
                    for (int kk = 0; kk < kKHalf; ++kk)
#pragma unroll
                        for (int r = 0; r < 4; ++r) qa[kk][r] = bf16x2_to_f16x2(qa[kk][r]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.q_empty);
                q_in_regs = true;
            } else {
                failed = true;
            }
        }

        float m_ref[2] = {-INFINITY, -INFINITY};
        float l_own[2] = {0.f, 0.f};
        const int my_slots = it.n_slots > grp ? (it.n_slots - grp + 1) / 2 : 0;
        bool gstop = false;
        for (int k = 0; k < my_slots && !gstop; ++k) {
            const int j = grp + 2 * k;
            const int st = stage + j;
            const int slot = st % kSlots;
            if (!failed && !warp_wait(&sh.full[slot][0], (st / kSlots) & 1, &sh.abort_flag)) failed = true;
            const uint32_t e_slot = it.e0 + static_cast<uint32_t>(j * kStageRows);
            const int v_hi = static_cast<int>(min(it.e1 - e_slot, static_cast<uint32_t>(kStageRows)));
            const long long first_row = it.base + e_slot;
            const int v_lo =
                first_row >= 0 ? 0 : first_row <= -kStageRows ? kStageRows : static_cast<int>(-first_row);
            const uint32_t sbase = kv_base + static_cast<uint32_t>(slot) * kSlotBytes;
            const int pb = issued & 1;
            const uint32_t pt_w = pb ? pt_lane1 : pt_lane0;
            const int ksteps = (v_hi + 15) >> 4;

            // ---- scores of this warp's 8-row tile: two contraction halves ------
            float acc[2][4];
            qk_scores<true, kFp8>(acc, qa, sbase, qk_off, !failed);
            sh.red[grp][pr][1 - kh][lane] = kh ? as_float4(acc[0]) : as_float4(acc[1]);
            named_barrier_sync(bar_pair, 64);
            const float4 other = sh.red[grp][pr][kh][lane];
            const float4 mine = kh ? as_float4(acc[1]) : as_float4(acc[0]);
            const bool v0 = r_own >= v_lo && r_own < v_hi;
            const bool v1 = r_own + 1 >= v_lo && r_own + 1 < v_hi;
            float sc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (!failed) {
                sc[0] = v0 ? (mine.x + other.x) * p.scale_log2 : -INFINITY;
                sc[1] = v1 ? (mine.y + other.y) * p.scale_log2 : -INFINITY;
                sc[2] = v0 ? (mine.z + other.z) * p.scale_log2 : -INFINITY;
                sc[3] = v1 ? (mine.w + other.w) * p.scale_log2 : -INFINITY;
            }
            float mx0 = fmaxf(sc[0], sc[1]);
            float mx1 = fmaxf(sc[2], sc[3]);

            // the P buffer's batch before last must have been read by the tensor cores
            if (issued >= 2 && !failed && !warp_wait(&sh.tc.pv_done[grp][pb], ((issued >> 1) - 1) & 1, &sh.abort_flag))
                failed = true;
            // rows past the slice end that the P . V k-steps read may hold anything
            // (NaN too): zero their latent features (their scores are masked, so a
            // score computed from half-zeroed bytes is discarded)
            if (v_hi < 16 * ksteps) {
                const int n_units = (16 * ksteps - v_hi) * 64;   // 8 chunks x 8 units per row
                for (int u = gw * 32 + lane; u < n_units; u += kGroupThreads) {
                    const int r = v_hi + (u >> 6);
                    st_shared_v4_zero(sbase + ((u >> 3) & 7) * kDenseChunkBytes + r * 128 + (u & 7) * 16);
                }
                fence_proxy_async_smem();
            }

            // ---- P against the group's reference; move it only when needed ----
            float pv[4];
            bool need = true;
            if (k > 0) {
                const float ref0 = m_ref[0] == -INFINITY ? 0.f : m_ref[0];
                const float ref1 = m_ref[1] == -INFINITY ? 0.f : m_ref[1];
                pv[0] = ex2_approx(sc[0] - ref0);
                pv[1] = ex2_approx(sc[1] - ref0);
                pv[2] = ex2_approx(sc[2] - ref1);
                pv[3] = ex2_approx(sc[3] - ref1);
                uint32_t hi0, lo0, hi1, lo1;
                split_pair<kFp8>(pv, hi0, lo0, hi1, lo1);
                st_shared_b32(pt_w, hi0);
                st_shared_b32(pt_w + 1024, hi1);
                st_shared_b32(pt_w + 2048, lo0);
                st_shared_b32(pt_w + 3072, lo1);
                fence_proxy_async_smem();
                const bool over = mx0 > m_ref[0] + kRescaleThreshold || mx1 > m_ref[1] + kRescaleThreshold;
                need = named_barrier_or(bar_group, kGroupThreads, over || failed);
            }
            if (need) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                if (tq == 0) {
                    sh.mx[grp][gw][g] = mx0;
                    sh.mx[grp][gw][g + 8] = mx1;
                }
                if (named_barrier_or(bar_group, kGroupThreads, failed)) {
                    gstop = true;
                    break;
                }
                float n0 = m_ref[0], n1 = m_ref[1];
#pragma unroll
                for (int v = 0; v < kGroupWarps; ++v) {
                    n0 = fmaxf(n0, sh.mx[grp][v][g]);
                    n1 = fmaxf(n1, sh.mx[grp][v][g + 8]);
                }
                if (k > 0) {
                    // what was accumulated against the old reference, scaled to the new
                    // one: O^T in tensor memory once the group's last batch is done
                    const float a0 = m_ref[0] == -INFINITY ? 0.f : ex2_approx(m_ref[0] - n0);
                    const float a1 = m_ref[1] == -INFINITY ? 0.f : ex2_approx(m_ref[1] - n1);
                    l_own[0] *= a0;
                    l_own[1] *= a1;
                    const int last = issued - 1;
                    if (!warp_wait(&sh.tc.pv_done[grp][last & 1], (last >> 1) & 1, &sh.abort_flag)) failed = true;
                    tc_fence_after_sync();
                    if (!failed) {
                        float al[kHeadGroup];
#pragma unroll
                        for (int h = 0; h < 8; ++h) {
                            al[h] = __shfl_sync(0xffffffffu, a0, 4 * h);
                            al[h + 8] = __shfl_sync(0xffffffffu, a1, 4 * h);
                        }
#pragma unroll 1
                        for (int blk = 0; blk < 4; ++blk) {
                            float v[32];
                            const uint32_t ta = tmem_grp + tmem_lane + 32u * blk;
                            tmem_ld32(ta, v);
                            float v_hi16[16], v_lo16[16];
#pragma unroll
                            for (int h = 0; h < kHeadGroup; ++h) {
                                v_hi16[h] = v[h] * al[h];
                                v_lo16[h] = v[16 + h] * al[h];
                            }
                            tmem_st16(ta, v_hi16);
                            tmem_st16(ta + 16, v_lo16);
                        }
                    }
                    tc_fence_before_sync();
                }
                m_ref[0] = n0;
                m_ref[1] = n1;
                const float ref0 = n0 == -INFINITY ? 0.f : n0;
                const float ref1 = n1 == -INFINITY ? 0.f : n1;
                pv[0] = ex2_approx(sc[0] - ref0);
                pv[1] = ex2_approx(sc[1] - ref0);
                pv[2] = ex2_approx(sc[2] - ref1);
                pv[3] = ex2_approx(sc[3] - ref1);
                uint32_t hi0, lo0, hi1, lo1;
                split_pair<kFp8>(pv, hi0, lo0, hi1, lo1);
                st_shared_b32(pt_w, hi0);
                st_shared_b32(pt_w + 1024, hi1);
                st_shared_b32(pt_w + 2048, lo0);
                st_shared_b32(pt_w + 3072, lo1);
                fence_proxy_async_smem();
                if (named_barrier_or(bar_group, kGroupThreads, failed)) {
                    gstop = true;
                    break;
                }
            }
            l_own[0] += pv[0] + pv[1];
            l_own[1] += pv[2] + pv[3];

            // ---- O^T += V^T . [P_hi | P_lo]^T on the tensor cores ---------------
            if (issuer) {
                tc_fence_after_sync();
                const uint64_t vb = v_desc0 + ((static_cast<uint32_t>(slot) * kSlotBytes) >> 4);
                const uint64_t pbd = p_desc0 + ((static_cast<uint32_t>(pb) * 64u) >> 4);
#pragma unroll
                for (int jb = 0; jb < 4; ++jb) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        if (kk < ksteps)
                            umma_bf16(tmem_grp + 32u * jb,
                                      vb + ((static_cast<uint32_t>(2 * jb * kDenseChunkBytes + kk * 2048)) >> 4),
                                      pbd + ((static_cast<uint32_t>(kk) * 32u) >> 4), idesc,
                                      (k == 0 && kk == 0) ? 0u : 1u);
                    }
                }
                umma_commit(&sh.empty[slot]);
                umma_commit(&sh.tc.pv_done[grp][pb]);
            }
            __syncwarp();
            ++issued;
        }
        // the other group's batches of this item (every thread follows both counts)
        issued_other += grp == 0 ? it.n_slots / 2 : (it.n_slots + 1) / 2;

        // ---- epilogue ---------------------------------------------------------
        float l0 = l_own[0], l1 = l_own[1];
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        if (tq == 0) {
            sh.lsum[grp][gw][g] = l0;
            sh.lsum[grp][gw][g + 8] = l1;
        }
        if (named_barrier_or(kBarMma, kMmaThreads, failed || gstop)) {
            stop = true;
            break;
        }
        if (gw == 0 && tq == 0) {
            float L0 = 0.f, L1 = 0.f;
#pragma unroll
            for (int v = 0; v < kGroupWarps; ++v) {
                L0 += sh.lsum[grp][v][g];
                L1 += sh.lsum[grp][v][g + 8];
            }
            sh.tc.merge_m[grp][g] = m_ref[0];
            sh.tc.merge_m[grp][g + 8] = m_ref[1];
            sh.tc.merge_l[grp][g] = L0;
            sh.tc.merge_l[grp][g + 8] = L1;
        }
        named_barrier_sync(kBarMma, kMmaThreads);
        // merge weights of head (lane & 15): group 1 holds rows only with two or more slots
        const bool two = it.n_slots > 1;
        const long long row_h0 = row_b + it.s;
        float c0_l, c1_l;
        {
            const int h = lane & 15;
            const float m0 = sh.tc.merge_m[0][h];
            const float m1 = two ? sh.tc.merge_m[1][h] : -INFINITY;
            const float mm = fmaxf(m0, m1);
            const float s0 = m0 == -INFINITY ? 0.f : ex2_approx(m0 - mm);
            const float s1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - mm);
            const float L = sh.tc.merge_l[0][h] * s0 + (two ? sh.tc.merge_l[1][h] * s1 : 0.f);
            // (v_scale: the E4M3 cache's scale, 1 for bf16; oscale adds the 2^-7 of P)
            const float oscale = kFp8 ? p.v_scale * (1.f / kFp8PScale) : p.v_scale;
            const float inv = L > 0.f ? rcp_approx(L) * oscale : 0.f;
            c0_l = s0 * inv;
            c1_l = s1 * inv;
            if (w == 0 && lane < 16)
                p.lse_part[row_h0 + static_cast<long long>(h) * p.splits] =
                    L > 0.f ? (mm + lg2_approx(L)) * kLn2 : -INFINITY;
        }
        // every P . V batch of both groups has completed (group 0 has at least one)
        if (!failed) {
            const int last0 = (grp == 0 ? issued : issued_other) - 1;
            if (!warp_wait(&sh.tc.pv_done[0][last0 & 1], (last0 >> 1) & 1, &sh.abort_flag)) failed = true;
        }
        if (two && !failed) {
            const int last1 = (grp == 1 ? issued : issued_other) - 1;
            if (!warp_wait(&sh.tc.pv_done[1][last1 & 1], (last1 >> 1) & 1, &sh.abort_flag)) failed = true;
        }
        tc_fence_after_sync();
        if (!failed) {
            // this warp: lane quarter gw of feature blocks 2 grp, 2 grp + 1
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
                const int jb = 2 * grp + jj;
                float a[32], b[32];
                tmem_ld32(tmem + tmem_lane + 32u * jb, a);
                if (two) {
                    tmem_ld32(tmem + 128u + tmem_lane + 32u * jb, b);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) b[i] = 0.f;
                }
                float* dst = p.o_part + row_h0 * kDLatent + 128 * jb + 32 * gw + lane;
#pragma unroll
                for (int h = 0; h < kHeadGroup; ++h) {
                    const float c0 = __shfl_sync(0xffffffffu, c0_l, h);
                    const float c1 = __shfl_sync(0xffffffffu, c1_l, h);
                    dst[static_cast<long long>(h) * p.splits * kDLatent] =
                        (a[h] + a[16 + h]) * c0 + (b[h] + b[16 + h]) * c1;
                }
            }
        }
        // every tensor-memory read of this item precedes the next item's MMAs
        tc_fence_before_sync();
        if (named_barrier_or(kBarMma, kMmaThreads, failed)) {
            stop = true;
            break;
        }
        stage += it.n_slots;
    }
    if ((stop || failed) && lane == 0) raise_device_error(sh, p.status);
    // no MMA in flight once the CTA frees its tensor memory
    if (issuer) {
        umma_commit(&sh.tc.drain[grp]);
        volatile int never = 0;
        if (!mbar_wait_bounded(&sh.tc.drain[grp], 0, &never)) raise_device_error(sh, p.status);
    }
    __syncwarp();
    tc_fence_before_sync();
    named_barrier_sync(kBarMma, kMmaThreads);
    if (w == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kDense, bool kFp8 = false, bool kTcPv = false>
__global__ void __launch_bounds__(kThreads, 1) mla_partial_mma_kernel(const __grid_constant__ TcMaps maps,
                                                                       const PartialParams p) {
    static_assert(!kTcPv || kDense, "tcgen05 P . V: dense caches");
    using S = SharedStorage<kDense, kFp8, kTcPv>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    S& sh = *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            for (int q = 0; q < (kDense ? 1 : kProdWarps); ++q) mbar_init(&sh.full[i][q], 1);
            // released by the group that consumed the slot (its four warps, or
            // the commit of its P . V MMAs)
            mbar_init(&sh.empty[i], kTcPv ? 1 : kGroupWarps);
        }
        if constexpr (kTcPv) {
            for (int gg = 0; gg < kGroups; ++gg) {
                mbar_init(&sh.tc.pv_done[gg][0], 1);
                mbar_init(&sh.tc.pv_done[gg][1], 1);
                mbar_init(&sh.tc.drain[gg], 1);
            }
        }
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, kComputeWarps);
        mbar_init(&sh.stall_bar, 1);
        mbar_init(&sh.patch_bar, 1);
        if constexpr (kFp8) {
            for (int i = 0; i < kSlots; ++i) mbar_init(&sh.fp8.full[i], 1);
        }
        sh.abort_flag = 0;
        mbar_init_fence();
    }
    if (threadIdx.x == kProducerWarp * 32) {
        // the descriptors are kernel parameters: fetch them while the grid
        // dependency is pending
        prefetch_tensormap(&maps.q);
        if constexpr (kDense) prefetch_tensormap(&maps.kv);
    }
    __syncthreads();
    // Inputs (d_pos, cache rows, indices, q) may be written by the kernel
    // before this one on the stream: every read that counts waits for it.
    // Each role's register share is set right before its code.
    if (warp >= kComputeWarps) {
        warpgroup_regs_decrease<RegSplit<kFp8>::kProducer>();
        if constexpr (kDense) {
            if (warp == kProducerWarp + 1 && lane == 0) prefetch_first_slots(maps, p);
        }
        if (warp == kProducerWarp + 2 && lane == 0) prefetch_first_inputs<kDense>(maps, p);
        if constexpr (kFp8) {
            // all four warps widen the E4M3 rows; one thread also stages them
            grid_dependency_wait();
            allow_dependent_launch();
            producer_fp8(maps, p, sh, warp - kProducerWarp, lane);
        } else if (warp == kProducerWarp || !kDense) {
            grid_dependency_wait();
            allow_dependent_launch();
            producer<kDense>(maps, p, sh, warp - kProducerWarp, lane);
        }
    } else {
        warpgroup_regs_increase<RegSplit<kFp8>::kMma>();
        grid_dependency_wait();
        allow_dependent_launch();
        if constexpr (kTcPv)
            consumer_tcpv<kFp8>(p, sh, warp, lane);
        else
            consumer<kDense, kFp8>(p, sh, warp, lane);
    }
}

template <bool kDense, bool kFp8 = false, bool kTcPv = false>
size_t smem_bytes() {
    return sizeof(SharedStorage<kDense, kFp8, kTcPv>) + 1024;
}
static_assert(sizeof(SharedStorage<true>) + 1024 <= 227 * 1024, "dense shared memory");
static_assert(sizeof(SharedStorage<true, false, true>) + 1024 <= 227 * 1024, "dense shared memory (tcgen05 P . V)");
static_assert(sizeof(SharedStorage<true, true, true>) + 1024 <= 227 * 1024,
              "E4M3 dense shared memory (tcgen05 P . V)");
using TcPvStorage = SharedStorage<true, false, true>;
static_assert(offsetof(TcPvStorage, tc) % 1024 == 0, "P^T buffers 1024-byte aligned");
static_assert(sizeof(SharedStorage<false>) + 1024 <= 227 * 1024, "sparse shared memory");
static_assert(sizeof(SharedStorage<true, true>) + 1024 <= 227 * 1024, "E4M3 dense shared memory");

}  // namespace

size_t partial_mma_smem_bytes(bool fp8, bool tc_pv) {
    if (fp8) return tc_pv ? smem_bytes<true, true, true>() : smem_bytes<true, true>();
    if (tc_pv) return smem_bytes<true, false, true>();
    return smem_bytes<false>() > smem_bytes<true>() ? smem_bytes<false>() : smem_bytes<true>();
}
int partial_mma_block_threads() { return kThreads; }

template <bool kDense, bool kFp8 = false, bool kTcPv = false>
cudaError_t prepare_one() {
    // the register split assumes kLaunchRegs per thread at launch: with fewer,
    // the MMA warpgroups' increase could never be granted
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, mla_partial_mma_kernel<kDense, kFp8, kTcPv>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < kLaunchRegs || fa.maxThreadsPerBlock < kThreads) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(mla_partial_mma_kernel<kDense, kFp8, kTcPv>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem_bytes<kDense, kFp8, kTcPv>()));
}

cudaError_t partial_mma_prepare(int /*device*/) {
    cudaError_t e = prepare_one<true>();
    if (e == cudaSuccess) e = prepare_one<false>();
    if (e == cudaSuccess) e = prepare_one<true, true>();
    if (e == cudaSuccess) e = prepare_one<true, false, true>();
    if (e == cudaSuccess) e = prepare_one<true, true, true>();
    return e;
}

cudaError_t partial_mma_occupancy(int* ctas_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, mla_partial_mma_kernel<false>, kThreads,
                                                         smem_bytes<false>());
}

cudaError_t launch_partial_mma(const TcMaps& maps, const PartialParams& p, dim3 grid, bool pdl,
                               cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = p.sparse   ? smem_bytes<false>()
                           : p.kv_fp8 ? (p.tc_pv ? smem_bytes<true, true, true>() : smem_bytes<true, true>())
                           : p.tc_pv  ? smem_bytes<true, false, true>()
                                      : smem_bytes<true>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (p.sparse) return cudaLaunchKernelEx(&cfg, mla_partial_mma_kernel<false>, maps, p);
    if (p.kv_fp8 && p.tc_pv) return cudaLaunchKernelEx(&cfg, mla_partial_mma_kernel<true, true, true>, maps, p);
    if (p.kv_fp8) return cudaLaunchKernelEx(&cfg, mla_partial_mma_kernel<true, true>, maps, p);
    if (p.tc_pv) return cudaLaunchKernelEx(&cfg, mla_partial_mma_kernel<true, false, true>, maps, p);
    return cudaLaunchKernelEx(&cfg, mla_partial_mma_kernel<true>, maps, p);
}

}  // namespace mla
