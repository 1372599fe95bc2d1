// mla_decode_api.cu -- the C ABI declared in include/mla_decode.h: the
// planner, argument checks and kernel launches.  Host code only.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "mla_decode.h"
#include "mla_internal.h"
#include "slicing.cuh"

namespace {

constexpr int kPlanMagic = 0x4d4c4131;       // "MLA1"
static_assert(mla::kStaticScratchBytes == MLA_STATIC_SCRATCH_BYTES, "static scratch size differs from the header");
constexpr int kMaxDevices = 64;
// The partial kernel is persistent with one CTA per SM: its 5-stage ring of
// cache rows fills the shared memory.  The two-CTAs-per-SM target named in
// "Launch Geometry" (Lecture 04, s.4: kMlaBlocksPerSm = 2) was there so one
// CTA's loads overlap another's math; here the producer warp and the MMA warps
// of one CTA overlap them through the ring instead.
constexpr int kCtasPerSm = 1;
constexpr size_t kScratchAlign = 256;
constexpr int kVariantWarpMma = 1;           // mma.sync head-group-16 kernel, 64-row steps of 32-row slots
constexpr int kVariantTc = 2;                // tcgen05 head-group-16 kernel, 80-row tiles
constexpr int kVariantTc32 = 3;              // tcgen05 head-group-32 kernel, 64-row tiles (dense)
constexpr int kVariantTc64 = 4;              // tcgen05 head-group-64 kernel, 64-row tiles (dense)
constexpr int kVariantMmaTcPv = 5;           // warp-MMA kernel with P . V on tcgen05 (dense bf16)

int variant_tile_rows(int v) {
    // warp-MMA: the model counts 32-row slots (a 64-row step costs about two)
    return v == kVariantTc ? mla::kTcTileRows : (v == kVariantTc32 || v == kVariantTc64) ? mla::kTcTileRows32
                                                                                          : mla::kStageRows;
}
bool variant_is_mma(int v) { return v == kVariantWarpMma || v == kVariantMmaTcPv; }
int variant_granule(int v) { return variant_is_mma(v) ? mla::kStageRows : mla::kTcGranule; }
int variant_head_group(int v) { return v == kVariantTc64 ? 64 : v == kVariantTc32 ? 32 : mla::kHeadGroup; }
bool variant_is_tc(int v) { return v == kVariantTc || v == kVariantTc32 || v == kVariantTc64; }

// cuTensorMapEncodeTiled, reached through the runtime (no link-time libcuda).
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult qr{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode;
}

// Rank-3 view of bf16 rows of 576: {64 elements, rows, 9 chunks of 64} with
// strides {row stride, 128 bytes}; a box {64, box_rows, box_chunks} lands in
// shared memory as [chunk][row][64], 128-byte swizzled.
int encode_bf16_row_chunks(CUtensorMap* map, const void* base, long long rows, long long row_stride_elems,
                           uint32_t box_rows, uint32_t box_chunks) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return MLA_ECUDA;
    const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(MLA_D_ROW / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_stride_elems) * 2u, 128u};
    const cuuint32_t box[3] = {64u, box_rows, box_chunks};
    const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                           elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MLA_OK : MLA_ECUDA;
}

// Rank-3 view of E4M3 rows of 576 bytes: {64 bytes, rows, 9 chunks of 64}
// with strides {row stride, 64 bytes}; a box {64, 32, 9} lands in shared
// memory unswizzled as [chunk][row][64 bytes].
int encode_e4m3_row_chunks(CUtensorMap* map, const void* base, long long rows, long long row_stride_bytes) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return MLA_ECUDA;
    const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(MLA_D_ROW / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_stride_bytes), 64u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(mla::kStageRows), static_cast<cuuint32_t>(MLA_D_ROW / 64)};
    const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                           elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MLA_OK : MLA_ECUDA;
}

std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_prepared[kMaxDevices];
std::mutex g_prepare_mutex;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
bool misaligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; }

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ECUDA;
    }
    if (*dev < 0 || *dev >= kMaxDevices) return MLA_ECUDA;
    return MLA_OK;
}

int device_sm_count(int dev, int* sms) {
    int cached = g_sm_count[dev].load(std::memory_order_relaxed);
    if (cached == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
            cudaGetLastError();
            return MLA_ECUDA;
        }
        g_sm_count[dev].store(v, std::memory_order_relaxed);
        cached = v;
    }
    *sms = cached;
    return MLA_OK;
}

// Kernel attributes are set once per device, outside any capture
// ("Graph-resident decode", Lecture 08, s.3: lazy initialisation inside a
// capture breaks it, so it is done up front).
int prepare_device(int dev) {
    if (g_prepared[dev].load(std::memory_order_acquire)) return MLA_OK;
    std::lock_guard<std::mutex> lock(g_prepare_mutex);
    if (g_prepared[dev].load(std::memory_order_acquire)) return MLA_OK;
    if (mla::partial_mma_prepare(dev) != cudaSuccess || mla::partial_tc_prepare(dev) != cudaSuccess ||
        mla::combine_prepare() != cudaSuccess) {
        cudaGetLastError();
        return MLA_ECUDA;
    }
    g_prepared[dev].store(1, std::memory_order_release);
    return MLA_OK;
}

int ensure_prepared(cudaStream_t stream) {
    int dev = 0;
    int rc = current_device(&dev);
    if (rc != MLA_OK) return rc;
    if (g_prepared[dev].load(std::memory_order_acquire)) return MLA_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ECUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return MLA_ENOTREADY;
    return prepare_device(dev);
}

int check_shape(const mla_decode_shape* s) {
    if (!s) return MLA_EINVAL;
    if (s->batch < 1 || s->batch > 65535) return MLA_EINVAL;
    if (s->sparse != 0 && s->sparse != 1) return MLA_EINVAL;
    if (s->pdl != 0 && s->pdl != 1) return MLA_EINVAL;
    if (s->stall_test != 0 && s->stall_test != 1) return MLA_EINVAL;
    if (s->kv_fp8 != 0 && s->kv_fp8 != 1) return MLA_EINVAL;
    if (s->variant < 0 || s->variant > 5) return MLA_EINVAL;
    if (s->num_sms < 0 || s->splits_override < 0 || s->splits_override > MLA_MAX_SPLITS) return MLA_EINVAL;
    if (!(s->scale > 0.f) || !std::isfinite(s->scale)) return MLA_EINVAL;
    if (!s->sparse && s->max_ctx < 1) return MLA_EINVAL;
    if (s->sparse && s->topk < 1) return MLA_EINVAL;
    if (s->d_latent != MLA_D_LATENT || s->d_rope != MLA_D_ROPE) return MLA_EUNSUPPORTED;
    if (s->heads != 16 && s->heads != 32 && s->heads != 64 && s->heads != 128) return MLA_EUNSUPPORTED;
    // 32 heads per CTA: dense decode with a multiple of 32 heads
    if (s->variant == kVariantTc32 && (s->sparse || s->heads % 32 != 0)) return MLA_EUNSUPPORTED;
    // 64 heads per CTA: dense decode with a multiple of 64 heads
    if (s->variant == kVariantTc64 && (s->sparse || s->heads % 64 != 0)) return MLA_EUNSUPPORTED;
    // E4M3 cache: dense decode on the warp-MMA kernel
    if (s->kv_fp8 && (s->sparse || (s->variant != 0 && !variant_is_mma(s->variant)))) return MLA_EUNSUPPORTED;
    // P . V on tcgen05 reads V in place from the swizzled dense slots: dense only
    if (s->variant == kVariantMmaTcPv && s->sparse) return MLA_EUNSUPPORTED;
    return MLA_OK;
}

// Scratch layout of a plan: the status word at 0, then o_part fp32
// [B][H][S][512] and lse_part fp32 [B][H][S], each 256-byte aligned.
struct ScratchLayout {
    size_t status, o_part, lse_part, bytes;
};
ScratchLayout scratch_layout(int batch, int heads, int splits) {
    const size_t bhs = static_cast<size_t>(batch) * heads * splits;
    ScratchLayout l;
    l.status = 0;
    l.o_part = kScratchAlign;
    l.lse_part = align_up(l.o_part + bhs * MLA_D_LATENT * sizeof(float), kScratchAlign);
    l.bytes = align_up(l.lse_part + bhs * sizeof(float), kScratchAlign);
    return l;
}

int check_plan(const mla_decode_plan_t* pl) {
    if (!pl || pl->magic != kPlanMagic) return MLA_EINVAL;
    if (check_shape(&pl->shape) != MLA_OK) return MLA_EINVAL;
    if (pl->splits < 1 || pl->splits > MLA_MAX_SPLITS) return MLA_EINVAL;
    if (!variant_is_mma(pl->variant) && !variant_is_tc(pl->variant)) return MLA_EINVAL;
    if ((pl->variant == kVariantTc32 || pl->variant == kVariantTc64 || pl->variant == kVariantMmaTcPv) &&
        pl->shape.sparse)
        return MLA_EINVAL;
    if (pl->head_group != variant_head_group(pl->variant) || pl->n_head_groups * pl->head_group != pl->shape.heads)
        return MLA_EINVAL;
    const long long items = static_cast<long long>(pl->shape.batch) * pl->n_head_groups * pl->splits;
    if (pl->grid_x < 1 || pl->grid_x > items || pl->grid_y != 1 || pl->grid_z != 1) return MLA_EINVAL;
    if (items > 0x7fffffffLL) return MLA_EINVAL;
    if (pl->flat_ranges < 0) return MLA_EINVAL;
    if (pl->flat_ranges > 0) {
        // flat split: batched sparse decode on the warp-MMA kernel, whole slots per range,
        // at most two requests per range, one CTA per range and head group
        if (!pl->shape.sparse || pl->variant != kVariantWarpMma || pl->shape.batch < 2) return MLA_EINVAL;
        const long long per = pl->entries_per_split;
        if (per < mla::kStageRows || per % mla::kStageRows != 0 || per > pl->shape.topk) return MLA_EINVAL;
        if (static_cast<long long>(pl->flat_ranges) * per <
                static_cast<long long>(pl->shape.batch) * pl->shape.topk ||
            static_cast<long long>(pl->flat_ranges - 1) * per >=
                static_cast<long long>(pl->shape.batch) * pl->shape.topk)
            return MLA_EINVAL;
        if (static_cast<long long>(pl->grid_x) != static_cast<long long>(pl->flat_ranges) * pl->n_head_groups)
            return MLA_EINVAL;
    }
    if (pl->combine_grid_x != mla::combine_grid_rows(pl->shape.batch * pl->shape.heads, pl->splits) ||
        pl->combine_grid_y != MLA_D_LATENT / mla::kCombineChunk || pl->combine_block != mla::combine_block_threads())
        return MLA_EINVAL;
    // the kernels write B*H*S partial rows at these offsets: a plan whose
    // layout does not match its split count would write past the region
    const ScratchLayout l = scratch_layout(pl->shape.batch, pl->shape.heads, pl->splits);
    if (pl->status_offset != l.status || pl->o_part_offset != l.o_part || pl->lse_part_offset != l.lse_part ||
        pl->scratch_bytes != l.bytes)
        return MLA_EINVAL;
    return MLA_OK;
}

int check_args(const mla_decode_plan_t* pl, const mla_decode_args* a) {
    if (!a || !a->q || !a->kv || !a->out || !a->lse) return MLA_EINVAL;
    if (a->kv_rows < 1 || a->row_stride < MLA_D_ROW) return MLA_EINVAL;
    if (pl->shape.kv_fp8) {
        // row stride in bytes, 16-byte aligned rows; a finite positive scale
        if (a->row_stride % 16 != 0) return MLA_EALIGN;
        if (!(a->kv_scale > 0.f) || !std::isfinite(a->kv_scale)) return MLA_EINVAL;
    } else if (a->row_stride % 8 != 0) {
        return MLA_EALIGN;
    }
    if (misaligned(a->q, 16) || misaligned(a->kv, 16) || misaligned(a->out, 16) || misaligned(a->lse, 4))
        return MLA_EALIGN;
    if (a->row_offset && misaligned(a->row_offset, 8)) return MLA_EALIGN;
    if (!pl->shape.sparse) {
        if (!a->d_pos) return MLA_EINVAL;
        if (misaligned(a->d_pos, 4)) return MLA_EALIGN;
        if (pl->shape.batch > 1 && !a->row_offset) return MLA_EINVAL;
    } else {
        if (!a->indices || !a->cache_len || !a->row_offset) return MLA_EINVAL;
        if (misaligned(a->indices, 4) || misaligned(a->cache_len, 4)) return MLA_EALIGN;
    }
    return MLA_OK;
}

int check_scratch(const mla_decode_plan_t* pl, const void* scratch, size_t bytes) {
    if (!scratch || misaligned(scratch, kScratchAlign) || bytes < pl->scratch_bytes) return MLA_ESCRATCH;
    return MLA_OK;
}

int launch_status(cudaError_t e) {
    if (e == cudaSuccess) return MLA_OK;
    cudaGetLastError();
    return MLA_ECUDA;
}

// Fused decode-step state update (mla_decode_forward_step): the new rows
// and whether d_pos advances after the merge.
struct StepUpdate {
    const uint16_t* new_rows;
    int advance;
};

int do_run(const mla_decode_plan_t* pl, const mla_decode_args* a, void* scratch, size_t bytes, void* stream,
           const StepUpdate* up = nullptr) {
    int rc = check_plan(pl);
    if (rc == MLA_OK) rc = check_args(pl, a);
    if (rc == MLA_OK) rc = check_scratch(pl, scratch, bytes);
    if (rc != MLA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = ensure_prepared(st);
    if (rc != MLA_OK) return rc;
    char* base = static_cast<char*>(scratch);
    mla::PartialParams p{};
    p.q = static_cast<const uint16_t*>(a->q);
    p.kv = static_cast<const uint16_t*>(a->kv);
    p.kv_rows = a->kv_rows;
    p.row_stride = a->row_stride;
    p.d_pos = a->d_pos;
    p.row_offset = a->row_offset;
    p.cache_len = a->cache_len;
    p.indices = a->indices;
    p.batch = pl->shape.batch;
    p.heads = pl->shape.heads;
    p.topk = pl->shape.topk;
    p.splits = pl->splits;
    p.sparse = pl->shape.sparse;
    p.n_groups = pl->n_head_groups;
    p.n_items = pl->shape.batch * pl->n_head_groups * pl->splits;
    p.flat_ranges = pl->flat_ranges;
    p.flat_per = pl->entries_per_split;
    if (pl->flat_ranges > 0) p.n_items = 2 * pl->flat_ranges * pl->n_head_groups;
    p.granule = variant_granule(pl->variant);
    p.scale_log2 = pl->shape.scale * 1.4426950408889634f;
    p.kv_fp8 = pl->shape.kv_fp8;
    p.v_scale = 1.f;
    if (pl->shape.kv_fp8) {
        // every value is e4m3(byte) * kv_scale: the scores carry it through the
        // score scale, the partial multiplies O by it
        p.scale_log2 *= a->kv_scale;
        p.v_scale = a->kv_scale;
    }
    p.o_part = reinterpret_cast<float*>(base + pl->o_part_offset);
    p.lse_part = reinterpret_cast<float*>(base + pl->lse_part_offset);
    p.status = reinterpret_cast<int*>(base + pl->status_offset);
    p.stall_test = pl->shape.stall_test;
    p.new_rows = up ? up->new_rows : nullptr;
    p.tc_pv = pl->variant == kVariantMmaTcPv ? 1 : 0;
    const dim3 grid(pl->grid_x, pl->grid_y, pl->grid_z);
    if (variant_is_tc(pl->variant)) {
        // TMA coordinates are 32-bit: the cache must be addressable by them
        if (a->kv_rows > 0x7fffff00LL) return MLA_EUNSUPPORTED;
        const int hg = variant_head_group(pl->variant);
        mla::TcMaps maps;
        rc = encode_bf16_row_chunks(&maps.kv, a->kv, a->kv_rows, a->row_stride,
                                    static_cast<uint32_t>(variant_tile_rows(pl->variant)), mla::kTcBoxChunks);
        if (rc == MLA_OK)
            rc = encode_bf16_row_chunks(&maps.q, a->q, static_cast<long long>(pl->shape.batch) * pl->shape.heads,
                                        MLA_D_ROW, static_cast<uint32_t>(hg), MLA_D_ROW / 64);
        if (rc != MLA_OK) return rc;
        return launch_status(mla::launch_partial_tc(maps, p, hg, grid, pl->shape.pdl != 0, st));
    }
    // warp-MMA kernel: the query tile by TMA; dense cache rows by one TMA box
    // per 32-row slot (E4M3 rows: one box of bytes, widened in shared memory),
    // sparse rows by per-row bulk copies
    mla::TcMaps maps{};
    if (!pl->shape.sparse) {
        if (a->kv_rows > 0x7fffff00LL) return MLA_EUNSUPPORTED;
        rc = pl->shape.kv_fp8
                 ? encode_e4m3_row_chunks(&maps.kv, a->kv, a->kv_rows, a->row_stride)
                 : encode_bf16_row_chunks(&maps.kv, a->kv, a->kv_rows, a->row_stride, mla::kStageRows, MLA_D_ROW / 64);
        if (rc != MLA_OK) return rc;
    }
    rc = encode_bf16_row_chunks(&maps.q, a->q, static_cast<long long>(pl->shape.batch) * pl->shape.heads, MLA_D_ROW,
                                mla::kHeadGroup, MLA_D_ROW / 64);
    if (rc != MLA_OK) return rc;
    return launch_status(mla::launch_partial_mma(maps, p, grid, pl->shape.pdl != 0, st));
}

int do_combine(const mla_decode_plan_t* pl, const mla_decode_args* a, const void* scratch, size_t bytes,
               void* stream, const StepUpdate* up = nullptr) {
    int rc = check_plan(pl);
    if (rc == MLA_OK) rc = check_args(pl, a);
    if (rc == MLA_OK) rc = check_scratch(pl, scratch, bytes);
    if (rc != MLA_OK) return rc;
    const char* base = static_cast<const char*>(scratch);
    mla::CombineParams c{};
    c.o_part = reinterpret_cast<const float*>(base + pl->o_part_offset);
    c.lse_part = reinterpret_cast<const float*>(base + pl->lse_part_offset);
    c.status = reinterpret_cast<const int*>(base + pl->status_offset);
    c.out = a->out;
    c.lse = a->lse;
    c.batch = pl->shape.batch;
    c.heads = pl->shape.heads;
    c.splits = pl->splits;
    c.sparse = pl->shape.sparse;
    c.topk = pl->shape.topk;
    c.d_pos = a->d_pos;
    c.row_offset = a->row_offset;
    c.kv_rows = a->kv_rows;
    c.granule = variant_granule(pl->variant);
    if (up) {
        // the step's caller hands over the cache and d_pos for writing
        c.new_rows = up->new_rows;
        c.kv = static_cast<uint16_t*>(const_cast<void*>(a->kv));
        c.row_stride = a->row_stride;
        c.d_pos_rw = const_cast<int*>(a->d_pos);
        c.advance = up->advance;
    }
    const bool spread = static_cast<long long>(pl->combine_grid_x) * pl->combine_grid_y <= pl->num_sms;
    return launch_status(mla::launch_combine(c, dim3(pl->combine_grid_x, pl->combine_grid_y, 1), pl->combine_block,
                                             pl->shape.pdl != 0, spread, static_cast<cudaStream_t>(stream)));
}

// Split count derived from the shape ("Launch Geometry", Lecture 04, s.4:
// derive it, do not pin it): minimise the modelled partial-kernel time
//   waves(S) * (kernel steps per slice(S) + 1),  waves = ceil(items / grid),
// over S, where a slice is ceil(rows / S) rounded up to the kernel's granule,
// a step is its tile (80 rows tcgen05, 32 rows warp-MMA) and only non-empty
// slices are items; the smallest S wins ties.
long long derive_splits(long long rows, long long pairs, long long grid_cap, int variant) {
    const int tile = variant_tile_rows(variant);
    const int granule = variant_granule(variant);
    long long best_s = 1, best_cost = -1;
    const long long s_hi = std::min<long long>(MLA_MAX_SPLITS, ceil_div(rows, granule));
    for (long long S = 1; S <= s_hi; ++S) {
        const long long per = mla::slice_entries(rows, static_cast<int>(S), granule);
        const long long items = pairs * ceil_div(rows, per);
        const long long waves = ceil_div(items, std::min(items, grid_cap));
        const long long cost = waves * (ceil_div(per, tile) + 1);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_s = S;
        }
    }
    return best_s;
}

// Kernel choice when the caller leaves it open, from measurements on GB300:
// the warp-MMA kernel wins every sparse shape (per-row bulk copies gather
// more rows per SM than the tcgen05 kernel's 16-byte cp.async) and every
// dense shape with 16 heads (T = 256 .. 131072).  With 32 or more heads it
// reads each cache row once per 16-head group, so once its slices grow past
// 768 rows per item a tcgen05 kernel with the widest head group that divides
// H (64 heads per CTA: one read per 64 heads; else 32) is faster (measured,
// H = 64: tie at 864 rows per warp-MMA item, 64 heads per CTA 16% ahead at
// 1728; H = 128: 4% ahead at 864, 19% at 1728; H = 32: tie at 864, 32 heads
// per CTA ahead at 1728); below that the warp-MMA kernel wins.
constexpr long long kMmaMaxRowsPerItemWide = 768;
long long rows_per_item(long long rows, int batch, int heads, long long grid_cap, int variant) {
    const long long pairs = static_cast<long long>(batch) * (heads / variant_head_group(variant));
    const long long S = derive_splits(rows, pairs, grid_cap, variant);
    return mla::slice_entries(rows, static_cast<int>(S), variant_granule(variant));
}
// E4M3 caches: the warp-MMA kernel with P . V on tcgen05 (measured 5% faster
// than P . V on the warps at T = 8192, 32768 and 131072: its MMA warps, which
// bound the E4M3 path, then only take the scores).
int auto_variant(bool sparse, bool fp8, int batch, int heads, long long rows, long long grid_cap) {
    if (fp8) return kVariantMmaTcPv;
    if (sparse || heads == mla::kHeadGroup) return kVariantWarpMma;
    if (rows_per_item(rows, batch, heads, grid_cap, kVariantWarpMma) <= kMmaMaxRowsPerItemWide) return kVariantWarpMma;
    return heads % 64 == 0 ? kVariantTc64 : kVariantTc32;
}

// Flat split of batched sparse decode (warp-MMA kernel).  The uniform split
// gives every request S slices; B * S items either leave SMs idle or run in
// waves.  The flat split cuts the B * topk list entries (request after
// request) into one range per CTA and head group, a whole number of 32-row
// slots each and at most topk (so a range touches at most two requests: two
// items, the second often empty).  Modelled time: slots per range + 2 (two
// item set-ups) against the uniform waves * (slots per slice + 1); the flat
// split is taken only when strictly cheaper.
struct FlatSplit {
    int ranges, per, s_max;
    long long cost;
};
bool derive_flat(int batch, int topk, int n_groups, long long grid_cap, FlatSplit* out) {
    if (batch < 2 || n_groups < 1) return false;
    const long long G = grid_cap / n_groups;
    if (G < 2) return false;
    const long long total = static_cast<long long>(batch) * topk;
    long long per = ceil_div(total, G);
    per = ceil_div(per, mla::kStageRows) * mla::kStageRows;
    if (per > topk || per > 0x7fffffffLL) return false;
    const long long ranges = ceil_div(total, per);
    long long s_max = 1;
    for (long long b = 0; b < batch; ++b) {
        const long long first = b * topk / per, last = ((b + 1) * topk - 1) / per;
        s_max = std::max(s_max, last - first + 1);
    }
    if (s_max > MLA_MAX_SPLITS) return false;
    out->ranges = static_cast<int>(ranges);
    out->per = static_cast<int>(per);
    out->s_max = static_cast<int>(s_max);
    out->cost = per / mla::kStageRows + 2;
    return true;
}
long long uniform_cost(long long rows, long long pairs, long long grid_cap, int variant, long long S) {
    const long long per = mla::slice_entries(rows, static_cast<int>(S), variant_granule(variant));
    const long long items = pairs * ceil_div(rows, per);
    const long long waves = ceil_div(items, std::min(items, grid_cap));
    return waves * (ceil_div(per, variant_tile_rows(variant)) + 1);
}

// The static array of the current device (looked up on first use, outside capture).
int static_scratch_for(void* stream, void** out) {
    int dev = 0;
    const int rc = current_device(&dev);
    if (rc != MLA_OK) return rc;
    void* scratch = mla::static_scratch_if_ready(dev);
    if (!scratch) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) {
            cudaGetLastError();
            return MLA_ECUDA;
        }
        if (cs != cudaStreamCaptureStatusNone) return MLA_ENOTREADY;
        if (mla::static_scratch_set_up(dev, &scratch) != cudaSuccess) return MLA_ECUDA;
    }
    *out = scratch;
    return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode_abi_version(void) { return MLA_DECODE_ABI_VERSION; }

int mla_decode_plan(const mla_decode_shape* shape, mla_decode_plan_t* plan) {
    if (!plan) return MLA_EINVAL;
    int rc = check_shape(shape);
    if (rc != MLA_OK) return rc;
    const mla_decode_shape s = *shape;
    int sms = s.num_sms;
    if (sms == 0) {
        int dev = 0;
        rc = current_device(&dev);
        if (rc == MLA_OK) rc = device_sm_count(dev, &sms);
        if (rc == MLA_OK) rc = prepare_device(dev);
        if (rc != MLA_OK) return rc;
    }
    mla_decode_plan_t pl{};
    pl.shape = s;
    pl.magic = kPlanMagic;
    pl.head_group = mla::kHeadGroup;                      // set again once the kernel is chosen
    pl.n_head_groups = s.heads / mla::kHeadGroup;
    pl.ctas_per_sm = kCtasPerSm;
    pl.num_sms = sms;

    const long long rows = s.sparse ? s.topk : s.max_ctx;
    const long long grid_cap = static_cast<long long>(kCtasPerSm) * sms;
    pl.variant =
        s.variant != 0 ? s.variant : auto_variant(s.sparse != 0, s.kv_fp8 != 0, s.batch, s.heads, rows, grid_cap);
    pl.head_group = variant_head_group(pl.variant);
    pl.n_head_groups = s.heads / pl.head_group;
    const long long best_s =
        derive_splits(rows, static_cast<long long>(s.batch) * pl.n_head_groups, grid_cap, pl.variant);
    long long S = best_s;
    if (s.splits_override > 0) S = s.splits_override;
    pl.splits = static_cast<int>(S);
    pl.entries_per_split = static_cast<int>(mla::slice_entries(rows, pl.splits, variant_granule(pl.variant)));
    const long long items = static_cast<long long>(s.batch) * pl.n_head_groups * pl.splits;
    pl.grid_x = static_cast<int>(std::min(items, grid_cap));
    pl.flat_ranges = 0;
    FlatSplit fs{};
    if (s.sparse && pl.variant == kVariantWarpMma && s.splits_override == 0 &&
        derive_flat(s.batch, s.topk, pl.n_head_groups, grid_cap, &fs) &&
        fs.cost < uniform_cost(rows, static_cast<long long>(s.batch) * pl.n_head_groups, grid_cap, pl.variant, S)) {
        pl.flat_ranges = fs.ranges;
        pl.splits = fs.s_max;
        pl.entries_per_split = fs.per;
        pl.grid_x = fs.ranges * pl.n_head_groups;
    }
    pl.grid_y = 1;
    pl.grid_z = 1;
    const bool tc = variant_is_tc(pl.variant);
    pl.block = tc ? mla::partial_tc_block_threads(pl.head_group) : mla::partial_mma_block_threads();
    pl.smem_bytes = static_cast<int>(tc ? mla::partial_tc_smem_bytes(pl.head_group)
                                        : mla::partial_mma_smem_bytes(s.kv_fp8 != 0, pl.variant == kVariantMmaTcPv));
    pl.combine_grid_x = mla::combine_grid_rows(s.batch * s.heads, pl.splits);
    pl.combine_grid_y = MLA_D_LATENT / mla::kCombineChunk;
    pl.combine_block = mla::combine_block_threads();

    const ScratchLayout l = scratch_layout(s.batch, s.heads, pl.splits);
    pl.status_offset = l.status;
    pl.o_part_offset = l.o_part;
    pl.lse_part_offset = l.lse_part;
    pl.scratch_bytes = l.bytes;
    *plan = pl;
    return MLA_OK;
}

int mla_decode_run(const mla_decode_plan_t* plan, const mla_decode_args* args, void* scratch, size_t scratch_bytes,
                   void* stream) {
    return do_run(plan, args, scratch, scratch_bytes, stream);
}

int mla_decode_combine(const mla_decode_plan_t* plan, const mla_decode_args* args, const void* scratch,
                       size_t scratch_bytes, void* stream) {
    return do_combine(plan, args, scratch, scratch_bytes, stream);
}

int mla_decode_forward(const mla_decode_plan_t* plan, const mla_decode_args* args, void* scratch,
                       size_t scratch_bytes, void* stream) {
    int rc = do_run(plan, args, scratch, scratch_bytes, stream);
    if (rc != MLA_OK) return rc;
    return do_combine(plan, args, scratch, scratch_bytes, stream);
}

int mla_decode_forward_step(const mla_decode_plan_t* plan, const mla_decode_args* args, void* scratch,
                            size_t scratch_bytes, const void* new_rows, int advance, void* stream) {
    int rc = check_plan(plan);
    if (rc != MLA_OK) return rc;
    if (plan->shape.sparse || plan->shape.kv_fp8) return MLA_EUNSUPPORTED;
    if (!new_rows || (advance != 0 && advance != 1)) return MLA_EINVAL;
    if (misaligned(new_rows, 16)) return MLA_EALIGN;
    const StepUpdate up{static_cast<const uint16_t*>(new_rows), advance};
    rc = do_run(plan, args, scratch, scratch_bytes, stream, &up);
    if (rc != MLA_OK) return rc;
    return do_combine(plan, args, scratch, scratch_bytes, stream, &up);
}

int mla_decode_append(void* kv, long long kv_rows, long long row_stride, const void* new_rows, const int* d_pos,
                      const long long* row_offset, int batch, void* stream) {
    if (!kv || !new_rows || !d_pos || batch < 1 || kv_rows < 1 || row_stride < MLA_D_ROW) return MLA_EINVAL;
    if (batch > 1 && !row_offset) return MLA_EINVAL;
    if (row_stride % 8 != 0 || misaligned(kv, 16) || misaligned(new_rows, 16) || misaligned(d_pos, 4) ||
        (row_offset && misaligned(row_offset, 8)))
        return MLA_EALIGN;
    mla::AppendParams p{};
    p.kv = static_cast<uint16_t*>(kv);
    p.kv_rows = kv_rows;
    p.row_stride = row_stride;
    p.new_rows = static_cast<const uint16_t*>(new_rows);
    p.d_pos = d_pos;
    p.row_offset = row_offset;
    p.batch = batch;
    return launch_status(mla::launch_append(p, false, static_cast<cudaStream_t>(stream)));
}

int mla_decode_project(const float* latent, const void* wv_b, int batch, int heads, int v_dim, float* y, int pdl,
                       void* stream) {
    if (!latent || !wv_b || !y || batch < 1 || batch > 65535 || (pdl != 0 && pdl != 1)) return MLA_EINVAL;
    if (heads < 1 || heads > 128 || v_dim < 16 || v_dim > 512 || v_dim % 16 != 0) return MLA_EUNSUPPORTED;
    if (misaligned(latent, 16) || misaligned(wv_b, 16) || misaligned(y, 16)) return MLA_EALIGN;
    mla::ProjectParams p{};
    p.latent = latent;
    p.wv_b = static_cast<const uint16_t*>(wv_b);
    p.y = y;
    p.batch = batch;
    p.heads = heads;
    p.v_dim = v_dim;
    return launch_status(mla::launch_project(p, pdl != 0, static_cast<cudaStream_t>(stream)));
}

int mla_decode_advance(int* d_pos, int batch, void* stream) {
    if (!d_pos || batch < 1) return MLA_EINVAL;
    if (misaligned(d_pos, 4)) return MLA_EALIGN;
    return launch_status(mla::launch_advance(d_pos, batch, false, static_cast<cudaStream_t>(stream)));
}

int mla_decode_forward_static(const mla_decode_plan_t* plan, const mla_decode_args* args, void* stream) {
    int rc = check_plan(plan);
    if (rc == MLA_OK) rc = check_args(plan, args);
    if (rc != MLA_OK) return rc;
    if (plan->scratch_bytes > mla::kStaticScratchBytes) return MLA_ESTATICLIMIT;
    void* scratch = nullptr;
    rc = static_scratch_for(stream, &scratch);
    if (rc != MLA_OK) return rc;
    rc = do_run(plan, args, scratch, mla::kStaticScratchBytes, stream);
    if (rc != MLA_OK) return rc;
    return do_combine(plan, args, scratch, mla::kStaticScratchBytes, stream);
}

int mla_decode_static_status(int* status, void* stream) {
    if (!status) return MLA_EINVAL;
    if (misaligned(status, 4)) return MLA_EALIGN;
    void* scratch = nullptr;
    const int rc = static_scratch_for(stream, &scratch);
    if (rc != MLA_OK) return rc;
    return launch_status(cudaMemcpyAsync(status, scratch, sizeof(int), cudaMemcpyDefault,
                                         static_cast<cudaStream_t>(stream)));
}

int mla_decode_static_reset(void* stream) {
    void* scratch = nullptr;
    const int rc = static_scratch_for(stream, &scratch);
    if (rc != MLA_OK) return rc;
    return launch_status(cudaMemsetAsync(scratch, 0, sizeof(int), static_cast<cudaStream_t>(stream)));
}

int mla_decode_scratch_init(void* scratch, size_t scratch_bytes, void* stream) {
    if (!scratch || scratch_bytes == 0) return MLA_EINVAL;
    return launch_status(cudaMemsetAsync(scratch, 0, scratch_bytes, static_cast<cudaStream_t>(stream)));
}

const char* mla_decode_strerror(int status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_EINVAL: return "invalid argument (null pointer, bad shape, size or plan)";
        case MLA_EUNSUPPORTED: return "unsupported shape (needs d_latent 512, d_rope 64, heads 16/32/64/128)";
        case MLA_ESCRATCH: return "scratch missing, not 256-byte aligned, or smaller than plan scratch_bytes";
        case MLA_EALIGN: return "misaligned pointer or row stride";
        case MLA_ECUDA: return "CUDA runtime error";
        case MLA_EDEVICE: return "a kernel wait ran out of time (device status word set)";
        case MLA_ENOTREADY: return "kernels not prepared on this device; call mla_decode_plan before capture";
        case MLA_ESTATICLIMIT:
            return "plan scratch_bytes exceeds the 8 MiB static scratch of mla_decode_forward_static";
        default: return "unknown status";
    }
}

}  // extern "C"
