// mla_internal.h -- parameters shared between the C-ABI host code and the
// kernel translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mla {

constexpr int kDLatent = 512;
constexpr int kDRope = 64;
constexpr int kDRow = kDLatent + kDRope;       // 576 bf16 per cache row
constexpr int kRowBytes = kDRow * 2;           // 1152
constexpr int kStageRows = 32;                 // rows per pipeline stage (warp-MMA partial kernel)
constexpr int kTcTileRows = 80;                // rows per tile (tcgen05 partial kernel, 16 heads per CTA)
constexpr int kTcTileRows32 = 64;              // rows per tile (tcgen05 partial kernel, 32 heads per CTA)
constexpr int kTcGranule = 16;                 // slice granule of the tcgen05 kernel (one MMA k-step)
constexpr int kHeadGroup = 16;                 // heads per CTA (warp-MMA kernel; tcgen05 kernel: 16 or 32)
constexpr int kCombineChunk = 128;             // features per combine CTA
// Size of the library's own scratch array used by mla_decode_forward_static
// (8 MiB: the status word, B*H*S partial rows of 2 KiB and B*H*S lse values,
// each region 256-byte aligned; e.g. B = 1, H = 16 up to S = 255).
constexpr size_t kStaticScratchBytes = size_t(8) << 20;

// Everything the split partial kernel needs; passed by value.
struct PartialParams {
    const uint16_t* q;          // bf16 [B][H][576]
    const uint16_t* kv;         // bf16 rows
    long long kv_rows;
    long long row_stride;       // elements
    const int* d_pos;           // dense [B]
    const long long* row_offset;// [B] or null (dense, B == 1)
    const int* cache_len;       // sparse [B]
    const int* indices;         // sparse [B][topk]
    int batch, heads, topk, splits, sparse;
    int n_groups;               // heads / head group
    int granule;                // slices are whole multiples of this many entries
    int n_items;                // batch * n_groups * splits work items, walked round-robin by the CTAs
                                // (flat split: 2 * flat_ranges * n_groups)
    // Flat split (batched sparse decode, warp-MMA kernel): the B * topk list
    // entries are cut into flat_ranges contiguous ranges of flat_per entries
    // (a multiple of 32, at most topk), one per CTA and head group; a range
    // holds pieces of at most two requests (two items), and request b's piece
    // in range r is its slice r - floor(b * topk / flat_per).  0 = the uniform
    // split of every request into `splits` slices.
    int flat_ranges;
    int flat_per;
    float scale_log2;           // scale * log2(e): scores are kept in base-2 units
    float* o_part;              // [B][H][S][512]
    float* lse_part;            // [B][H][S]
    int* status;                // status word
    int stall_test;             // test hook: run the timeout path (see mla_decode_shape)
    // fused append (dense): bf16 [B][576], row b taking the place of cache row
    // d_pos[b] of request b in the CTA's staged tile; null = read the cache only
    const uint16_t* new_rows;
    // E4M3 cache (dense, warp-MMA kernel): kv holds bytes and every value is
    // e4m3(byte) * v_scale; scale_log2 already carries v_scale, and the partial
    // multiplies O by it.  v_scale = 1 for bf16 caches.
    int kv_fp8;
    float v_scale;
    // dense bf16 cache on the warp-MMA kernel: 1 = P . V on the tcgen05 tensor
    // cores (O in tensor memory), 0 = P . V on the warps (mma.sync)
    int tc_pv;
};

struct CombineParams {
    const float* o_part;
    const float* lse_part;
    const int* status;
    float* out;                 // [B][H][512]
    float* lse;                 // [B][H]
    int batch, heads, splits;
    int sparse, topk;           // with d_pos / row_offset / kv_rows: which slices hold entries
    int granule;
    const int* d_pos;
    const long long* row_offset;
    long long kv_rows;
    // fused state update after the merge (dense): new_rows[b] written to cache
    // row d_pos[b] of request b (rows outside [0, kv_rows) are not written),
    // then d_pos[b] += 1 when advance is set; new_rows null = neither
    const uint16_t* new_rows;
    uint16_t* kv;
    long long row_stride;
    int* d_pos_rw;
    int advance;
};

struct ProjectParams {
    const float* latent;        // fp32 [B][H][512] (the merged, normalised latent)
    const uint16_t* wv_b;       // bf16 [H][v_dim][512]
    float* y;                   // fp32 [B][H][v_dim]
    int batch, heads, v_dim;
};

struct AppendParams {
    uint16_t* kv;
    long long kv_rows;
    long long row_stride;
    const uint16_t* new_rows;   // [B][576]
    const int* d_pos;
    const long long* row_offset;
    int batch;
};

// TMA descriptors of the tcgen05 kernel, both rank 3 with the 128-byte
// swizzle: dimension 0 = 64 bf16 of a row (128 bytes), dimension 1 = rows
// (stride: the row stride), dimension 2 = the 9 column chunks of a row
// (stride 128 bytes).  One box lands as [chunk][row][64 bf16], the layout the
// tensor cores read.  kv: boxes of 64 x tile rows x 3 chunks (a third of a
// tile; one-chunk boxes, nine barriers per tile, measured slower); q: boxes
// of 64 x head-group rows x 9 chunks (the whole query tile).
constexpr int kTcBoxChunks = 3;
// The warp-MMA kernel uses the same query map (its cache map is unused).
struct TcMaps {
    CUtensorMap kv;
    CUtensorMap q;
};

// Launch helpers (each returns the cudaError_t of the launch).
cudaError_t partial_mma_prepare(int device);
size_t partial_mma_smem_bytes(bool fp8 = false, bool tc_pv = false);
int partial_mma_block_threads();
cudaError_t partial_mma_occupancy(int* ctas_per_sm);
cudaError_t launch_partial_mma(const TcMaps& maps, const PartialParams& p, dim3 grid, bool pdl, cudaStream_t stream);
cudaError_t partial_tc_prepare(int device);
size_t partial_tc_smem_bytes(int head_group);
int partial_tc_block_threads(int head_group);
cudaError_t launch_partial_tc(const TcMaps& maps, const PartialParams& p, int head_group, dim3 grid, bool pdl,
                              cudaStream_t stream);
int combine_block_threads();
int combine_grid_rows(int rows, int splits);    // combine grid x for B*H rows
cudaError_t combine_prepare();
cudaError_t launch_project(const ProjectParams& p, bool pdl, cudaStream_t stream);
// spread: one CTA per SM (for grids no larger than the SM count)
cudaError_t launch_combine(const CombineParams& p, dim3 grid, int block, bool pdl, bool spread,
                           cudaStream_t stream);

// Static scratch (mla_static_scratch.cu): its address on `device` once set up
// there (nullptr before), and the one-time set-up with `device` current.
void* static_scratch_if_ready(int device);
cudaError_t static_scratch_set_up(int device, void** out);
cudaError_t launch_append(const AppendParams& p, bool pdl, cudaStream_t stream);
cudaError_t launch_advance(int* d_pos, int batch, bool pdl, cudaStream_t stream);

}  // namespace mla
