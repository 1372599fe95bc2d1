/*
 * mla_decode.h -- C ABI of libmla_decode.so: split-KV multi-head latent
 * attention (MLA) decode on one GB300 (sm_103a).
 *
 * One query token per request attends over a latent KV cache whose rows are
 * [c (512 bf16) | k_rope (64 bf16)] = 576 bf16 = 1152 bytes.  For request b
 * and head h over the attended rows R_b:
 *
 *     s_t    = (q_lat[h] . c_t + q_rope[h] . k_rope_t) * scale
 *     lse    = ln sum_t exp(s_t)                           (natural log)
 *     out[f] = sum_t exp(s_t - lse) * c_t[f]               (normalised latent)
 *
 * Dense : R_b = rows base_b + 0 .. base_b + d_pos[b]; the context bound
 *         n_ctx = d_pos[b] + 1 is read from device memory by the kernels
 *         ("Graph-resident decode", Lecture 08, s.2: the MLA kernels read
 *         *d_pos + 1 as their loop bound, so a captured graph stays valid as
 *         the position advances).
 * Sparse: R_b = rows base_b + indices[b][j] for each list entry j with
 *         0 <= indices[b][j] < cache_len[b] ("The Commit That Changed
 *         Direction": split-KV sparse MLA decode gathers scattered rows of a
 *         large cache).  Out-of-range entries are skipped.
 *
 * The context (or index list) is cut into `splits` slices; a partial kernel
 * computes each (head group, slice) online-softmax partial and a separate
 * combine kernel merges them with a log-sum-exp weighting, slices summed in
 * ascending order ("Graph-resident decode", Lecture 08, s.6; "Launch
 * Geometry", Lecture 04, s.8).  The split count and the grid are derived from
 * the SM count and the context length by mla_decode_plan ("Launch Geometry",
 * Lecture 04, s.4: derive the slice floor, name the blocks-per-SM target).
 *
 * Conventions for every call:
 *   - Pointers marked (device) are CUDA device pointers owned by the caller;
 *     the library never allocates, frees or synchronises, and keeps no state
 *     other than a per-device cache of the SM count and of kernel attributes.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Launches are
 *     asynchronous and legal inside stream capture once mla_decode_plan has
 *     been called on the device (it prepares the kernels; "Graph-resident
 *     decode", Lecture 08, s.3: pre-warm lazy initialisation before capture).
 *   - Every call returns an mla_status; arguments are checked on the host
 *     before anything is launched.  Nothing throws across the ABI.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_DECODE_ABI_VERSION 4
#define MLA_D_LATENT 512
#define MLA_D_ROPE 64
#define MLA_D_ROW 576        /* elements per cache row */
#define MLA_MAX_SPLITS 256   /* largest split count a plan may hold */

typedef enum {
    MLA_OK = 0,
    MLA_EINVAL = -1,        /* null pointer, bad shape, size or plan */
    MLA_EUNSUPPORTED = -2,  /* shape the kernels do not implement (d_c != 512, d_r != 64, H,
                               or a dense cache of 2^31 rows or more: TMA row coordinates
                               are 32-bit) */
    MLA_ESCRATCH = -3,      /* scratch missing, misaligned or smaller than plan->scratch_bytes */
    MLA_EALIGN = -4,        /* q, kv, out or lse misaligned, or row stride not a multiple of 8 (16 bytes for E4M3) */
    MLA_ECUDA = -5,         /* the CUDA runtime reported an error for a launch or query */
    MLA_EDEVICE = -6,       /* a kernel's bounded wait ran out (see the scratch status word) */
    MLA_ENOTREADY = -7,     /* kernels not prepared on this device and the stream is capturing */
    MLA_ESTATICLIMIT = -8   /* plan->scratch_bytes > MLA_STATIC_SCRATCH_BYTES (forward_static) */
} mla_status;

/* Problem description given to the planner. */
typedef struct {
    int batch;            /* B >= 1 requests, one query token each */
    int heads;            /* H in {16, 32, 64, 128} */
    int d_latent;         /* must be 512 */
    int d_rope;           /* must be 64 */
    int sparse;           /* 0 = dense context, 1 = top-k index gather */
    int max_ctx;          /* dense: largest n_ctx = d_pos + 1 any request reaches (>= 1) */
    int topk;             /* sparse: index-list length per request (>= 1) */
    float scale;          /* softmax scale, finite and > 0 (1/sqrt(576) for these shapes) */
    int num_sms;          /* SMs to plan for; 0 = query the current device */
    int splits_override;  /* 0 = derive; 1..MLA_MAX_SPLITS = force this split count */
    int variant;          /* 1 = warp-MMA (mma.sync) kernel, 64-row steps, 16 heads per CTA;
                             2 = tcgen05/TMEM kernel, 80-row TMA tiles, 16 heads per CTA;
                             3 = tcgen05/TMEM kernel, 64-row tiles, 32 heads per CTA (dense,
                                 heads a multiple of 32);
                             4 = tcgen05/TMEM kernel, 64-row tiles, 64 heads per CTA (dense,
                                 heads a multiple of 64);
                             5 = the warp-MMA kernel with P . V on tcgen05: scores and softmax
                                 on the warps (mma.sync), P . V issued by one thread per warp
                                 group into tensor memory (dense only);
                             0 = auto (measured crossovers): E4M3 cache -> 5; sparse or H = 16
                                 -> 1; dense H >= 32 -> 1 while its slices hold <= 768 rows,
                                 else 4 (H a multiple of 64) or 3 */
    int pdl;              /* 1 = launch with programmatic dependent launch */
    int stall_test;       /* test hook, 0 in normal use.  1 = one thread of the partial kernel
                             waits (about 1 ms) on a barrier nothing arrives at, so the timeout
                             path runs for real: the CTA aborts, drains its copies and MMAs,
                             frees its tensor memory and leaves MLA_EDEVICE in the status word;
                             the outputs of that call are undefined, the context stays usable */
    int kv_fp8;           /* 0 = bf16 cache rows (576 x 2 bytes); 1 = OCP FP8 E4M3 cache rows (576
                             bytes), value = e4m3(byte) * args.kv_scale: dense decode on the
                             warp-MMA kernel (variant 0, 1 or 5; otherwise MLA_EUNSUPPORTED) */
} mla_decode_shape;

/* Launch plan (plain data; copy freely).  The plan is the capture key of a
 * graph: a graph stays valid as long as the plan it was captured with does
 * ("Graph-resident decode", Lecture 08, s.2: splits sizes the grid, so it is
 * decided on the host by the same function the launcher uses).  Every launch
 * re-derives the grids and the scratch layout from the shape and the split
 * count and rejects a plan that differs (MLA_EINVAL): edit a plan only through
 * mla_decode_plan. */
typedef struct {
    mla_decode_shape shape;
    int magic;                 /* set by mla_decode_plan; checked by every launch */
    int variant;               /* kernel chosen */
    int splits;                /* S: slices per (request, head group) = work items per pair */
    int entries_per_split;     /* rows (dense) or list entries (sparse) per slice at max_ctx / topk */
    int head_group;            /* heads per CTA */
    int n_head_groups;         /* H / head_group */
    int ctas_per_sm;           /* resident CTAs per SM of the partial kernel (persistent: 1) */
    int num_sms;               /* SM count planned for */
    int grid_x, grid_y, grid_z, block, smem_bytes;          /* partial kernel launch */
    int combine_grid_x, combine_grid_y, combine_block;      /* combine kernel launch */
    size_t scratch_bytes;      /* bytes of caller scratch needed by run + combine */
    size_t o_part_offset;      /* fp32 [B][H][S][512] normalised slice outputs */
    size_t lse_part_offset;    /* fp32 [B][H][S] slice log-sum-exp (-inf for an empty slice) */
    size_t status_offset;      /* int32 status word: 0 healthy, else an mla_status */
    int flat_ranges;           /* 0: every request cut into `splits` slices of entries_per_split entries.
                                  > 0 (batched sparse decode, chosen when the cost model prefers it):
                                  the B * topk list entries, request after request, cut into
                                  flat_ranges ranges of entries_per_split entries, one CTA per range
                                  and head group, so no SM idles when B * S slices would not fill
                                  the GPU; a range holds pieces of at most two requests, and
                                  `splits` = the most pieces any request has (the merge reads that
                                  many slices per request, missing ones written empty) */
} mla_decode_plan_t;

/* Per-call tensors. */
typedef struct {
    const void *q;               /* (device) bf16 [B][H][576] = [q_lat | q_rope], 16-byte aligned */
    const void *kv;              /* (device) bf16 cache rows, row r at kv + r * row_stride, 16-byte aligned */
    long long kv_rows;           /* rows addressable in kv (bounds for every row the kernels read) */
    long long row_stride;        /* elements between rows: >= 576 and a multiple of 8 */
    const int *d_pos;            /* (device) dense: int32 [B]; n_ctx of request b = d_pos[b] + 1 */
    const long long *row_offset; /* (device) int64 [B]: first row of request b's segment;
                                    may be NULL for a dense batch of 1 (segment starts at row 0) */
    const int *cache_len;        /* (device) sparse: int32 [B] rows in request b's segment */
    const int *indices;          /* (device) sparse: int32 [B][topk] request-local row ids */
    float *out;                  /* (device) fp32 [B][H][512], 16-byte aligned */
    float *lse;                  /* (device) fp32 [B][H], natural log; -inf if no row is attended */
    float kv_scale;              /* E4M3 caches (shape.kv_fp8 = 1): the cache's one scale, finite and > 0;
                                    kv then holds bytes, row_stride counts bytes (>= 576, a multiple
                                    of 16); ignored for bf16 caches */
} mla_decode_args;

/* Version of this ABI (MLA_DECODE_ABI_VERSION). */
MLA_API int mla_decode_abi_version(void);

/* Plan a decode: validates the shape, derives the split count and fills the
 * launch geometry and scratch layout.  The partial kernel runs a persistent
 * grid of min(items, num_sms) CTAs (one per SM) that walk the
 * B * n_head_groups * S work items round-robin; S is the split count that
 * minimises the modelled time ceil(items / grid) * (tiles per slice + 1),
 * a tile being the kernel's row step (80 or 64 rows for tcgen05; for warp-MMA
 * its 32-row slot, two of which make one 64-row step)
 * and the +1 the item's partial write, the smallest such S on ties; slices
 * are whole multiples of 16 (tcgen05) or 32 (warp-MMA) rows and
 * S <= MLA_MAX_SPLITS.  With num_sms == 0 it queries the
 * current device and prepares the kernels there (call it before capturing a
 * graph).  Host only; the plan does not depend on any device pointer.
 * ("Launch Geometry", Lecture 04, s.1 and s.4; "Graph-resident decode",
 * Lecture 08, s.2.)  Errors: MLA_EINVAL (null or bad field),
 * MLA_EUNSUPPORTED (shape), MLA_ECUDA (device query failed). */
MLA_API int mla_decode_plan(const mla_decode_shape *shape, mla_decode_plan_t *plan);

/* Launch the split partial kernel: each CTA computes one (request, head group,
 * slice) online-softmax partial into scratch (o_part normalised, lse_part).
 * `scratch` (device) must be 256-byte aligned and at least
 * plan->scratch_bytes long; the caller zeroes it once before first use (see
 * mla_decode_scratch_init) and must not reuse it for an overlapping call.
 * Errors: MLA_EINVAL, MLA_EALIGN, MLA_ESCRATCH, MLA_ENOTREADY, MLA_ECUDA. */
MLA_API int mla_decode_run(const mla_decode_plan_t *plan, const mla_decode_args *args, void *scratch,
                   size_t scratch_bytes, void *stream);

/* Launch the log-sum-exp combine: M = max_s lse_s, lse = M + ln sum_s
 * exp(lse_s - M), out = sum_s exp(lse_s - lse) * o_s with s ascending, for
 * every (request, head), over a (B*H, 512/128) grid of 256-thread CTAs ("Graph-resident decode",
 * Lecture 08, s.6: a merge grid wider than n_head, no serial prologue).
 * Must follow mla_decode_run on the same stream with the same plan and
 * scratch.  Errors as mla_decode_run. */
MLA_API int mla_decode_combine(const mla_decode_plan_t *plan, const mla_decode_args *args, const void *scratch,
                       size_t scratch_bytes, void *stream);

/* mla_decode_run followed by mla_decode_combine (two launches). */
MLA_API int mla_decode_forward(const mla_decode_plan_t *plan, const mla_decode_args *args, void *scratch,
                       size_t scratch_bytes, void *stream);

/* One dense decode step with the cache append and the position advance folded
 * into the two kernels ("Graph-resident decode", Lecture 08, s.2: append,
 * attention and the increment inside the captured region; fewer graph nodes
 * per step).  Same results, bit for bit, as
 *   mla_decode_append(kv, .., new_rows, d_pos, ..); mla_decode_forward(..);
 *   if (advance) mla_decode_advance(d_pos, ..);
 * in two launches instead of three or four: the partial kernel's CTA whose
 * slice holds row d_pos[b] of request b takes that row from new_rows[b]
 * (after its tile lands, in shared memory), and after the merge the combine
 * kernel writes new_rows[b] to cache row row_offset[b] + d_pos[b] (rows
 * outside [0, kv_rows) are neither written nor attended, as with the append)
 * and, if advance = 1, increments d_pos[b].  new_rows: (device) bf16 [B][576],
 * 16-byte aligned, read during the call.  Unlike mla_decode_run, this call
 * writes args->kv (one row per request) and args->d_pos (when advancing): both
 * must be writable device memory that no other work on other streams touches
 * meanwhile.  Dense plans only (MLA_EUNSUPPORTED for sparse).  advance: 0 or 1
 * (with several caches sharing one position, e.g. the layers of a model, pass
 * 1 only for the last).  Errors: as mla_decode_forward, and MLA_EINVAL (null
 * new_rows, advance not 0/1), MLA_EALIGN (new_rows), MLA_EUNSUPPORTED. */
MLA_API int mla_decode_forward_step(const mla_decode_plan_t *plan, const mla_decode_args *args, void *scratch,
                                    size_t scratch_bytes, const void *new_rows, int advance, void *stream);

/* Size of the library's own scratch array used by mla_decode_forward_static. */
#define MLA_STATIC_SCRATCH_BYTES (8u << 20)

/* mla_decode_forward without a caller scratch buffer and without allocating.
 * The pages that define the method have no counterpart of this call: it
 * exists for callers that may not allocate device memory (code running under
 * an allocator it does not own, e.g. inside another framework's memory pool
 * or a plug-in with a fixed memory budget, has no scratch buffer to pass).
 * The partial and combine kernels run exactly as in mla_decode_forward (same
 * plan, same results bit for bit), but their scratch is an 8 MiB
 * (MLA_STATIC_SCRATCH_BYTES) file-scope __device__ array of the library, one
 * per device context; the call makes no cudaMalloc/cudaFree or other
 * allocating call.
 *   - Set-up: the first call on a device looks the array's address up
 *     (cudaGetSymbolAddress, with that device current, its return code
 *     checked) and keeps it with the id of the current CUDA context; make that
 *     first call before any stream capture (a first call on a capturing stream
 *     returns MLA_ENOTREADY).  A call made in another context than the one of
 *     the lookup (e.g. after cudaDeviceReset, which ends the primary context
 *     and with it the array) looks the address up again, so it too must be
 *     made outside capture.
 *   - Size: a plan whose scratch_bytes exceeds MLA_STATIC_SCRATCH_BYTES is
 *     rejected with MLA_ESTATICLIMIT before anything is launched; use
 *     mla_decode_forward with a caller buffer for such plans.  scratch_bytes
 *     is 256 + align256(B*H*S*2048) + align256(B*H*S*4): e.g. B = 1, H = 16
 *     fits up to S = 255, H = 128 up to S = 31.
 *   - Zero start: only the status word (offset 0) must start at zero; the
 *     array is zero when the library's module is loaded.  A device-side
 *     wait timeout sets it (MLA_EDEVICE) and it stays set until
 *     mla_decode_static_reset; mla_decode_static_status reads it.  The
 *     partial and LSE arrays need no initial value.
 *   - Races: every call on a device shares the one array, so calls that can
 *     overlap (on different streams, or from several host threads without
 *     ordering) race on it and give wrong results; calls on one stream are
 *     ordered and safe.
 * Errors: as mla_decode_forward, minus MLA_ESCRATCH, plus MLA_ESTATICLIMIT. */
MLA_API int mla_decode_forward_static(const mla_decode_plan_t *plan, const mla_decode_args *args, void *stream);

/* The static array's status word (0 healthy, else an mla_status such as
 * MLA_EDEVICE after a wait timeout), for the current device: a stream-ordered
 * copy of the 4-byte word into *status, which may be device memory or
 * host memory the device can write (pinned or managed), 4-byte aligned; read
 * it after `stream` has reached this point.  Like mla_decode_forward_static,
 * the first use on a device looks the array up and must be outside stream
 * capture (MLA_ENOTREADY otherwise); nothing is allocated.
 * Errors: MLA_EINVAL (null status), MLA_EALIGN, MLA_ENOTREADY, MLA_ECUDA. */
MLA_API int mla_decode_static_status(int *status, void *stream);

/* Clear the static array's status word on the current device (a
 * stream-ordered 4-byte memset), so that a later timeout can be told apart
 * from an earlier one.  Same first-use rule as mla_decode_static_status.
 * Errors: MLA_ENOTREADY, MLA_ECUDA. */
MLA_API int mla_decode_static_reset(void *stream);

/* Write the new token's cache row from device memory: for each request b,
 * copy new_rows[b] (bf16 [576]) to row base_b + d_pos[b] of kv, where base_b
 * = row_offset[b] (row_offset may be NULL for batch 1).  The destination is
 * computed on the device so a captured graph writes a new row on every replay
 * ("Graph-resident decode", Lecture 08, s.2: the K-cache row write derives
 * the row from a device-resident d_pos and moves the same bytes).  Rows
 * outside [0, kv_rows) are not written.  kv and new_rows 16-byte aligned.
 * Errors: MLA_EINVAL, MLA_EALIGN, MLA_ECUDA. */
MLA_API int mla_decode_append(void *kv, long long kv_rows, long long row_stride, const void *new_rows,
                      const int *d_pos, const long long *row_offset, int batch, void *stream);

/* d_pos[b] += 1 for b < batch, on the device ("Graph-resident decode",
 * Lecture 08, s.2: the position increment runs inside the captured region).
 * Errors: MLA_EINVAL, MLA_ECUDA. */
MLA_API int mla_decode_advance(int *d_pos, int batch, void *stream);

/* Project the merged latent through wv_b, per head:
 *   y[b][h][v] = sum_{r < 512} latent[b][h][r] * wv_b[h][v][r]
 * ("Graph-resident decode", Lecture 08, s.6: after the merge writes the
 * normalised latent, a second kernel with grid (n_head, 16) projects it,
 * each block owning a slice of v_dim and reading only its own wv_b rows; the
 * dot strides r by 32 across the warp).  latent: (device) fp32 [B][H][512],
 * e.g. mla_decode_combine's out; wv_b: (device) bf16 [H][v_dim][512], row v
 * of head h contiguous over r; y: (device) fp32 [B][H][v_dim].  All three
 * 16-byte aligned, owned by the caller, not retained.  v_dim a multiple of 16
 * in [16, 512]; 1 <= heads <= 128; 1 <= batch <= 65535.  fp32 arithmetic in a
 * fixed order (bit-identical across runs).  pdl = 1 launches with
 * programmatic dependent launch (the kernel waits on the preceding one before
 * reading latent).  Async on `stream`, capture-safe.  Errors: MLA_EINVAL (null
 * pointer, batch, pdl), MLA_EUNSUPPORTED (heads, v_dim), MLA_EALIGN,
 * MLA_ECUDA. */
MLA_API int mla_decode_project(const float *latent, const void *wv_b, int batch, int heads, int v_dim, float *y,
                               int pdl, void *stream);

/* Zero the scratch region (async memset on `stream`), clearing the status
 * word.  Errors: MLA_EINVAL, MLA_ECUDA. */
MLA_API int mla_decode_scratch_init(void *scratch, size_t scratch_bytes, void *stream);

/* Static description of a status code. */
MLA_API const char *mla_decode_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
