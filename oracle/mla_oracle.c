/*
 * mla_oracle.c -- plain fp64 CPU oracle for split-KV multi-head latent
 * attention (MLA) decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no source, header, constant or
 * helper with the CUDA library.
 *
 * What it computes (one query token per request, one output per head):
 *
 *   Attended row set R_b of request b
 *     dense : rows base_b + t for t = 0 .. d_pos[b]        (n_ctx = d_pos + 1)
 *     sparse: rows base_b + idx[b][j] for every list entry j with
 *             0 <= idx[b][j] < cache_len[b]                 (one term per entry)
 *   Score of row t for head h
 *     s_t = ( sum_i q_lat[h][i] * c[t][i] + sum_i q_rope[h][i] * k_rope[t][i] ) * scale
 *   Log-sum-exp (natural log) and normalised latent output
 *     lse    = m + ln sum_t exp(s_t - m),          m = max_t s_t
 *     out[f] = sum_t exp(s_t - lse) * c[t][f]      (value = latent c only)
 *   An empty row set gives lse = -inf and out = 0.
 *
 * Passages followed (page title, section):
 *   - "Graph-resident decode" (Lecture 08) s.2: the cache row of position p
 *     lives at cache + p * key_length, and the MLA kernels bound their loop
 *     by n_ctx = *d_pos + 1.
 *   - "Graph-resident decode" (Lecture 08) s.6: per-slice attention partials
 *     are merged into a normalised latent; the slice sum runs in ascending
 *     slice order.
 *   - "Launch Geometry" (Lecture 04) s.8: splitting attention over more
 *     context slices only re-associates the online-softmax combine.
 *   - "The Commit That Changed Direction": sparse MLA decode gathers the
 *     indexed rows of a large latent KV cache.
 *   The softmax((q_lat.c + q_rope.k_rope) * scale) . c formula itself is not
 *   written on the pages; it is the statement of the problem this oracle
 *   implements, with the row layout [c (d_latent) | k_rope (d_rope)].
 *
 * Arithmetic: every stored bf16 value is widened exactly to double; every
 * score, exponential and sum is formed in double with plain sequential
 * loops; the two-pass form (max, then sum) is used.
 *
 * FP8 cache ("Graph-resident decode" s.9 narrows the latent cache from F32
 * to F16 for bandwidth; this takes that one step further and is not on the
 * pages): the rows hold OCP FP8 E4M3 bytes and one scale for the whole
 * cache; the dequantisation step value = e4m3(byte) * kv_scale is done in
 * double before the definition above, which is otherwise unchanged (q
 * stays bf16).  The split emulation
 * computes per-slice partials and merges them exactly as a split-KV decode
 * does, still in double, to pin the combine algebra.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* Exact widening of a bf16 bit pattern: bf16 is the high half of a binary32. */
static double widen_bf16(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Value of an OCP FP8 E4M3 byte: sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits; exponent field 0 holds the subnormals m/8 * 2^-6; there are
 * no infinities, and S.1111.111 is NaN (so the largest finite value is
 * 1.75 * 2^8 = 448). */
static double widen_e4m3(uint8_t bits) {
    const int e = (bits >> 3) & 15, m = bits & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return (bits & 0x80) ? -v : v;
}

typedef struct {
    const uint16_t *q;          /* [B][H][d_latent + d_rope] */
    const void *kv;             /* rows of [d_latent + d_rope], row_stride apart: bf16, or E4M3 bytes */
    int kv_fp8;                 /* 1: the rows are E4M3 bytes, dequantised with kv_scale */
    double kv_scale;
    long long kv_rows;
    long long row_stride;       /* elements */
    int batch, heads, d_latent, d_rope;
    double scale;
    int sparse;
    const int *d_pos;           /* dense: [B] */
    const long long *row_offset;/* [B] or NULL (dense, batch 1: base 0) */
    const int *cache_len;       /* sparse: [B] */
    const int *indices;         /* sparse: [B][topk] */
    int topk;
    int splits;                 /* 0 = two-pass over all rows; >=1 = split emulation */
    int granule;                /* split slice size rounded up to a multiple of this */
    double *out;                /* [B][H][d_latent] */
    double *lse;                /* [B][H] */
    double *o_part;             /* optional [B][H][splits][d_latent] */
    double *lse_part;           /* optional [B][H][splits] */
    /* work distribution */
    long long next_item;
    pthread_mutex_t lock;
    int status;
} job_t;

/* Element i of cache row r, in double. */
static double kv_at(const job_t *J, long long r, int i) {
    if (J->kv_fp8) return widen_e4m3(((const uint8_t *)J->kv)[r * J->row_stride + i]) * J->kv_scale;
    return widen_bf16(((const uint16_t *)J->kv)[r * J->row_stride + i]);
}

/* Collect the attended absolute row ids of request b into rows[]; returns count. */
static long long attended_rows(const job_t *J, int b, long long *rows) {
    long long base = J->row_offset ? J->row_offset[b] : 0;
    long long n = 0;
    if (!J->sparse) {
        long long ctx = (long long)J->d_pos[b] + 1;
        for (long long t = 0; t < ctx; ++t) {
            long long r = base + t;
            if (r >= 0 && r < J->kv_rows) rows[n++] = r;
        }
    } else {
        const int *idx = J->indices + (long long)b * J->topk;
        for (int j = 0; j < J->topk; ++j) {
            int i = idx[j];
            if (i < 0 || i >= J->cache_len[b]) continue;
            long long r = base + i;
            if (r < 0 || r >= J->kv_rows) continue;
            rows[n++] = r;
        }
    }
    return n;
}

/* s_t for one head over the listed rows. */
static void scores(const job_t *J, int b, int h, const long long *rows, long long n, double *s) {
    const int D = J->d_latent + J->d_rope;
    const uint16_t *qh = J->q + ((long long)b * J->heads + h) * D;
    for (long long t = 0; t < n; ++t) {
        double lat = 0.0, rope = 0.0;
        for (int i = 0; i < J->d_latent; ++i) lat += widen_bf16(qh[i]) * kv_at(J, rows[t], i);
        for (int i = 0; i < J->d_rope; ++i)
            rope += widen_bf16(qh[J->d_latent + i]) * kv_at(J, rows[t], J->d_latent + i);
        s[t] = (lat + rope) * J->scale;
    }
}

/* Two-pass softmax-weighted average over rows[lo, hi): writes o (normalised) and lse. */
static void attend(const job_t *J, const long long *rows, const double *s, long long lo, long long hi,
                   double *o, double *lse_out) {
    const int F = J->d_latent;
    for (int f = 0; f < F; ++f) o[f] = 0.0;
    if (hi <= lo) { *lse_out = -INFINITY; return; }
    double m = -INFINITY;
    for (long long t = lo; t < hi; ++t) if (s[t] > m) m = s[t];
    double l = 0.0;
    for (long long t = lo; t < hi; ++t) l += exp(s[t] - m);
    double lse = m + log(l);
    for (long long t = lo; t < hi; ++t) {
        double w = exp(s[t] - lse);
        for (int f = 0; f < F; ++f) o[f] += w * kv_at(J, rows[t], f);
    }
    *lse_out = lse;
}

static void do_item(job_t *J, long long item, long long *rows, double *s, double *o_tmp) {
    int b = (int)(item / J->heads), h = (int)(item % J->heads);
    const int F = J->d_latent;
    long long n = attended_rows(J, b, rows);
    scores(J, b, h, rows, n, s);
    double *out = J->out + ((long long)b * J->heads + h) * F;
    double *lse = J->lse + (long long)b * J->heads + h;
    if (J->splits <= 0) { attend(J, rows, s, 0, n, out, lse); return; }

    /* Split emulation: the attended entries, in list order, are cut into
     * `splits` contiguous slices of ceil(n_entries / splits) entries rounded
     * up to `granule`; trailing slices may be empty.  For sparse requests the
     * slices cut the index list (masked entries included), as a split-KV
     * kernel walking the list would. */
    const int S = J->splits;
    long long n_entries = J->sparse ? J->topk : (long long)J->d_pos[b] + 1;
    long long per = (n_entries + S - 1) / S;
    if (J->granule > 1) per = (per + J->granule - 1) / J->granule * J->granule;
    double *lse_s = (double *)malloc(sizeof(double) * S);
    double *o_s = (double *)malloc(sizeof(double) * (size_t)S * F);
    if (!lse_s || !o_s) { free(lse_s); free(o_s); J->status = ORACLE_ENOMEM; return; }
    /* map list entries to positions in rows[] (masked entries are absent from rows[]) */
    long long pos = 0;
    for (int sp = 0; sp < S; ++sp) {
        long long e_lo = (long long)sp * per, e_hi = e_lo + per;
        if (e_lo > n_entries) e_lo = n_entries;
        if (e_hi > n_entries) e_hi = n_entries;
        long long cnt = 0;
        if (!J->sparse) {
            /* dense entries are rows base + t; masking only drops rows past kv_rows */
            long long base = J->row_offset ? J->row_offset[b] : 0;
            for (long long e = e_lo; e < e_hi; ++e) if (base + e >= 0 && base + e < J->kv_rows) ++cnt;
        } else {
            const int *idx = J->indices + (long long)b * J->topk;
            long long base = J->row_offset ? J->row_offset[b] : 0;
            for (long long e = e_lo; e < e_hi; ++e) {
                int i = idx[e];
                if (i < 0 || i >= J->cache_len[b]) continue;
                if (base + i < 0 || base + i >= J->kv_rows) continue;
                ++cnt;
            }
        }
        attend(J, rows, s, pos, pos + cnt, o_s + (size_t)sp * F, lse_s + sp);
        pos += cnt;
    }
    /* merge: M = max lse_s, lse = M + ln sum exp(lse_s - M), out = sum_s exp(lse_s - lse) o_s */
    double M = -INFINITY;
    for (int sp = 0; sp < S; ++sp) if (lse_s[sp] > M) M = lse_s[sp];
    for (int f = 0; f < F; ++f) out[f] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
    } else {
        double L = 0.0;
        for (int sp = 0; sp < S; ++sp) L += exp(lse_s[sp] - M);
        double tot = M + log(L);
        for (int sp = 0; sp < S; ++sp) {
            double w = exp(lse_s[sp] - tot);
            for (int f = 0; f < F; ++f) out[f] += w * o_s[(size_t)sp * F + f];
        }
        *lse = tot;
    }
    if (J->o_part) memcpy(J->o_part + (size_t)item * S * F, o_s, sizeof(double) * (size_t)S * F);
    if (J->lse_part) memcpy(J->lse_part + (size_t)item * S, lse_s, sizeof(double) * S);
    (void)o_tmp;
    free(lse_s);
    free(o_s);
}

static long long max_entries(const job_t *J) {
    long long mx = 1;
    for (int b = 0; b < J->batch; ++b) {
        long long e = J->sparse ? J->topk : (long long)J->d_pos[b] + 1;
        if (e > mx) mx = e;
    }
    return mx;
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    long long cap = max_entries(J);
    long long *rows = (long long *)malloc(sizeof(long long) * cap);
    double *s = (double *)malloc(sizeof(double) * cap);
    if (!rows || !s) {
        pthread_mutex_lock(&J->lock); J->status = ORACLE_ENOMEM; pthread_mutex_unlock(&J->lock);
        free(rows); free(s); return NULL;
    }
    const long long total = (long long)J->batch * J->heads;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        long long item = J->next_item++;
        pthread_mutex_unlock(&J->lock);
        if (item >= total) break;
        do_item(J, item, rows, s, NULL);
    }
    free(rows);
    free(s);
    return NULL;
}

static int run_job(job_t *J, int n_threads) {
    if (!J->q || !J->kv || !J->out || !J->lse) return ORACLE_EINVAL;
    if (J->batch < 1 || J->heads < 1 || J->d_latent < 1 || J->d_rope < 0) return ORACLE_EINVAL;
    if (J->row_stride < J->d_latent + J->d_rope || J->kv_rows < 0) return ORACLE_EINVAL;
    if (!J->sparse && !J->d_pos) return ORACLE_EINVAL;
    if (J->sparse && (!J->indices || !J->cache_len || !J->row_offset || J->topk < 1)) return ORACLE_EINVAL;
    if (!J->sparse) for (int b = 0; b < J->batch; ++b) if (J->d_pos[b] < 0) return ORACLE_EINVAL;
    if (n_threads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = n > 0 ? (int)n : 1;
    }
    long long total = (long long)J->batch * J->heads;
    if (n_threads > total) n_threads = (int)total;
    J->next_item = 0;
    J->status = ORACLE_OK;
    pthread_mutex_init(&J->lock, NULL);
    if (n_threads == 1) {
        worker(J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * n_threads);
        if (!th) { pthread_mutex_destroy(&J->lock); return ORACLE_ENOMEM; }
        int started = 0;
        for (int i = 0; i < n_threads; ++i)
            if (pthread_create(&th[i], NULL, worker, J) == 0) ++started;
        if (started == 0) worker(J);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J->lock);
    return J->status;
}

/* Two-pass fp64 reference.  See the file header for the definition. */
int oracle_mla_decode_f64(const uint16_t *q, const uint16_t *kv, long long kv_rows, long long row_stride,
                          int batch, int heads, int d_latent, int d_rope, double scale, int sparse,
                          const int *d_pos, const long long *row_offset, const int *cache_len,
                          const int *indices, int topk, double *out, double *lse, int n_threads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.kv = kv; J.kv_rows = kv_rows; J.row_stride = row_stride;
    J.batch = batch; J.heads = heads; J.d_latent = d_latent; J.d_rope = d_rope;
    J.scale = scale; J.sparse = sparse; J.d_pos = d_pos; J.row_offset = row_offset;
    J.cache_len = cache_len; J.indices = indices; J.topk = topk;
    J.splits = 0; J.granule = 1; J.out = out; J.lse = lse;
    return run_job(&J, n_threads);
}

/* Split emulation: per-slice partials (normalised o_s and lse_s) merged by
 * the log-sum-exp combine.  o_part / lse_part may be NULL. */
int oracle_mla_decode_split_f64(const uint16_t *q, const uint16_t *kv, long long kv_rows, long long row_stride,
                                int batch, int heads, int d_latent, int d_rope, double scale, int sparse,
                                const int *d_pos, const long long *row_offset, const int *cache_len,
                                const int *indices, int topk, int splits, int granule,
                                double *out, double *lse, double *o_part, double *lse_part, int n_threads) {
    if (splits < 1) return ORACLE_EINVAL;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.kv = kv; J.kv_rows = kv_rows; J.row_stride = row_stride;
    J.batch = batch; J.heads = heads; J.d_latent = d_latent; J.d_rope = d_rope;
    J.scale = scale; J.sparse = sparse; J.d_pos = d_pos; J.row_offset = row_offset;
    J.cache_len = cache_len; J.indices = indices; J.topk = topk;
    J.splits = splits; J.granule = granule < 1 ? 1 : granule;
    J.out = out; J.lse = lse; J.o_part = o_part; J.lse_part = lse_part;
    return run_job(&J, n_threads);
}

/* The two-pass reference (or, with splits >= 1, the split emulation) over an
 * E4M3 cache with one scale: kv holds bytes, row_stride in bytes (elements). */
int oracle_mla_decode_e4m3_f64(const uint16_t *q, const uint8_t *kv, double kv_scale, long long kv_rows,
                               long long row_stride, int batch, int heads, int d_latent, int d_rope, double scale,
                               int sparse, const int *d_pos, const long long *row_offset, const int *cache_len,
                               const int *indices, int topk, int splits, int granule, double *out, double *lse,
                               double *o_part, double *lse_part, int n_threads) {
    if (splits < 0 || !(kv_scale > 0.0) || !isfinite(kv_scale)) return ORACLE_EINVAL;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.kv = kv; J.kv_fp8 = 1; J.kv_scale = kv_scale; J.kv_rows = kv_rows; J.row_stride = row_stride;
    J.batch = batch; J.heads = heads; J.d_latent = d_latent; J.d_rope = d_rope;
    J.scale = scale; J.sparse = sparse; J.d_pos = d_pos; J.row_offset = row_offset;
    J.cache_len = cache_len; J.indices = indices; J.topk = topk;
    J.splits = splits; J.granule = granule < 1 ? 1 : granule;
    J.out = out; J.lse = lse; J.o_part = o_part; J.lse_part = lse_part;
    return run_job(&J, n_threads);
}

/* Values of n E4M3 bytes (the dequantisation step with scale 1). */
int oracle_e4m3_to_f64(const uint8_t *in, long long n, double *out) {
    if ((!in || !out) && n > 0) return ORACLE_EINVAL;
    for (long long i = 0; i < n; ++i) out[i] = widen_e4m3(in[i]);
    return 0;
}

/* Projection of a merged latent through wv_b, per head ("Graph-resident
 * decode", Lecture 08, s.6: the merged latent is projected through wv_b by a
 * second kernel):
 *   y[b][h][v] = sum_{r < d_latent} latent[b][h][r] * wv_b[h][v][r]
 * latent fp64 [B][H][d_latent]; wv_b bf16 [H][v_dim][d_latent], widened
 * exactly; the sum runs r ascending in double. */
int oracle_mla_project_f64(const double *latent, const uint16_t *wv_b, int batch, int heads, int d_latent,
                           int v_dim, double *y) {
    if (!latent || !wv_b || !y || batch < 0 || heads < 1 || d_latent < 1 || v_dim < 1) return ORACLE_EINVAL;
    for (int b = 0; b < batch; ++b)
        for (int h = 0; h < heads; ++h) {
            const double *lat = latent + ((long long)b * heads + h) * d_latent;
            for (int v = 0; v < v_dim; ++v) {
                const uint16_t *w = wv_b + ((long long)h * v_dim + v) * d_latent;
                double acc = 0.0;
                for (int r = 0; r < d_latent; ++r) acc += lat[r] * widen_bf16(w[r]);
                y[((long long)b * heads + h) * v_dim + v] = acc;
            }
        }
    return 0;
}

int oracle_hardware_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
