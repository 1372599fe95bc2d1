/*
 * mla_floor.h -- floor probes of libmla_decode.so: what a decode call costs
 * with no decode work in it.
 *
 * A dense decode call is two kernels chained by programmatic dependent launch
 * (the split partial kernel and the log-sum-exp combine, "Graph-resident
 * decode", Lecture 08, s.6 and s.7) that stream the cache once (or gather
 * its indexed rows, "The Commit That Changed Direction").  The probes below
 * measure the parts of that call no kernel body can remove: two kernels with
 * empty bodies launched with the partial and combine kernels' launch shapes,
 * one kernel that does nothing but read a region of device memory over the
 * whole GPU, and one that does nothing but gather listed rows.  They compute
 * nothing of the method.
 *
 * Conventions as in mla_decode.h: (device) pointers are owned by the caller,
 * nothing is allocated, freed or synchronised, arguments are checked on the
 * host before anything is launched, and every call returns an mla_status.
 * The first call on a device sets the kernels' shared-memory limits; make it
 * outside stream capture (a first call on a capturing stream returns
 * MLA_ENOTREADY).
 */
#ifndef MLA_FLOOR_H_
#define MLA_FLOOR_H_

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Two kernels whose bodies only wait for their grid dependency and allow the
 * dependent launch: the first with grid_a CTAs of block_a threads and smem_a
 * bytes of dynamic shared memory, the second with grid_b, block_b, smem_b.
 * pdl = 1 launches both as programmatic dependents (as the decode kernels of
 * a plan with pdl = 1 are), pdl = 0 in plain stream order.  grid: 1..65535,
 * block: a multiple of 32 in 32..1024, smem: 0..232448 (227 KiB), pdl: 0 or 1;
 * anything else is MLA_EINVAL.  Errors: MLA_EINVAL, MLA_ENOTREADY, MLA_ECUDA. */
MLA_API int mla_floor_empty_pair(int grid_a, int block_a, int smem_a, int grid_b, int block_b, int smem_b, int pdl,
                                 void *stream);

/* One kernel of `ctas` single-warp CTAs that reads `bytes` of device memory at
 * `src` into shared memory with bulk copies (the copy engine the decode
 * kernels load the cache with), CTA i taking the i-th of `ctas` equal
 * 16-byte-aligned pieces, up to 192 KiB in flight per CTA, and writes one
 * 32-bit word of what it read to sink[i] so the reads are used.  Its waits are
 * bounded (about 2 s); one that runs out writes MLA_EDEVICE to *status (an
 * int32 the caller zeroes) and the CTA leaves after its copies land.
 * src: (device) 16-byte aligned; bytes: a positive multiple of 16; ctas:
 * 1..65535; sink: (device) uint32 [ctas]; status: (device) int32; pdl: 0 or 1
 * as above.  Errors: MLA_EINVAL, MLA_EALIGN, MLA_ENOTREADY, MLA_ECUDA. */
MLA_API int mla_floor_read(const void *src, size_t bytes, int ctas, unsigned *sink, int *status, int pdl,
                           void *stream);

/* One kernel of `ctas` single-warp CTAs that gathers listed rows of a cache
 * into shared memory, one bulk copy per row (as the sparse decode's producer
 * warps fetch indexed rows), and computes nothing: rows[] holds n_rows row
 * numbers of the cache at `kv` (kv_rows rows, row_stride bytes apart, each
 * row_bytes long); CTA i takes the i-th of `ctas` equal runs of the list, in
 * rounds of up to 96 KiB, two rounds in flight.  Entries outside [0, kv_rows)
 * are skipped.  One 32-bit word of what a CTA read goes to sink[i]; waits are
 * bounded as for mla_floor_read (MLA_EDEVICE in *status).
 * kv: (device) 16-byte aligned; row_stride, row_bytes: multiples of 16,
 * 16 <= row_bytes <= 98304 and row_bytes <= row_stride; rows: (device)
 * int64 [n_rows], 8-byte aligned; n_rows >= 1; ctas: 1..65535; sink: (device)
 * uint32 [ctas]; status: (device) int32; pdl: 0 or 1.
 * Errors: MLA_EINVAL, MLA_EALIGN, MLA_ENOTREADY, MLA_ECUDA. */
MLA_API int mla_floor_gather(const void *kv, long long kv_rows, long long row_stride, int row_bytes,
                             const long long *rows, long long n_rows, int ctas, unsigned *sink, int *status, int pdl,
                             void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_FLOOR_H_ */
