/*
 * gc_gb300_testing.h -- test hooks of libgc_gb300.so.  Not part of the
 * production ABI; they exist so that the failure paths of the library can be
 * exercised without faulting, trapping or hanging a GPU, and its host-side
 * launch rules checked without one.
 */
#ifndef GC_GB300_TESTING_H
#define GC_GB300_TESTING_H

#include "gc_gb300.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gc_testing_saps_mask_compact_withhold -- saps_mask_compact in which tile
 * `withhold_tile` (4096 elements per tile) never publishes its look-back
 * state, and every look-back wait is bounded by `wait_ns` nanoseconds
 * (1 .. 10^9).  Its successors' waits run out, they count the silent tile as
 * empty, record GC_ERR_TIMEOUT in *d_status and finish; the kernel returns
 * and the CUDA context stays usable.  Arguments otherwise as
 * saps_mask_compact (SAPS section II-B; the bounded decoupled look-back).
 * Errors: as saps_mask_compact, and GC_ERR_INVALID for wait_ns out of range.
 */
GC_API int gc_testing_saps_mask_compact_withhold(int64_t n, double p, uint64_t seed_t,
                                                 const float *const *models, int W,
                                                 uint32_t *idx, float *const *vals,
                                                 int64_t capacity, uint64_t *d_count,
                                                 void *workspace, size_t workspace_bytes,
                                                 int *d_status, int64_t withhold_tile,
                                                 uint64_t wait_ns, gc_stream_t stream);

/*
 * gc_testing_saps_round_one_pass -- saps_round with the one-pass kernel
 * whatever p is (saps_round itself takes the two-launch path when a tile's
 * expected masked count would not fit the kernel's shared-memory stash), so
 * that the kernel's own overflow path -- a tile whose stash fills fetches
 * its prefix mid-tile and writes the rest directly -- can be tested.
 * W <= 16.  Arguments and errors as saps_round.
 */
GC_API int gc_testing_saps_round_one_pass(int64_t n, double p, uint64_t seed_t,
                                          float *const *models, int W, const int *pairs,
                                          float alpha, float beta, float *center,
                                          uint32_t *idx, float *const *vals, int64_t capacity,
                                          uint64_t *d_count, void *workspace,
                                          size_t workspace_bytes, int *d_status,
                                          gc_stream_t stream);

/*
 * gc_testing_decode_buckets_per_cta -- the Elias decoders' host rule for the
 * buckets each decoding CTA takes ("QSGD ...", Knowl 2; a thread walks one
 * bucket's stream, so an SM's time is its bucket count), on given sizes and
 * without a device: W streams of nb buckets, CTAs of at most maxb buckets,
 * `slots` CTAs resident at once (SMs x CTAs per SM).  The rule takes the
 * fewest waves of `slots` CTAs that hold the buckets and spreads the buckets
 * evenly over them; the decoders then launch ceil(nb / *bpc) CTAs per stream.
 *   nb       1 .. 2^40       W      1 .. GC_MAX_WORKERS
 *   slots    1 .. 2^20       maxb   1 .. 1024
 *   bpc      host int64, out: 1 .. maxb
 * Errors: GC_ERR_INVALID for an argument out of range or a NULL bpc.
 */
GC_API int gc_testing_decode_buckets_per_cta(int64_t nb, int W, int64_t slots, int maxb, int64_t *bpc);

/*
 * gc_testing_qsgd_elias_encode_withhold -- qsgd_elias_encode in which bucket
 * `withhold_bucket` never publishes its look-back state (word count or
 * prefix), and every look-back wait is bounded by `wait_ns` nanoseconds
 * (1 .. 10^9).  The buckets after it wait out their bound, count it as
 * empty, record GC_ERR_TIMEOUT in the workspace's status word and finish;
 * the kernel returns and the CUDA context stays usable.  Arguments otherwise
 * as qsgd_elias_encode ("QSGD ...", Knowl 2; the bounded look-back).
 * Errors: as qsgd_elias_encode, and GC_ERR_INVALID for wait_ns out of range
 * or a negative bucket.
 */
GC_API int gc_testing_qsgd_elias_encode_withhold(const uint8_t *codes, const float *norms,
                                                 int64_t n, int bucket, int s_levels,
                                                 uint32_t *words, uint64_t capacity_words,
                                                 uint32_t *offsets, void *workspace,
                                                 size_t ws_bytes, int64_t withhold_bucket,
                                                 uint64_t wait_ns, gc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GC_GB300_TESTING_H */
