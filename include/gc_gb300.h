/*
 * gc_gb300.h -- C ABI of the GB300 (sm_103a) gradient-compression library
 * (libgc_gb300.so).
 *
 * Gradient compression with error feedback for data-parallel SGD, with the
 * W data-parallel workers held as separate buffers on one GPU:
 *   - MXNet-style 2-bit threshold quantisation with a residual, its
 *     dequantise-sum fused with an SGD or EASGD update, and CD-SGD's periodic
 *     full-precision correction step;
 *   - QSGD bucketed stochastic quantisation to 4- or 8-bit sign-magnitude
 *     codes, its dequantise-sum, and the lossless Elias-omega coding of the
 *     codes (dense and sparse regimes);
 *   - SAPS seeded random-mask sparsification compacted to (index, value)
 *     pairs, peer averaging over a random or bandwidth-aware perfect
 *     matching, and the EASGD elastic step;
 *   - one-pass forms of each method's step (gc_2bit_step, qsgd_step,
 *     saps_round), bit-identical to the separate calls, and S successive
 *     2-bit steps of one worker in one launch (gc_2bit_quantize_steps);
 *   - per-worker forms of the SAPS exchange steps for workers that live in
 *     different processes (saps_pair_average_remote, easgd_step_from_sum).
 *
 * Conventions shared by every entry point
 *   Ownership   The caller allocates and owns every buffer.  The library
 *               allocates no memory, holds no state between calls (except
 *               the fixed scratch array of saps_mask_compact_noalloc) and
 *               never synchronises the device.
 *   Execution   Each call validates its arguments on the host, enqueues its
 *               kernels on `stream` (a cudaStream_t; NULL is the legacy
 *               default stream) and returns.  Results are valid once the
 *               stream reaches that point.  `stream` belongs to the current
 *               device: launch shapes (SM count, shared-memory sizes) are
 *               taken from it.
 *   Status      The return value is GC_OK or a negative GC_ERR_* code from
 *               host validation, or GC_ERR_CUDA when a launch failed.  Errors
 *               found on the device (compaction capacity, look-back timeout,
 *               a coded stream that does not decode) are written to the
 *               caller's device int `d_status`.
 *   Pointers    "device" pointers are CUDA device memory of the current
 *               device; pointer arrays (const float* const* ...) are HOST
 *               arrays of device pointers, read during the call only.
 *               Data pointers must be 16-byte aligned (GC_ERR_ALIGN).
 *   Sizes       n is an element count; n == 0 is a successful no-op, n < 0
 *               is GC_ERR_INVALID.  Every n up to 2^40 is accepted
 *               (64-bit indexing).
 *   Aliasing    Inputs and outputs of one call must not overlap unless the
 *               argument is documented as in/out.
 *   Floating    All kernels are IEEE fp32 with round-to-nearest, no
 *               flush-to-zero and no fast-math.
 */
#ifndef GC_GB300_H
#define GC_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GC_API __attribute__((visibility("default")))
#else
#define GC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle, ABI-compatible with cudaStream_t. */
typedef struct CUstream_st *gc_stream_t;

/* Status codes. */
enum {
    GC_OK = 0,
    GC_ERR_INVALID = -1,  /* bad size, count, parameter or NULL pointer      */
    GC_ERR_ALIGN = -2,    /* a data pointer is not 16-byte aligned           */
    GC_ERR_CUDA = -3,     /* a CUDA launch or runtime call failed            */
    GC_ERR_CAPACITY = -4, /* device: more masked entries than the capacity   */
    GC_ERR_TIMEOUT = -5,  /* device: a bounded wait in the compaction ran out */
    GC_ERR_CORRUPT = -6   /* device: a coded stream does not decode           */
};

/* Gradient element type. */
typedef enum { GC_F32 = 0, GC_BF16 = 1 } gc_dtype;

/* Update applied after the dequantise-sum. */
typedef enum { GC_UPD_NONE = 0, GC_UPD_SGD = 1, GC_UPD_EASGD = 2 } gc_update;

#define GC_MAX_WORKERS 64

/* Human-readable name of a status code (static string, never NULL). */
GC_API const char *gc_status_string(int status);

/* Library ABI version, (major << 16) | minor. */
GC_API int gc_version(void);

/*
 * gc_l2_fetch_granularity -- sets the CUDA runtime's L2 fetch-granularity
 * hint (cudaLimitMaxL2FetchGranularity) of the calling thread's current
 * device context to `bytes` (0 .. 128) and, when previous is not NULL,
 * stores the value it replaces there.  A per-process setting, gone with the
 * context: it changes nothing on the GPU beyond it.  Random 4-byte gathers
 * (saps_mask_compact) run faster at 32 or 64 bytes; streaming kernels were
 * measured unchanged.  It applies to kernels launched after the call:
 * synchronise first if work already queued should keep the old value.
 * Errors: GC_ERR_INVALID (bytes > 128), GC_ERR_CUDA.
 */
GC_API int gc_l2_fetch_granularity(size_t bytes, size_t *previous);

/* ---------------------------------------------------------------------- */
/* 2-bit threshold quantisation with error feedback                       */
/* ---------------------------------------------------------------------- */

/*
 * gc_2bit_quantize -- "2bit gradient compression" (MXNet PR #8662),
 * sections "Two bit quantization" and "Format of compressed gradient".
 *
 * For every element i:  r = residual[i] + grad[i]  (one fp32 add);
 *   r >= +threshold -> code 11, residual[i] = r - threshold
 *   r <= -threshold -> code 10, residual[i] = r + threshold
 *   otherwise       -> code 00, residual[i] = r
 * Codes are packed 16 per uint32 word, element 16k+j in bits (31-2j, 30-2j)
 * of word k (first element in the most significant bits); the unused bits of
 * the last word are zero.
 *
 *   grad       n elements of type `dtype` (fp32 or bf16), read only; device
 *              memory, or page-locked host memory the GPU addresses directly
 *              (read in place over the host link)
 *   residual   device fp32 [n], in/out (the error-feedback memory)
 *   codes      device uint32 [ceil(n/16)], written
 *   threshold  finite, > 0
 * Errors: GC_ERR_INVALID (n < 0, threshold not finite and positive, bad
 * dtype, NULL), GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int gc_2bit_quantize(const void *grad, gc_dtype dtype, float *residual,
                     uint32_t *codes, int64_t n, float threshold,
                     gc_stream_t stream);

/*
 * gc_2bit_quantize_batched -- gc_2bit_quantize on B buffers in one launch
 * (the W workers held on this GPU, or the many gradient tensors of one
 * worker); same rule, layout and residual update per buffer.
 *
 *   grads      host array of B pointers, n[b] elements of `dtype` each, in
 *              device memory or GPU-addressable page-locked host memory
 *   residuals  host array of B device pointers, fp32 [n[b]], in/out
 *   codes      host array of B device pointers, uint32 [ceil(n[b]/16)]
 *   n          host array of B sizes (0 allowed: that buffer is skipped)
 *   B          1 .. GC_MAX_WORKERS
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int gc_2bit_quantize_batched(const void *const *grads, gc_dtype dtype,
                                    float *const *residuals, uint32_t *const *codes,
                                    const int64_t *n, int B, float threshold,
                                    gc_stream_t stream);

/*
 * gc_2bit_dequant_sum_update -- MXNet PR #8662 "Local kvstore" / "Dist
 * kvstore" (the receiver dequantises every worker's codes, 11 -> +t,
 * 10 -> -t, 00 and 01 -> 0, and sums them); CD-SGD eq. 10 (global update
 * with the averaged compressed gradients); EASGD local update (IMerge design
 * notes) with the averaged gradient as g.
 *
 *   avg_i = (sum_w dec(codes[w], i)) * threshold / W
 *   GC_UPD_NONE : out[i] = avg_i                       (weights, center unused)
 *   GC_UPD_SGD  : weights[i] -= lr * avg_i             (out, center unused)
 *   GC_UPD_EASGD: weights[i] = weights[i] - lr * avg_i
 *                              - alpha * (weights[i] - center[i])
 *
 *   codes      host array of W device pointers, each uint32 [ceil(n/16)]
 *   W          1 .. GC_MAX_WORKERS
 *   center     device fp32 [n] (EASGD only, read), else may be NULL
 *   weights    device fp32 [n] in/out (SGD, EASGD), else may be NULL
 *   out        device fp32 [n] written (NONE), else may be NULL
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int gc_2bit_dequant_sum_update(const uint32_t *const *codes, int W, int64_t n,
                               float threshold, gc_update kind, float lr,
                               float alpha, const float *center,
                               float *weights, float *out, gc_stream_t stream);

/*
 * gc_2bit_step -- gc_2bit_quantize_batched over W equal-sized gradient
 * buffers followed by gc_2bit_dequant_sum_update, in one pass: each
 * element's decoded sum is formed while its codes are produced, so the codes
 * are written but not read back.  Codes, residuals and the update are
 * bit-identical to the two separate calls.  (MXNet PR #8662 "Local kvstore":
 * every device quantises, one sums the dequantised values; CD-SGD eq. 10 and
 * Algorithm 1's compressed iteration.)
 *
 *   grads      host array of W device pointers, fp32 or bf16 (dtype) [n]
 *   residuals, codes
 *              host arrays of W pointers as in the batched quantiser
 *   kind, lr, alpha, center, weights, out
 *              as gc_2bit_dequant_sum_update
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int gc_2bit_step(const void *const *grads, gc_dtype dtype,
                        float *const *residuals, uint32_t *const *codes, int W,
                        int64_t n, float threshold, gc_update kind, float lr,
                        float alpha, const float *center, float *weights,
                        float *out, gc_stream_t stream);

/*
 * gc_2bit_step_local -- gc_2bit_step that also writes each worker's CD-SGD
 * local weights (eq. 11 and Algorithm 1's local step):
 *   local_weights[w][i] = weights[i] - local_lr * g_w[i]
 * from the weights as they are before this call's update, i.e. the same
 * values gc_2bit_quantize_local writes; everything else as gc_2bit_step.
 * Bit-identical to gc_2bit_quantize_local followed by
 * gc_2bit_dequant_sum_update.
 *
 *   local_weights  host array of W device pointers, fp32 [n], out (must not
 *                  alias weights or each other)
 *   local_lr       eta_loc, finite
 *   weights        required (read for the local weights) for every kind
 * Errors: GC_ERR_INVALID (also local_weights NULL), GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int gc_2bit_step_local(const void *const *grads, gc_dtype dtype,
                              float *const *residuals, uint32_t *const *codes,
                              float *const *local_weights, float local_lr, int W,
                              int64_t n, float threshold, gc_update kind, float lr,
                              float alpha, const float *center, float *weights,
                              float *out, gc_stream_t stream);

/*
 * gc_2bit_quantize_steps -- S successive 2-bit steps of one worker in one
 * launch (MXNet PR #8662 "Two bit quantization": the residual carries what
 * was not sent to the next step).  Step s (0-based) quantises grads[s] with
 * the residual left by step s-1 and writes codes[s]; with `out`, also the
 * dequantised values out[s][i] = +t, -t or 0 (the W = 1 dequant-sum).  The
 * residual is read once and written once, after the last step.
 * Bit-identical to S calls of gc_2bit_quantize (each followed by
 * gc_2bit_dequant_sum_update with W = 1 and GC_UPD_NONE when out is given).
 *
 *   grads      host array of S device pointers, fp32 or bf16 (dtype) [n]
 *   residual   device fp32 [n], in/out
 *   codes      host array of S device pointers, uint32 [ceil(n/16)], out
 *   out        host array of S device pointers, fp32 [n], out; or NULL
 *   S          1 .. GC_MAX_WORKERS
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int gc_2bit_quantize_steps(const void *const *grads, gc_dtype dtype,
                                  float *residual, uint32_t *const *codes,
                                  float *const *out, int S, int64_t n,
                                  float threshold, gc_stream_t stream);

/*
 * gc_2bit_quantize_local -- gc_2bit_quantize on B workers' gradients (one
 * launch), each also producing the worker's local weights of CD-SGD eq. 11
 * (Algorithm 1 line 24): local_weights[b][i] = weights[i] - local_lr *
 * grad[b][i] (one fma), from the global weights before this step's update.
 *
 *   weights        device fp32 [n], the global weights, read only
 *   local_weights  host array of B device pointers, fp32 [n], written
 *   other arguments as gc_2bit_quantize_batched, with one size n for all
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int gc_2bit_quantize_local(const void *const *grads, gc_dtype dtype,
                                  float *const *residuals, uint32_t *const *codes,
                                  const float *weights, float *const *local_weights,
                                  int B, int64_t n, float threshold, float local_lr,
                                  gc_stream_t stream);

/*
 * gc_compensated_sum_update -- CD-SGD, Algorithm 1 (the branch taken every
 * k-th step, where the 32-bit gradient is pushed uncompressed) and section
 * 3.1 (k-step correction).  Reading: the pushed message is the
 * residual-compensated gradient, after which the residual is empty:
 *   m_w = residuals[w][i] + grads[w][i]   (fp32);  residuals[w][i] = 0
 *   weights[i] -= lr * (sum_w m_w) / W    (CD-SGD eq. 1)
 * No fp32 message is written to memory.
 *
 *   grads      host array of W device pointers, n elements of `dtype`
 *   residuals  host array of W device pointers, fp32 [n], in/out (zeroed)
 *   weights    device fp32 [n], in/out
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int gc_compensated_sum_update(const void *const *grads, gc_dtype dtype,
                              float *const *residuals, int W, int64_t n,
                              float lr, float *weights, gc_stream_t stream);

/* ---------------------------------------------------------------------- */
/* QSGD                                                                   */
/* ---------------------------------------------------------------------- */

/*
 * qsgd_quantize -- "QSGD: Communication-Efficient SGD via Gradient
 * Quantization and Encoding", Knowl 1 (operator Q_s), Knowl 2 (norm stored
 * as fp32, sign and level per coordinate), Knowl 8 (bucketing).
 *
 * Per bucket b of `bucket` consecutive elements (the last may be shorter):
 *   norms[b] = the l2 norm of the bucket, rounded to nearest fp32
 *   S = s_levels / norms[b]                       (fp32 division)
 *   per element: a = |v| * S, x = a + u, level = min(floor(x), s_levels)
 *   with u = f * 2^-24, f the 24-bit dither field of element i: with
 *   z = splitmix64(seed_w ^ floor(i/2)), bits 40..63 of z for even i and
 *   bits 8..31 for odd i (one SplitMix64 output per pair of elements),
 *   seed_w = seed ^ ((uint64)worker << 48), i the global element index; a
 *   bucket whose norm is 0 has level 0 everywhere.  Sign bit = (v < 0), so
 *   sgn(0) = +1.
 * Codes are sign-magnitude:
 *   1 <= s_levels <= 7  : 4-bit codes (sign in bit 3), two per byte, element
 *                         2j in the HIGH nibble of byte j; codes has
 *                         ceil(n/2) bytes, the unused low nibble is 0
 *   8 <= s_levels <= 127: 8-bit codes (sign in bit 7), codes has n bytes
 *
 *   grad       device fp32 [n], read only
 *   bucket     128, 256, 512, 1024 or 2048
 *   norms      device fp32 [ceil(n/bucket)], written
 *   codes      device uint8 [ceil(n/2)] or [n], written
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int qsgd_quantize(const float *grad, int64_t n, int bucket, int s_levels,
                  uint64_t seed, int worker, float *norms, uint8_t *codes,
                  gc_stream_t stream);

/*
 * qsgd_quantize_maxnorm -- QSGD Knowl 8, max-norm scaling: as qsgd_quantize
 * but each bucket is scaled by its largest coordinate magnitude ||v||_inf
 * (stored exactly in scales[b]) instead of its l2 norm; qsgd_dequant_sum
 * decodes the result unchanged (scales in place of norms).
 * Errors: as qsgd_quantize.
 */
GC_API int qsgd_quantize_maxnorm(const float *grad, int64_t n, int bucket,
                                 int s_levels, uint64_t seed, int worker,
                                 float *scales, uint8_t *codes, gc_stream_t stream);

/*
 * qsgd_dequant_sum -- QSGD Knowl 2 (decode the tuple: value = norm * sign *
 * level / s) and Knowl 3 (sum the K decoded messages; scale = 1/K gives
 * their average).
 *   out[i] = sum_w sgn_w(i) * (norms[w][b] * (scale / s_levels)) * level_w(i),
 *   summed in fp32 in worker order (one fma per term).
 *
 *   codes, norms  host arrays of W device pointers laid out as qsgd_quantize
 *                 writes them
 *   out           device fp32 [n], written
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int qsgd_dequant_sum(const uint8_t *const *codes, const float *const *norms,
                     int W, int64_t n, int bucket, int s_levels, float scale,
                     float *out, gc_stream_t stream);

/*
 * qsgd_step -- synchronous parallel QSGD's compression and aggregation for W
 * simulated workers in one pass (Knowl 3: each worker quantises its
 * gradient; the decoded messages are summed): the results of
 *   qsgd_quantize(grads[w], n, bucket, s_levels, seed, w, norms[w], codes[w])
 *   for w = 0 .. W-1 (qsgd_quantize_maxnorm when maxnorm = 1), then
 *   qsgd_dequant_sum(codes, norms, W, n, bucket, s_levels, scale, out)
 * bit for bit, with each bucket's W gradients read once and the sum kept in
 * registers (the codes and norms are still written: they are the messages).
 *   grads      host array of W device pointers, fp32 [n], read only
 *   norms, codes   host arrays of W device pointers, written as qsgd_quantize
 *   out        device fp32 [n], written
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int qsgd_step(const float *const *grads, int W, int64_t n, int bucket, int s_levels,
                     uint64_t seed, int maxnorm, float *const *norms, uint8_t *const *codes,
                     float scale, float *out, gc_stream_t stream);

/* ---------------------------------------------------------------------- */
/* QSGD Elias-omega coding                                                */
/* ---------------------------------------------------------------------- */

/*
 * qsgd_elias_encode -- "QSGD: Communication-Efficient SGD via Gradient
 * Quantization and Encoding", Knowl 2, dense regime: the lossless code of the
 * quantised tuple (norm, signs, levels) that qsgd_quantize writes.  Per bucket
 * b, in a stream of 32-bit words read most significant bit first:
 *   the 32 bits of norms[b], then for each coordinate in order
 *   Elias-omega(level + 1) (Elias, IEEE Trans. Inf. Theory 21(2), 1975),
 *   followed by its sign bit (1 = negative) when level > 0;
 *   the bucket's last word is padded with zero bits.
 * Every bucket starts on a word boundary; offsets[b] is its first word and
 * offsets[nbuckets] the number of words written, so that the receiver
 * decodes the buckets in parallel (side information not on the pages: 32
 * bits per bucket).  The sign of a level-0 coordinate is not sent.
 *
 *   codes, norms   device, as qsgd_quantize writes them (read only)
 *   words          device uint32 [capacity_words]; capacity_words must be at
 *                  least qsgd_elias_max_words(n, bucket, s_levels)
 *   offsets        device uint32 [ceil(n/bucket) + 1], written
 *   workspace      device, qsgd_elias_workspace_bytes(n, bucket) bytes
 *                  (contents need not be preserved between calls); after
 *                  the call its first 4 bytes hold the device status: GC_OK,
 *                  or GC_ERR_TIMEOUT when a wait of the look-back below ran
 *                  out (only a fault elsewhere can delay a CTA that long;
 *                  the stream is then not valid)
 * One memset and one kernel launch on `stream`; the kernel reads the codes
 * once: each bucket's first word comes from a decoupled look-back (Merrill
 * and Garland 2016) over the word counts of the buckets before it.  The
 * total length is offsets[nbuckets] on the device.
 * Errors: GC_ERR_INVALID (bad bucket or s_levels, n < 0, NULL, workspace too
 * small, a bound above 2^32 - 1 words), GC_ERR_CAPACITY (capacity_words below
 * the bound), GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int qsgd_elias_encode(const uint8_t *codes, const float *norms, int64_t n,
                             int bucket, int s_levels, uint32_t *words,
                             uint64_t capacity_words, uint32_t *offsets,
                             void *workspace, size_t ws_bytes, gc_stream_t stream);

/*
 * Upper bound on the words qsgd_elias_encode writes, whatever the codes:
 * per bucket of L coordinates 1 + ceil(L * c / 32) with c = 8 bits for 4-bit
 * codes (level 7) and c = 15 for 8-bit codes (level 127).  0 for invalid
 * arguments.
 */
GC_API uint64_t qsgd_elias_max_words(int64_t n, int bucket, int s_levels);

/* Bytes of device workspace qsgd_elias_encode needs (0 for invalid arguments). */
GC_API size_t qsgd_elias_workspace_bytes(int64_t n, int bucket);

/*
 * qsgd_elias_decode -- the inverse of qsgd_elias_encode (Knowl 2: decode the
 * tuple): norms and codes in qsgd_quantize's layout; a level-0 coordinate
 * comes back with sign 0.  Bucket b reads only words[offsets[b] ..
 * offsets[b+1]); missing bits read as zeros.
 *   d_status   device int or NULL; set to GC_ERR_CORRUPT when a bucket's
 *              codewords run past its words, a level exceeds s_levels (it is
 *              written as s_levels, with its sign, and the codes after it
 *              decode as they would otherwise), a codeword is not an
 *              Elias-omega codeword of at most 8 binary digits, or a bucket
 *              has no norm word
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int qsgd_elias_decode(const uint32_t *words, const uint32_t *offsets, int64_t n,
                             int bucket, int s_levels, uint8_t *codes, float *norms,
                             int *d_status, gc_stream_t stream);

/*
 * qsgd_elias_decode_batched -- qsgd_elias_decode of W streams of the same n,
 * bucket and s_levels (the W workers' messages a receiver decodes before
 * their sum, Knowl 3) in one launch; stream w's results are those of
 * qsgd_elias_decode on (words[w], offsets[w]).  The decoder gives one thread
 * to each bucket, so W streams keep W times more of the GPU busy.
 *   words, offsets, codes, norms   host arrays of W device pointers, each as
 *                                  in qsgd_elias_decode
 *   W          1 .. GC_MAX_WORKERS
 *   d_status   device int or NULL, shared by the W streams
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int qsgd_elias_decode_batched(const uint32_t *const *words,
                                     const uint32_t *const *offsets, int W, int64_t n,
                                     int bucket, int s_levels, uint8_t *const *codes,
                                     float *const *norms, int *d_status,
                                     gc_stream_t stream);

/*
 * qsgd_elias_encode_marked -- qsgd_elias_encode that also writes each
 * bucket's quarter marks: marks[3*b + k - 1], k = 1..3, is the bit (from the
 * start of bucket b's first word, the norm's 32 bits included) at which the
 * codeword of coordinate k*bucket/4 of that bucket begins; a quarter that
 * starts at or past a short last bucket's end gets the bucket's total bits.
 * The stream and offsets are those of qsgd_elias_encode, bit for bit.  The
 * marks are side information not on the pages (48 bits per bucket, 0.09 bits
 * per coordinate at bucket 512) that let a receiver decode a bucket's four
 * quarters in parallel (qsgd_elias_decode_quarters).
 *   marks   device uint16 [3 * ceil(n/bucket)], 16-byte aligned, written
 *           (a bucket holds at most 32 + 2048 * 15 < 2^16 bits)
 * Other arguments and errors as qsgd_elias_encode; GC_ERR_INVALID for a NULL
 * marks with n > 0.
 */
GC_API int qsgd_elias_encode_marked(const uint8_t *codes, const float *norms, int64_t n,
                                    int bucket, int s_levels, uint32_t *words,
                                    uint64_t capacity_words, uint32_t *offsets,
                                    uint16_t *marks, void *workspace, size_t ws_bytes,
                                    gc_stream_t stream);

/*
 * qsgd_elias_decode_quarters -- qsgd_elias_decode of a stream written by
 * qsgd_elias_encode_marked, with more decoding threads per bucket: for 8-bit
 * codes (s_levels > 7) one per quarter bucket, starting at the quarter
 * marks; for 4-bit codes, whose streams are about half as long, one per half
 * bucket, starting at the middle mark (marks[3*b + 1]).  Same results as
 * qsgd_elias_decode on (words, offsets).
 *   marks      device uint16 [3 * ceil(n/bucket)], as the encoder wrote them
 *   d_status   as in qsgd_elias_decode; also set to GC_ERR_CORRUPT when a
 *              part's codewords do not end exactly at the mark the next part
 *              starts from, or the last part holding coordinates of a short
 *              bucket does not end exactly at the marks of the parts after
 *              it (so that any mark the decoder starts from, other than the
 *              encoder's, is reported)
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int qsgd_elias_decode_quarters(const uint32_t *words, const uint32_t *offsets,
                                      const uint16_t *marks, int64_t n, int bucket,
                                      int s_levels, uint8_t *codes, float *norms,
                                      int *d_status, gc_stream_t stream);

/*
 * qsgd_elias_encode_sparse -- QSGD's Elias coding in the sparse regimes
 * ("QSGD ..." summary page, Knowl 2 items 1 (s >= 2) and 1' (s = 1)): only
 * the coordinates whose level is not 0 are sent, each as Elias-omega of its
 * distance from the previous one (the first from -1), one sign bit and, when
 * s_levels >= 2, Elias-omega(level); Elias-omega(bucket length - last index)
 * closes each bucket.  Stream conventions as qsgd_elias_encode: 32-bit words
 * read most significant bit first, every bucket on a word boundary behind
 * its fp32 norm, offsets[b] its first word, offsets[nbuckets] the length.
 * Worth it where most levels are 0 (s = 1, small s on peaked gradients).
 *
 *   codes, norms, n, bucket, s_levels, offsets, workspace, ws_bytes
 *                  as qsgd_elias_encode (same workspace size, same status
 *                  word in its first 4 bytes after the call)
 *   words          device uint32 [capacity_words], at least
 *                  qsgd_elias_sparse_max_words(n, bucket)
 * One memset and one kernel launch on `stream` (the codes are read once, as
 * in qsgd_elias_encode).
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CAPACITY, GC_ERR_CUDA.
 */
GC_API int qsgd_elias_encode_sparse(const uint8_t *codes, const float *norms, int64_t n,
                                    int bucket, int s_levels, uint32_t *words,
                                    uint64_t capacity_words, uint32_t *offsets,
                                    void *workspace, size_t ws_bytes, gc_stream_t stream);

/* Upper bound on the words qsgd_elias_encode_sparse writes: per bucket of
 * len coordinates 1 + ceil((18 len + 2) / 32) (0 for invalid arguments). */
GC_API uint64_t qsgd_elias_sparse_max_words(int64_t n, int bucket);

/*
 * qsgd_elias_decode_sparse -- the inverse of qsgd_elias_encode_sparse: norms
 * and codes in qsgd_quantize's layout, every coordinate not in the stream
 * (and the sign of every level-0 coordinate) 0.  Bucket b reads only
 * words[offsets[b] .. offsets[b+1]).
 *   d_status   device int or NULL; set to GC_ERR_CORRUPT when a distance
 *              runs past the bucket's end, a bucket's codewords run past its
 *              words, a level exceeds s_levels (written as s_levels), a
 *              codeword is longer than any valid one, or a bucket has no
 *              norm word
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int qsgd_elias_decode_sparse(const uint32_t *words, const uint32_t *offsets, int64_t n,
                                    int bucket, int s_levels, uint8_t *codes, float *norms,
                                    int *d_status, gc_stream_t stream);

/* ---------------------------------------------------------------------- */
/* SAPS sparsified gossip + EASGD                                         */
/* ---------------------------------------------------------------------- */

/*
 * saps_round_seed -- the shared seed of SAPS round t: splitmix64(base + t).
 * Host only; "Communication-Efficient Decentralized Learning with
 * Sparsification and Adaptive Peer Selection", section II-A (the
 * coordinator sends each round's seed to all workers).
 */
GC_API uint64_t saps_round_seed(uint64_t base_seed, uint64_t t);

/*
 * saps_matching -- the round's single-peer gossip partners (SAPS section
 * II-C: each worker exchanges with exactly one peer; the gossip matrix is
 * doubly stochastic).  The pages pick the matching from measured link
 * bandwidths; here it is a uniformly random perfect matching drawn from the
 * round seed: a Fisher-Yates shuffle with j = splitmix64(splitmix64(seed_t)
 * ^ i) mod (i + 1) for i = W-1 .. 1.  Host only.
 *   pairs_out  host int [W]; pairs are (pairs_out[2q], pairs_out[2q+1])
 * Errors: GC_ERR_INVALID (W not even, W < 2, W > GC_MAX_WORKERS, NULL).
 */
GC_API int saps_matching(uint64_t seed_t, int W, int *pairs_out);

/*
 * saps_matching_bandwidth -- the round's gossip partners chosen from link
 * bandwidths, as the coordinator of SAPS section II-C (Algorithm 3) does.
 * Host only.  Steps, in the page's order:
 *   - B_ij = B_ji = min(B_ij, B_ji) (the slower direction bounds the link);
 *   - B*: the pairs with B_ij > b_thres (section II-A's filtered matrix);
 *   - "recently connected" (RC) pairs: last_round[i][j] > t - t_thres;
 *   - if the RC pairs connect every worker, the candidate pairs are B*;
 *     otherwise they are the links (B_ij > 0) between different connected
 *     components of the RC graph;
 *   - a maximum matching of the candidates (Edmonds' blossom algorithm on a
 *     general graph), searched from a relabelling of the workers drawn from
 *     seed_t (the page's "RandomlyMaxMatch");
 *   - workers still unmatched are paired among themselves in an order drawn
 *     from seed_t, without regard to bandwidth;
 *   - last_round[i][j] = last_round[j][i] = t for every pair chosen.
 * The result is a perfect matching, so the gossip matrix (1/2 on i,i / i,j /
 * j,i / j,j of each pair) is doubly stochastic.  Reading: "maximum match" is
 * a matching of maximum cardinality (the blossom algorithm the page cites);
 * bandwidth enters through b_thres and through the bridging rule.
 *
 *   W           even, 2 .. GC_MAX_WORKERS
 *   bandwidth   host double [W*W], row-major, >= 0 and finite (0 = no link);
 *               the diagonal is ignored
 *   b_thres     B_thres (not NaN)
 *   last_round  host int64 [W*W], row-major, in/out: the round each pair was
 *               last matched (INT64_MIN, or any value <= t - t_thres, for
 *               never)
 *   t, t_thres  the round number and T_thres >= 1
 *   pairs_out   host int [W]; pairs (pairs_out[2q], pairs_out[2q+1]), the
 *               smaller worker first, pairs ordered by their first worker
 * Errors: GC_ERR_INVALID.
 */
GC_API int saps_matching_bandwidth(int W, const double *bandwidth, double b_thres,
                                   int64_t *last_round, int64_t t, int64_t t_thres,
                                   uint64_t seed_t, int *pairs_out);

/* Bytes of device workspace saps_mask_compact needs for n elements. */
GC_API size_t saps_workspace_bytes(int64_t n);

/*
 * saps_mask_compact -- SAPS section II-B: every worker draws the same
 * Bernoulli(p) mask from the round's shared seed and sends only the masked
 * coordinates.  m_i = [ (splitmix64(seed_t ^ i) >> 40) < ceil(p * 2^24) ],
 * i.e. uniform(seed_t ^ i) < p.  A single-pass prefix sum with decoupled
 * look-back writes the masked indices in ascending order, and in the same
 * pass gathers every worker's value at those indices.
 *
 *   p          in (0, 1]
 *   models     host array of W device pointers, fp32 [n], read only
 *   idx        device uint32 [capacity], written (n must be < 2^32)
 *   vals       host array of W device pointers, fp32 [capacity], written
 *   capacity   >= 0 entries available in idx and each vals[w]
 *   d_count    device uint64, written with the number of masked entries
 *              (also when it exceeds capacity)
 *   workspace  device, saps_workspace_bytes(n) bytes, 16-byte aligned; the
 *              call clears the part that must start at zero on `stream`,
 *              and leaves per-32-element mask tables there for
 *              saps_average_easgd_step
 *   d_status   device int; set to GC_ERR_CAPACITY when the count exceeds
 *              capacity (only `capacity` entries are written) and to
 *              GC_ERR_TIMEOUT if a look-back wait ran out (about one
 *              second; the output is then invalid).  Never cleared by the
 *              library: zero it before the first call.
 * The gather reads one 4-byte value at a time at random places: with the
 * context's L2 fetch granularity at 32 or 64 bytes (gc_l2_fetch_granularity)
 * instead of 128 it moves less DRAM traffic per value (about 18% faster at
 * p = 0.01 on 16 x 25.6 M, measured); the library never sets it itself.
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int saps_mask_compact(int64_t n, double p, uint64_t seed_t,
                      const float *const *models, int W, uint32_t *idx,
                      float *const *vals, int64_t capacity, uint64_t *d_count,
                      void *workspace, size_t workspace_bytes, int *d_status,
                      gc_stream_t stream);

/*
 * saps_peer_average -- SAPS Algorithm 2, lines 9-10: each worker receives
 * its peer's sparsified model and averages it with its own.  For every pair
 * (a, b) and k < min(*d_count, capacity):
 *   v = (vals[a][k] + vals[b][k]) * 0.5;  models[a][idx[k]] = models[b][idx[k]] = v
 *
 *   models     host array of W device pointers, fp32 [n], in/out
 *   vals, idx  as written by saps_mask_compact; the indices are used as they
 *              are (the call has no n to check them against), so they must
 *              come from a compaction over these models
 *   d_count    device uint64 written by saps_mask_compact
 *   pairs      host int [W], a perfect matching of 0..W-1 (saps_matching)
 * Errors: GC_ERR_INVALID (W odd, pairs not a permutation, NULL),
 * GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int saps_peer_average(float *const *models, const float *const *vals,
                      const uint32_t *idx, const uint64_t *d_count,
                      const int *pairs, int W, int64_t capacity,
                      gc_stream_t stream);

/*
 * saps_average_easgd_step -- saps_peer_average followed by easgd_step, in one
 * pass over the models (SAPS Algorithm 2 lines 9-10, then the EASGD
 * updates).  The received peer values are read from the compacted payload
 * vals[w][rank]; the rank of each masked coordinate comes from tables that
 * saps_mask_compact leaves in `workspace`, so the workspace must be the one
 * the preceding saps_mask_compact call (same n, same stream order) used.
 * Results are bit-identical to calling saps_peer_average then easgd_step.
 *
 *   models, vals, d_count, pairs, capacity   as saps_peer_average
 *   n, alpha, beta, center                   as easgd_step
 *   workspace                                as passed to saps_mask_compact
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int saps_average_easgd_step(float *const *models, const float *const *vals,
                                   const uint64_t *d_count, const int *pairs, int W,
                                   int64_t n, int64_t capacity, float alpha,
                                   float beta, float *center, const void *workspace,
                                   size_t workspace_bytes, gc_stream_t stream);

/*
 * saps_round -- one whole SAPS round (section II: mask, sparsified exchange,
 * single-peer gossip average; EASGD elastic step from the IMerge notes) in
 * one pass over the models: the results of
 *   saps_mask_compact(...); saps_peer_average(...); easgd_step(...)
 * bit for bit (idx, vals, d_count, models, center), as long as the masked
 * count fits the capacity.  When it does not, d_status gets GC_ERR_CAPACITY,
 * idx/vals hold the first `capacity` entries and every masked coordinate is
 * still averaged (the pair's values are at hand in the pass).
 *
 *   pairs      host int [W], a permutation of 0..W-1 (as saps_matching)
 *   others     as saps_mask_compact and easgd_step; W even, 2 <= W <= 64
 *              (W > 16 runs saps_mask_compact + saps_average_easgd_step)
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int saps_round(int64_t n, double p, uint64_t seed_t, float *const *models, int W,
                      const int *pairs, float alpha, float beta, float *center,
                      uint32_t *idx, float *const *vals, int64_t capacity,
                      uint64_t *d_count, void *workspace, size_t workspace_bytes,
                      int *d_status, gc_stream_t stream);

/*
 * easgd_step -- EASGD local and global updates (IMerge design notes,
 * "Interleaved Communication Scheduling"), without a gradient term:
 *   mean_i = (sum_k models[k][i]) / W                (values before the step)
 *   models[k][i] = models[k][i] - alpha * (models[k][i] - center[i])
 *   center[i]    = (1 - beta) * center[i] + beta * mean_i
 *
 *   models     host array of W device pointers, fp32 [n], in/out
 *   center     device fp32 [n], in/out
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int easgd_step(float *const *models, int W, int64_t n, float alpha, float beta,
               float *center, gc_stream_t stream);

/*
 * saps_pair_average_remote -- the SAPS pair average (section II-B/II-C: the
 * masked coordinates of both peers become their average) for a worker whose
 * peer lives in another process: after the two have exchanged their gathered
 * values (K floats each way, the indices being the same on both sides),
 *   model[idx[k]] = fl(fl(mine[k] + peer[k]) * 0.5)   for k < min(*d_count, capacity)
 * -- the value the peer writes on its side and saps_peer_average writes.
 *
 *   model      device fp32 [n], in/out
 *   idx        device uint32 [capacity], from saps_mask_compact (unchecked)
 *   d_count    device uint64, the masked count
 *   mine, peer device fp32 [capacity]: this worker's and the peer's values
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int saps_pair_average_remote(float *model, const uint32_t *idx,
                                    const uint64_t *d_count, const float *mine,
                                    const float *peer, int64_t capacity,
                                    gc_stream_t stream);

/*
 * easgd_step_from_sum -- easgd_step for one worker when the W workers'
 * models live in different processes: model_sum holds the elementwise sum of
 * all W pre-step models (e.g. an all-reduce of a copy of each model), and
 *   model[i]  = model[i] - alpha * (model[i] - center[i])
 *   center[i] = center[i] + beta * (model_sum[i] / W - center[i])
 * with the same fp32 operations as easgd_step (the sum's order is the
 * all-reduce's).  IMerge design notes, EASGD local and global updates.
 *
 *   model, center  device fp32 [n], in/out;  model_sum device fp32 [n]
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
GC_API int easgd_step_from_sum(float *model, const float *model_sum, int W, int64_t n,
                               float alpha, float beta, float *center,
                               gc_stream_t stream);

/*
 * saps_mask_compact_noalloc -- no counterpart on the pages: the same
 * compaction as saps_mask_compact, for callers that cannot provide or
 * allocate a workspace (a plug-in inside a host framework whose device
 * allocator it may not call, a loop whose device memory is fixed up front,
 * code that must avoid the implicit synchronisation of cudaMalloc/cudaFree).
 * The look-back scratch is a fixed array in device memory inside the library
 * (131,136 bytes, held by every GPU that loads the library until exit).  The
 * call allocates nothing.
 *
 *   n          0 .. GC_NOALLOC_MAX_N; larger n returns GC_ERR_INVALID
 *   other arguments as saps_mask_compact
 *   stream     must belong to the current device (the array used is that
 *              device's copy); a stream of another device returns
 *              GC_ERR_INVALID
 * Every call looks up the current device's copy of the array
 * (cudaGetSymbolAddress); the first call on a device may load the module,
 * so make that first call before any stream capture.  Every call on a device
 * shares the array and clears the part it uses on `stream`; calls that
 * overlap on the GPU race and must be ordered (one stream, or events).
 * Errors: GC_ERR_INVALID, GC_ERR_ALIGN, GC_ERR_CUDA.
 */
#define GC_NOALLOC_MAX_N (1LL << 26)
GC_API int saps_mask_compact_noalloc(int64_t n, double p, uint64_t seed_t,
                                     const float *const *models, int W,
                                     uint32_t *idx, float *const *vals,
                                     int64_t capacity, uint64_t *d_count,
                                     int *d_status, gc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GC_GB300_H */
