/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for the
 * gradient-compression hot path.
 *
 * THIS IS TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  The product library under
 * gradient_compression_sgd_gc_gb300/ shares no code, header, table or
 * constant generator with this file, and neither side includes the other.
 *
 * Conventions
 *   - Every loop runs element by element in index order; nothing is blocked,
 *     fused or reordered beyond what the cited definition says.
 *   - Where the pages fix fp32 state (the 2-bit residual carried between steps,
 *     the fp32 messages of the full-precision correction step) the oracle keeps
 *     that state in fp32 and rounds after every operation exactly as written.
 *     Where a quantised code is decided by floating point, the decision is made
 *     in fp32 with the operation order stated beside it.
 *   - Every other floating-point result (sums, averages, weight updates,
 *     dequantised values, elastic averaging) is computed in fp64.
 *   - Build flags: -O2 -ffp-contract=off (no fused multiply-add contraction),
 *     never -ffast-math.
 *
 * Sources (the web pages this method is taken from):
 *   [MX]   "2bit gradient compression", MXNet pull request #8662, sections
 *          "Two bit quantization", "Format of compressed gradient",
 *          "Local kvstore", "Dist kvstore".
 *   [CD]   "CD-SGD: Distributed Stochastic Gradient Descent with Compression
 *          and Delay Compensation", eq. 1, eq. 10, Algorithm 1, section 3.1.
 *   [QS]   "QSGD: Communication-Efficient SGD via Gradient Quantization and
 *          Encoding" (summary page), Knowl 1 (operator Q_s), Knowl 2 (the
 *          (norm, sign, level) tuple, norm stored as fp32), Knowl 3
 *          (synchronous parallel QSGD), Knowl 8 (bucketing).
 *   [SA]   "Communication-Efficient Decentralized Learning with Sparsification
 *          and Adaptive Peer Selection", section II (coordinator/worker,
 *          random mask with a shared seed, single-peer gossip matrix).
 *   [EA]   IMerge design notes (blog), "Interleaved Communication Scheduling",
 *          EASGD local and global update equations.
 *   The counter-based hash (splitmix64 of seed XOR index, 24-bit fields
 *   scaled to [0,1)) is not on the pages; it is the published SplitMix64
 *   finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
 *   generators", OOPSLA 2014).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Counter-based random numbers                                             */
/* ------------------------------------------------------------------------ */

/* SplitMix64 output function applied to one 64-bit counter value. */
uint64_t orc_splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* u(key) = (splitmix64(key) >> 40) / 2^24, a multiple of 2^-24 in [0, 1). */
double orc_uniform(uint64_t key)
{
    return (double)(orc_splitmix64(key) >> 40) / 16777216.0;
}

/*
 * QSGD's dither for global element index i of the worker whose seed is
 * seed_w: one SplitMix64 output serves a pair of elements,
 *     z = splitmix64(seed_w ^ floor(i / 2)),
 * the even element 2j taking bits 40..63 of z and the odd element 2j + 1
 * bits 8..31 (two disjoint 24-bit fields), each scaled by 2^-24.
 */
double orc_qsgd_dither(uint64_t seed_w, uint64_t i)
{
    uint64_t z = orc_splitmix64(seed_w ^ (i >> 1));
    uint64_t field = (i & 1u) ? (z >> 8) & 0xFFFFFFu : z >> 40;
    return (double)field / 16777216.0;
}

/* Round seed for SAPS round t: seed_t = splitmix64(base + t). */
uint64_t orc_round_seed(uint64_t base, uint64_t t)
{
    return orc_splitmix64(base + t);
}

/* ------------------------------------------------------------------------ */
/* [MX] 2-bit threshold quantisation with a residual                        */
/* ------------------------------------------------------------------------ */

static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float grad_at(const void *grad, int is_bf16, int64_t i)
{
    if (is_bf16)
        return bf16_bits_to_float(((const uint16_t *)grad)[i]);
    return ((const float *)grad)[i];
}

/*
 * [MX] "Two bit quantization": the residual accumulates the gradient; a value
 * greater than or equal to +t becomes code 11 and t is taken off the residual,
 * a value less than or equal to -t becomes code 10 and t is added back, every
 * other value becomes 00 and stays in the residual.
 * [MX] "Format of compressed gradient": one 32-bit word holds 16 codes, the
 * first element in the two most significant bits; unused tail bits are zero.
 * The residual is fp32 and updated with one fp32 add per step.
 */
void orc_2bit_quantize(const void *grad, int is_bf16, float *residual,
                       uint32_t *codes, int64_t n, float t)
{
    int64_t nwords = (n + 15) / 16;
    for (int64_t k = 0; k < nwords; ++k)
        codes[k] = 0u;
    for (int64_t i = 0; i < n; ++i) {
        float r = residual[i] + grad_at(grad, is_bf16, i);
        uint32_t q = 0u;
        if (r >= t) {
            q = 3u;
            r = r - t;
        } else if (r <= -t) {
            q = 2u;
            r = r + t;
        }
        residual[i] = r;
        codes[i / 16] |= q << (30 - 2 * (int)(i % 16));
    }
}

/* Decoded value of one 2-bit code: 11 -> +1, 10 -> -1, 00 and 01 -> 0. */
static int decode_2bit(const uint32_t *codes, int64_t i)
{
    uint32_t q = (codes[i / 16] >> (30 - 2 * (int)(i % 16))) & 3u;
    if (q == 3u)
        return 1;
    if (q == 2u)
        return -1;
    return 0;
}

/*
 * [MX] "Local kvstore" / "Dist kvstore": the receiver dequantises every
 * worker's codes (11 -> +t, 10 -> -t, 00 -> 0) into arrays of the original
 * size and sums them.  [CD] eq. 10: W <- W - (eta/N) * sum of the N workers'
 * compressed gradients.
 *   kind 0 (none):  out[i] = (sum_w dec_w(i) * t) / W
 *   kind 1 (SGD):   w[i]  -= lr * avg
 *   kind 2 (EASGD local step, [EA] with the averaged gradient as g):
 *                   w[i]  = w[i] - lr * avg - alpha * (w[i] - center[i])
 * All arithmetic in fp64.
 */
void orc_2bit_dequant_sum_update(const uint32_t *const *codes, int W, int64_t n,
                                 float t, int kind, double lr, double alpha,
                                 const double *center, double *w, double *out)
{
    for (int64_t i = 0; i < n; ++i) {
        double sum = 0.0;
        for (int k = 0; k < W; ++k)
            sum += (double)decode_2bit(codes[k], i) * (double)t;
        double avg = sum / (double)W;
        if (kind == 0) {
            out[i] = avg;
        } else if (kind == 1) {
            w[i] = w[i] - lr * avg;
        } else {
            w[i] = w[i] - lr * avg - alpha * (w[i] - center[i]);
        }
    }
}

/*
 * [CD] Algorithm 1 (formal training, the branch taken when count % k == 0)
 * and section 3.1: on the correction step no quantisation happens and each
 * worker pushes a 32-bit gradient.  Reading used here: the pushed message is
 * the residual-compensated gradient m = r + g in fp32, after which the
 * residual is empty.  The server applies eq. 1: W <- W - (eta/N) sum_j m_j,
 * in fp64.
 */
void orc_compensated_sum_update(const void *const *grads, int is_bf16,
                                float *const *residuals, int W, int64_t n,
                                double lr, double *w)
{
    for (int64_t i = 0; i < n; ++i) {
        double sum = 0.0;
        for (int k = 0; k < W; ++k) {
            float m = residuals[k][i] + grad_at(grads[k], is_bf16, i);
            residuals[k][i] = 0.0f;
            sum += (double)m;
        }
        w[i] = w[i] - lr * (sum / (double)W);
    }
}

/*
 * [CD] eq. 11 and Algorithm 1 line 24: each worker's local weights are the
 * global weights of the previous step moved by its own uncompressed
 * gradient, W_loc = W - eta_loc * grad (fp64).
 */
void orc_cdsgd_local_update(const void *grad, int is_bf16, const double *w,
                            double *local, int64_t n, double lr)
{
    for (int64_t i = 0; i < n; ++i)
        local[i] = w[i] - lr * (double)grad_at(grad, is_bf16, i);
}

/* ------------------------------------------------------------------------ */
/* [QS] QSGD stochastic quantisation                                        */
/* ------------------------------------------------------------------------ */

/*
 * Exact summation of doubles as a non-overlapping expansion (Shewchuk,
 * "Adaptive Precision Floating-Point Arithmetic and Fast Robust Geometric
 * Predicates", 1997 -- the partials method behind Python's math.fsum).
 */
#define ORC_MAX_PARTIALS 96
typedef struct {
    double p[ORC_MAX_PARTIALS];
    int n;
} orc_expansion;

static void expansion_add(orc_expansion *e, double x)
{
    int j = 0;
    for (int i = 0; i < e->n; ++i) {
        double y = e->p[i];
        if (fabs(x) < fabs(y)) {
            double tmp = x;
            x = y;
            y = tmp;
        }
        double hi = x + y;
        double lo = y - (hi - x);
        if (lo != 0.0)
            e->p[j++] = lo;
        x = hi;
    }
    e->p[j++] = x;
    e->n = j;
}

/* Sign of (X - m*m); m has at most 25 significant bits so m*m is exact. */
static int expansion_cmp_square(const orc_expansion *X, double m)
{
    orc_expansion e = *X;
    expansion_add(&e, -(m * m));
    for (int i = e.n - 1; i >= 0; --i)
        if (e.p[i] != 0.0)
            return e.p[i] > 0.0 ? 1 : -1;
    return 0;
}

static uint32_t float_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/*
 * [QS] Knowl 2: the l2 norm of the (bucketed) vector is stored as a single
 * precision float.  Reading: the stored value is the true l2 norm rounded to
 * nearest-even fp32.  The sum of squares is formed exactly, then the
 * candidate is moved until it is the fp32 value nearest to sqrt(sum).
 */
float orc_l2norm_fp32(const float *v, int64_t len)
{
    orc_expansion X;
    X.n = 0;
    for (int64_t i = 0; i < len; ++i) {
        double d = (double)v[i];
        expansion_add(&X, d * d); /* fp32 squared is exact in fp64 */
    }
    double approx = 0.0;
    for (int i = 0; i < X.n; ++i)
        approx += X.p[i];
    if (approx <= 0.0)
        return 0.0f;
    float r = (float)sqrt(approx);
    for (int guard = 0; guard < 64; ++guard) {
        float up = nextafterf(r, INFINITY);
        double mid_hi = ((double)r + (double)up) * 0.5;
        int c = expansion_cmp_square(&X, mid_hi);
        if (c > 0 || (c == 0 && (float_bits(r) & 1u))) {
            r = up;
            continue;
        }
        if (r > 0.0f) {
            float dn = nextafterf(r, 0.0f);
            double mid_lo = ((double)r + (double)dn) * 0.5;
            int c2 = expansion_cmp_square(&X, mid_lo);
            if (c2 < 0 || (c2 == 0 && (float_bits(r) & 1u))) {
                r = dn;
                continue;
            }
        }
        break;
    }
    return r;
}

/*
 * [QS] Knowl 1 and Knowl 8: per bucket of d coordinates (the last one may be
 * shorter), Q_s(v_i) = ||v|| * sgn(v_i) * xi_i with xi_i in {l/s, (l+1)/s},
 * sgn(0) = +1 and Q_s(0) = 0.  The random choice is made as
 *     level = floor(|v_i| / ||v|| * s + u),   u = qsgd_dither(seed_w, i)
 * with the worker folded into the seed as seed_w = seed ^ (worker << 48) and
 * i the global element index (i0 + local index, so that a bucket-aligned
 * slice of a long vector can be quantised on its own).  fp32 operation order
 * of the decision:
 *     S = s / norm,  a = |v_i| * S,  x = a + u,  level = min(floor(x), s)
 * A NaN x arises only as 0 * inf (a zero coordinate in a bucket whose s / norm
 * overflows fp32); Q_s scales |v_i|, so that coordinate gets level 0.  A
 * bucket with norm 0 gets level 0 everywhere.
 * Codes are sign-magnitude: sign bit = (v_i < 0), set above the level bits.
 *   1 <= s <= 7   : 4-bit codes, two per byte, element 2j in the HIGH nibble
 *   8 <= s <= 127 : 8-bit codes, one per byte, bit 7 = sign
 * Outputs: norms[ceil(n/d)] (fp32) and codes (ceil(n/2) or n bytes).
 */
static void qsgd_quantize_impl(const float *v, int64_t n, int64_t d, int s,
                               uint64_t seed, int worker, int64_t i0,
                               int maxnorm, float *norms, uint8_t *codes);

void orc_qsgd_quantize(const float *v, int64_t n, int64_t d, int s,
                       uint64_t seed, int worker, int64_t i0, float *norms,
                       uint8_t *codes)
{
    qsgd_quantize_impl(v, n, d, s, seed, worker, i0, 0, norms, codes);
}

/*
 * [QS] Knowl 8, max-norm scaling: each bucket is scaled by its largest
 * coordinate magnitude ||v||_inf instead of its l2 norm; everything else as
 * orc_qsgd_quantize (the stored scale is the max, exactly).
 */
void orc_qsgd_quantize_maxnorm(const float *v, int64_t n, int64_t d, int s,
                               uint64_t seed, int worker, int64_t i0,
                               float *norms, uint8_t *codes)
{
    qsgd_quantize_impl(v, n, d, s, seed, worker, i0, 1, norms, codes);
}

static float max_abs(const float *v, int64_t len)
{
    float m = 0.0f;
    for (int64_t i = 0; i < len; ++i)
        if (fabsf(v[i]) > m)
            m = fabsf(v[i]);
    return m;
}

static void qsgd_quantize_impl(const float *v, int64_t n, int64_t d, int s,
                               uint64_t seed, int worker, int64_t i0,
                               int maxnorm, float *norms, uint8_t *codes)
{
    int four_bit = (s <= 7);
    int64_t nbuckets = (n + d - 1) / d;
    uint64_t seed_w = seed ^ ((uint64_t)(uint32_t)worker << 48);
    if (four_bit)
        for (int64_t k = 0; k < (n + 1) / 2; ++k)
            codes[k] = 0;
    for (int64_t b = 0; b < nbuckets; ++b) {
        int64_t lo = b * d;
        int64_t hi = lo + d < n ? lo + d : n;
        float norm = maxnorm ? max_abs(v + lo, hi - lo) : orc_l2norm_fp32(v + lo, hi - lo);
        norms[b] = norm;
        float S = norm > 0.0f ? (float)s / norm : 0.0f;
        for (int64_t i = lo; i < hi; ++i) {
            uint32_t level = 0u;
            if (norm > 0.0f) {
                float a = fabsf(v[i]) * S;
                float u = (float)orc_qsgd_dither(seed_w, (uint64_t)(i0 + i));
                float x = a + u;
                if (x != x)
                    level = 0u;
                else if (x >= (float)s)
                    level = (uint32_t)s;
                else
                    level = (uint32_t)floorf(x);
                if (level > (uint32_t)s)
                    level = (uint32_t)s;
            }
            uint32_t sign = v[i] < 0.0f ? 1u : 0u;
            if (four_bit) {
                uint32_t code = (sign << 3) | level;
                if (i % 2 == 0)
                    codes[i / 2] |= (uint8_t)(code << 4);
                else
                    codes[i / 2] |= (uint8_t)code;
            } else {
                codes[i] = (uint8_t)((sign << 7) | level);
            }
        }
    }
}

/*
 * The fp32 value x = |v_i| * S + u whose floor decides each level above
 * (0 where the bucket's scale is 0), with S taken from the l2 norm or, when
 * maxnorm is set, from max |v_i| ([QS] Knowl 8).  The level written by the
 * quantiser is min(floor(x), s), and 0 where x is NaN.  Used by the tests to
 * tell a level that sits on a rounding boundary from a wrong one.
 */
static void qsgd_scaled_values_impl(const float *v, int64_t n, int64_t d, int s,
                                    uint64_t seed, int worker, int64_t i0,
                                    int maxnorm, float *x_out)
{
    int64_t nbuckets = (n + d - 1) / d;
    uint64_t seed_w = seed ^ ((uint64_t)(uint32_t)worker << 48);
    for (int64_t b = 0; b < nbuckets; ++b) {
        int64_t lo = b * d;
        int64_t hi = lo + d < n ? lo + d : n;
        float norm = maxnorm ? max_abs(v + lo, hi - lo) : orc_l2norm_fp32(v + lo, hi - lo);
        float S = norm > 0.0f ? (float)s / norm : 0.0f;
        for (int64_t i = lo; i < hi; ++i) {
            if (norm > 0.0f) {
                float a = fabsf(v[i]) * S;
                float u = (float)orc_qsgd_dither(seed_w, (uint64_t)(i0 + i));
                x_out[i] = a + u;
            } else {
                x_out[i] = 0.0f;
            }
        }
    }
}

void orc_qsgd_scaled_values(const float *v, int64_t n, int64_t d, int s,
                            uint64_t seed, int worker, int64_t i0, float *x_out)
{
    qsgd_scaled_values_impl(v, n, d, s, seed, worker, i0, 0, x_out);
}

void orc_qsgd_scaled_values_maxnorm(const float *v, int64_t n, int64_t d, int s,
                                    uint64_t seed, int worker, int64_t i0,
                                    float *x_out)
{
    qsgd_scaled_values_impl(v, n, d, s, seed, worker, i0, 1, x_out);
}

/* Sign and level of element i from a code buffer written as above. */
static void qsgd_code_at(const uint8_t *codes, int64_t i, int s, int *sign,
                         int *level)
{
    if (s <= 7) {
        uint8_t byte = codes[i / 2];
        uint32_t c = (i % 2 == 0) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 15u);
        *sign = (int)(c >> 3);
        *level = (int)(c & 7u);
    } else {
        uint8_t c = codes[i];
        *sign = (int)(c >> 7);
        *level = (int)(c & 127u);
    }
}

/*
 * [QS] Knowl 2 (decode the (norm, sign, level) tuple: value = norm * sign *
 * level / s) and Knowl 3 (sum the K decoded messages; scale = 1/K gives the
 * average).  out[i] = scale * sum_w sgn * norm_{w,b} * level / s, in fp64.
 */
void orc_qsgd_dequant_sum(const uint8_t *const *codes, const float *const *norms,
                          int W, int64_t n, int64_t d, int s, double scale,
                          double *out)
{
    for (int64_t i = 0; i < n; ++i) {
        double sum = 0.0;
        for (int k = 0; k < W; ++k) {
            int sign, level;
            qsgd_code_at(codes[k], i, s, &sign, &level);
            double val = (double)norms[k][i / d] * (double)level / (double)s;
            sum += sign ? -val : val;
        }
        out[i] = scale * sum;
    }
}

/* ------------------------------------------------------------------------ */
/* [SA] SAPS sparsification, matching and peer averaging                    */
/* ------------------------------------------------------------------------ */

/*
 * [SA] section II-B: every worker draws the same Bernoulli(p) mask from the
 * round's shared seed; only masked coordinates are sent, as (index, value)
 * pairs.  Reading: m_i = [uniform(seed_t ^ i) < p].  Indices come out in
 * ascending order; every worker's value at each index is gathered.  Returns
 * the number of masked coordinates; at most `capacity` are written.  The
 * arrays may be a slice starting at global index i0 (indices are global).
 */
int64_t orc_saps_mask_compact(int64_t n, double p, uint64_t seed_t,
                              const double *const *models, int W, int64_t i0,
                              uint32_t *idx, double *const *vals,
                              int64_t capacity)
{
    int64_t K = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (orc_uniform(seed_t ^ (uint64_t)(i0 + i)) < p) {
            if (K < capacity) {
                idx[K] = (uint32_t)(i0 + i);
                for (int k = 0; k < W; ++k)
                    vals[k][K] = models[k][i];
            }
            ++K;
        }
    }
    return K;
}

/*
 * [SA] section II-C: single-peer gossip, each worker exchanges with exactly
 * one peer per round (a perfect matching; the gossip matrix then has two
 * nonzeros of 1/2 per row and is doubly stochastic).  The pages choose the
 * matching from measured link bandwidths; with no links here the matching is
 * a uniformly random one drawn from the round seed: a Fisher-Yates shuffle
 * with j = splitmix64(splitmix64(seed_t) ^ i) mod (i + 1) for i = W-1 .. 1,
 * then pairs (perm[0], perm[1]), (perm[2], perm[3]), ...
 * Returns 0, or -1 when W is not a positive even number.
 */
int orc_saps_matching(uint64_t seed_t, int W, int *pairs)
{
    if (W <= 0 || W % 2 != 0)
        return -1;
    for (int i = 0; i < W; ++i)
        pairs[i] = i;
    uint64_t base = orc_splitmix64(seed_t);
    for (int i = W - 1; i >= 1; --i) {
        int j = (int)(orc_splitmix64(base ^ (uint64_t)i) % (uint64_t)(i + 1));
        int tmp = pairs[i];
        pairs[i] = pairs[j];
        pairs[j] = tmp;
    }
    return 0;
}

/*
 * [SA] Algorithm 2 lines 9-10: each worker sends its sparsified model to its
 * peer and averages what it receives with its own copy.  On masked
 * coordinates both members of a pair end with (x_a + x_b) / 2; every other
 * coordinate is unchanged.  fp64.
 */
void orc_saps_peer_average(double *const *models, const double *const *vals,
                           const uint32_t *idx, int64_t K, const int *pairs,
                           int W)
{
    for (int q = 0; q < W / 2; ++q) {
        int a = pairs[2 * q];
        int b = pairs[2 * q + 1];
        for (int64_t k = 0; k < K; ++k) {
            double m = (vals[a][k] + vals[b][k]) / 2.0;
            models[a][idx[k]] = m;
            models[b][idx[k]] = m;
        }
    }
}

/*
 * [EA] EASGD, with no gradient term:
 *   w^k_{t+1} = w^k_t - alpha * (w^k_t - c_t)
 *   c_{t+1}   = (1 - beta) * c_t + beta * (1/K) sum_k w^k_t
 * Both right-hand sides use the values before the step.  fp64.
 */
void orc_easgd_step(double *const *models, int W, int64_t n, double alpha,
                    double beta, double *center)
{
    for (int64_t i = 0; i < n; ++i) {
        double sum = 0.0;
        for (int k = 0; k < W; ++k)
            sum += models[k][i];
        double mean = sum / (double)W;
        double c = center[i];
        for (int k = 0; k < W; ++k)
            models[k][i] = models[k][i] - alpha * (models[k][i] - c);
        center[i] = (1.0 - beta) * c + beta * mean;
    }
}

/*
 * [EA] the same two updates for one worker when the other workers' models
 * are only known through their elementwise sum (one process per worker):
 * mean = sum / W; model <- model - alpha (model - c); c <- (1-beta) c + beta mean.
 */
void orc_easgd_step_from_sum(double *model, const double *sum, int W, int64_t n,
                             double alpha, double beta, double *center)
{
    for (int64_t i = 0; i < n; ++i) {
        double mean = sum[i] / (double)W;
        double c = center[i];
        model[i] = model[i] - alpha * (model[i] - c);
        center[i] = (1.0 - beta) * c + beta * mean;
    }
}

/* ------------------------------------------------------------------------ */
/* [QS] Knowl 2: lossless Elias-omega coding of the (norm, sign, level)     */
/* tuple, dense regime ("offset Elias coding": Elias'(k) = Elias(k + 1)).    */
/* ------------------------------------------------------------------------ */

/*
 * Bit stream: bit k of the stream is bit (31 - k % 32) of word k / 32 (most
 * significant bit first).  Reading used for the format (the page gives the
 * tuple and the per-coordinate code, not the layout): every bucket starts on
 * a word boundary; it holds the 32 bits of its fp32 norm, then for each
 * coordinate in order Elias-omega(level + 1) followed by one sign bit
 * (1 = negative) when level > 0; unused bits of its last word are 0.
 * offsets[b] is the first word of bucket b, offsets[nbuckets] the total.
 */
typedef struct {
    uint32_t *words;
    int64_t pos; /* bit position */
} orc_bitwriter;

static void put_bit(orc_bitwriter *w, int bit)
{
    if (bit)
        w->words[w->pos / 32] |= 1u << (31 - (int)(w->pos % 32));
    w->pos++;
}

/*
 * Elias omega code of N >= 1 (Elias, "Universal codeword sets and
 * representations of the integers", IEEE Trans. Inf. Theory 21(2), 1975):
 * write the final 0; while N > 1, prepend the binary form of N and set N to
 * (its number of digits) - 1.
 */
int orc_elias_omega_bits(uint32_t N, char *out)
{
    char buf[64];
    int len = 0;
    buf[len++] = '0';
    while (N > 1) {
        char grp[33];
        int L = 0;
        for (uint32_t m = N; m; m >>= 1)
            grp[L++] = (char)('0' + (m & 1u));
        /* grp holds the digits least significant first; prepend reversed */
        memmove(buf + L, buf, (size_t)len);
        for (int i = 0; i < L; ++i)
            buf[i] = grp[L - 1 - i];
        len += L;
        N = (uint32_t)(L - 1);
    }
    memcpy(out, buf, (size_t)len);
    out[len] = '\0';
    return len;
}

static void put_omega(orc_bitwriter *w, uint32_t N)
{
    char bits[64];
    int len = orc_elias_omega_bits(N, bits);
    for (int i = 0; i < len; ++i)
        put_bit(w, bits[i] == '1');
}

/* Returns the total number of words. */
int64_t orc_qsgd_elias_encode(const uint8_t *codes, const float *norms, int64_t n,
                              int64_t d, int s, uint32_t *words, uint32_t *offsets)
{
    int64_t nbuckets = (n + d - 1) / d;
    orc_bitwriter w = {words, 0};
    for (int64_t b = 0; b < nbuckets; ++b) {
        offsets[b] = (uint32_t)(w.pos / 32);
        uint32_t nb;
        memcpy(&nb, &norms[b], sizeof nb);
        for (int i = 31; i >= 0; --i)
            put_bit(&w, (int)((nb >> i) & 1u));
        int64_t hi = (b + 1) * d < n ? (b + 1) * d : n;
        for (int64_t i = b * d; i < hi; ++i) {
            int sign, level;
            qsgd_code_at(codes, i, s, &sign, &level);
            put_omega(&w, (uint32_t)level + 1u);
            if (level > 0)
                put_bit(&w, sign);
        }
        w.pos = (w.pos + 31) / 32 * 32; /* next bucket on a word boundary */
    }
    offsets[nbuckets] = (uint32_t)(w.pos / 32);
    return w.pos / 32;
}

typedef struct {
    const uint32_t *words;
    int64_t pos;
} orc_bitreader;

static int get_bit(orc_bitreader *r)
{
    int bit = (int)((r->words[r->pos / 32] >> (31 - (int)(r->pos % 32))) & 1u);
    r->pos++;
    return bit;
}

static uint32_t get_omega(orc_bitreader *r)
{
    uint32_t N = 1;
    while (get_bit(r)) {
        uint32_t v = 1;
        for (uint32_t i = 0; i < N; ++i)
            v = 2 * v + (uint32_t)get_bit(r);
        N = v;
    }
    return N;
}

/*
 * Inverse of orc_qsgd_elias_encode.  Codes come back in the same
 * sign-magnitude layout; a level-0 coordinate carries no sign in the stream
 * and comes back with sign 0.
 */
void orc_qsgd_elias_decode(const uint32_t *words, const uint32_t *offsets, int64_t n,
                           int64_t d, int s, uint8_t *codes, float *norms)
{
    int64_t nbuckets = (n + d - 1) / d;
    if (s <= 7)
        for (int64_t k = 0; k < (n + 1) / 2; ++k)
            codes[k] = 0;
    for (int64_t b = 0; b < nbuckets; ++b) {
        orc_bitreader r = {words, (int64_t)offsets[b] * 32};
        uint32_t nb = 0;
        for (int i = 0; i < 32; ++i)
            nb = (nb << 1) | (uint32_t)get_bit(&r);
        memcpy(&norms[b], &nb, sizeof nb);
        int64_t hi = (b + 1) * d < n ? (b + 1) * d : n;
        for (int64_t i = b * d; i < hi; ++i) {
            uint32_t level = get_omega(&r) - 1u;
            uint32_t sign = level > 0 ? (uint32_t)get_bit(&r) : 0u;
            if (s <= 7) {
                uint32_t code = (sign << 3) | level;
                codes[i / 2] |= (uint8_t)(i % 2 == 0 ? code << 4 : code);
            } else {
                codes[i] = (uint8_t)((sign << 7) | level);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* [QS] Knowl 2, sparse regimes: only the non-zero coordinates are sent.    */
/* ------------------------------------------------------------------------ */

/*
 * Items 1 (s >= 2) and 1' (s = 1) of Knowl 2: the distances between
 * non-zero coordinates are coded with Elias omega.  Reading used for the
 * format (the page gives what is coded, not the layout), with the stream
 * conventions of the dense code above (most significant bit first, every
 * bucket on a word boundary, its fp32 norm first, an offsets table):
 *   for each coordinate i of the bucket (0-based within it) whose level is
 *   not 0, in order:  Elias-omega(i - p)  (p = the previous such i, or -1),
 *                     one sign bit (1 = negative),
 *                     Elias-omega(level)  (only when s >= 2; for s = 1 every
 *                                          sent level is 1);
 *   then Elias-omega(len - p) with len the bucket's length: the running
 *   position reaches len exactly, which ends the bucket.
 * A level-0 coordinate carries nothing and decodes with sign 0.
 */
int64_t orc_qsgd_elias_encode_sparse(const uint8_t *codes, const float *norms, int64_t n,
                                     int64_t d, int s, uint32_t *words, uint32_t *offsets)
{
    int64_t nbuckets = (n + d - 1) / d;
    orc_bitwriter w = {words, 0};
    for (int64_t b = 0; b < nbuckets; ++b) {
        offsets[b] = (uint32_t)(w.pos / 32);
        uint32_t nb;
        memcpy(&nb, &norms[b], sizeof nb);
        for (int i = 31; i >= 0; --i)
            put_bit(&w, (int)((nb >> i) & 1u));
        int64_t lo = b * d;
        int64_t len = (b + 1) * d < n ? d : n - lo;
        int64_t p = -1;
        for (int64_t i = 0; i < len; ++i) {
            int sign, level;
            qsgd_code_at(codes, lo + i, s, &sign, &level);
            if (level == 0)
                continue;
            put_omega(&w, (uint32_t)(i - p));
            put_bit(&w, sign);
            if (s >= 2)
                put_omega(&w, (uint32_t)level);
            p = i;
        }
        put_omega(&w, (uint32_t)(len - p));
        w.pos = (w.pos + 31) / 32 * 32;
    }
    offsets[nbuckets] = (uint32_t)(w.pos / 32);
    return w.pos / 32;
}

/*
 * Inverse of orc_qsgd_elias_encode_sparse.  Returns the number of buckets
 * whose distances overshoot the bucket (a stream this encoder did not
 * write); such a bucket keeps the coordinates decoded before the overshoot.
 */
int64_t orc_qsgd_elias_decode_sparse(const uint32_t *words, const uint32_t *offsets, int64_t n,
                                     int64_t d, int s, uint8_t *codes, float *norms)
{
    int64_t nbuckets = (n + d - 1) / d;
    int64_t bad = 0;
    int64_t nbytes = s <= 7 ? (n + 1) / 2 : n;
    for (int64_t k = 0; k < nbytes; ++k)
        codes[k] = 0;
    for (int64_t b = 0; b < nbuckets; ++b) {
        orc_bitreader r = {words, (int64_t)offsets[b] * 32};
        uint32_t nb = 0;
        for (int i = 0; i < 32; ++i)
            nb = (nb << 1) | (uint32_t)get_bit(&r);
        memcpy(&norms[b], &nb, sizeof nb);
        int64_t lo = b * d;
        int64_t len = (b + 1) * d < n ? d : n - lo;
        int64_t p = -1;
        for (;;) {
            p += (int64_t)get_omega(&r);
            if (p >= len) {
                if (p > len)
                    ++bad;
                break;
            }
            uint32_t sign = (uint32_t)get_bit(&r);
            uint32_t level = s >= 2 ? get_omega(&r) : 1u;
            int64_t i = lo + p;
            if (s <= 7) {
                uint32_t code = (sign << 3) | (level & 7u);
                codes[i / 2] |= (uint8_t)(i % 2 == 0 ? code << 4 : code);
            } else {
                codes[i] = (uint8_t)((sign << 7) | (level & 127u));
            }
        }
    }
    return bad;
}

/*
 * Side information for decoding a dense-regime bucket in parallel (not on
 * the pages; the per-bucket offsets table above is side information of the
 * same kind): marks[3b + k - 1], k = 1..3, is the bit offset, counted from
 * the first bit of bucket b's first word, at which the codeword of the
 * bucket's coordinate k d/4 starts; a quarter that starts past the bucket's
 * last coordinate (a short last bucket) gets the bucket's end.
 */
void orc_qsgd_elias_quarter_marks(const uint8_t *codes, int64_t n, int64_t d, int s,
                                  uint16_t *marks)
{
    int64_t nbuckets = (n + d - 1) / d;
    int64_t q = d / 4;
    for (int64_t b = 0; b < nbuckets; ++b) {
        int64_t lo = b * d;
        int64_t len = (b + 1) * d < n ? d : n - lo;
        int64_t pos = 32;
        for (int64_t i = 0; i < len; ++i) {
            if (i > 0 && i % q == 0)
                marks[3 * b + i / q - 1] = (uint16_t)pos;
            int sign, level;
            qsgd_code_at(codes, lo + i, s, &sign, &level);
            char bits[64];
            pos += orc_elias_omega_bits((uint32_t)level + 1u, bits) + (level > 0 ? 1 : 0);
        }
        for (int64_t k = 1; k <= 3; ++k)
            if (k * q >= len)
                marks[3 * b + k - 1] = (uint16_t)pos;
    }
}
