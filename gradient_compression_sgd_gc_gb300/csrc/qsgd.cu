// qsgd.cu -- QSGD bucketed stochastic quantisation and its dequantise-sum.
//
// Source: "QSGD: Communication-Efficient SGD via Gradient Quantization and
// Encoding" (summary page), Knowl 1 (operator Q_s), Knowl 2 (norm stored as
// a single-precision float, sign and level per coordinate), Knowl 3 (sum /
// average of the decoded messages), Knowl 8 (bucketing).
//
// One warp owns one bucket of d = 128 * ROUNDS elements; lane l reads the
// 16-byte vectors at bucket offsets 128j + 4l (j < ROUNDS), so the bucket is
// read from HBM exactly once and kept in registers between the norm and the
// quantisation.  The dequant-sum copies each warp's next buckets' codes to
// shared memory (cp.async) while it sums the current one, and turns codes
// into signed levels through per-lane copies of a table in shared memory.
#include <atomic>

#include "gc_common.cuh"

namespace gc {
namespace {

// Knuth's TwoSum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// Adds x*x to the double-float accumulator (hi, lo) without losing the
// rounding error of the square (x*x == p + q exactly).
__device__ __forceinline__ void acc_square(float x, float& hi, float& lo) {
    const float p = __fmul_rn(x, x);
    const float q = __fmaf_rn(x, x, -p);
    float s, e;
    two_sum(hi, p, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, q));
}

// Two fp32 lanes in one 64-bit register, for the packed (f32x2) arithmetic of
// sm_100+: one instruction does the same IEEE round-to-nearest operation on
// both halves.
__device__ __forceinline__ uint64_t pack2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// acc_square on two independent accumulators at once (the even and the odd
// elements of a pair): the same operations, each rounded as there.  The
// square is formed as fma(x, x, +0) (the same value as x*x): a packed multiply
// feeding the packed add of the TwoSum was measured to be contracted into one
// fma by the assembler, which loses the error term this sum relies on.
__device__ __forceinline__ void acc_square2(uint64_t x, uint64_t& hi, uint64_t& lo) {
    const uint64_t p = fma2(x, x, 0ull);
    const uint64_t q = fma2(x, x, sub2(0ull, p));     // x*x - p, exactly
    const uint64_t s = add2(hi, p);                    // TwoSum(hi, p)
    const uint64_t bp = sub2(s, hi);
    const uint64_t e = add2(sub2(hi, sub2(s, bp)), sub2(p, bp));
    hi = s;
    lo = add2(lo, add2(e, q));
}

// Sum of squares of a double-float pair over the warp (every lane gets it).
__device__ __forceinline__ void warp_sum2(float& hi, float& lo) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        float s, e;
        two_sum(hi, h2, s, e);
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, l2), e);
    }
}

// sqrt of the double-float X + Xl, rounded to nearest fp32.
// 1 / (2r) for the Newton correction below: the hardware reciprocal refined by
// one step of Newton's method for 1/x (relative error near 2^-24, which the correction -- itself
// at most half an ulp of r -- scales down to about 2^-48 of the result).
__device__ __forceinline__ float half_recip(float r) {
    float c0;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(c0) : "f"(r));
    c0 = __fmul_rn(0.5f, c0);
    const float e = __fmaf_rn(__fmul_rn(-2.0f, r), c0, 1.0f);
    return __fmaf_rn(c0, e, c0);
}

__device__ __forceinline__ float df_sqrt(float hi, float lo) {
    const float X = __fadd_rn(hi, lo);
    const float Xl = __fsub_rn(lo, __fsub_rn(X, hi));
    if (!(X > 0.0f)) return 0.0f;
    const float r = __fsqrt_rn(X);
    const float rem = __fadd_rn(__fmaf_rn(-r, r, X), Xl);     // X + Xl - r^2
    return __fmaf_rn(rem, half_recip(r), r);                  // r + rem / (2r)
}

// The bucket's l2 norm, rounded to nearest fp32 (equal to the correctly
// rounded value unless sqrt(sum) lies within about 2^-40 relative of a
// rounding midpoint).  Every lane returns the same value.
__device__ __forceinline__ float warp_norm(float hi, float lo) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        float s, e;
        two_sum(hi, h2, s, e);
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, l2), e);
    }
    return df_sqrt(hi, lo);
}

struct QArgs {
    const float* v;
    int64_t n;
    int64_t nbuckets;
    uint64_t seed_w;      // seed ^ (worker << 48)
    int s;
    float* norms;
    uint8_t* codes;
};

// level = min(floor(|v| * S + u), s) in fp32, u = (24-bit dither field) * 2^-24.
// u is an exact multiple of 2^-24, so one fma rounds |v|*S + u exactly as the
// separate add does.  The floor runs on the conversion pipe (round toward
// -inf to an unsigned integer; +inf saturates, so min() gives s); a NaN y
// (0 * inf: a zero coordinate in a bucket whose s / norm overflows) converts
// to 0, the level of a zero coordinate.
__device__ __forceinline__ uint32_t qlevel(float x, float S, uint32_t s, uint32_t top24) {
    const float a = __fmul_rn(fabsf(x), S);
    const float y = __fmaf_rn(__uint2float_rn(top24), 5.9604644775390625e-8f, a);
    return min(__float2uint_rd(y), s);
}

// The dither fields of one SplitMix64 output: z = splitmix64(key); the even
// element of the pair takes bits 40..63 of z, the odd one bits 8..31.
__device__ __forceinline__ void splitmix64_fields(uint64_t key, uint32_t& even, uint32_t& odd) {
    const uint64_t z = splitmix64(key);
    even = static_cast<uint32_t>(z >> 40);
    odd = (static_cast<uint32_t>(z) >> 8);
}

// Dither fields of four consecutive elements e .. e + 3 (e a multiple of 4):
// the pairs use the keys kbase = seed_w ^ (e / 2) and kbase ^ 1.  The two
// keys differ only in their low bit, so x_k = x0 + j_k with x0 = kbase & ~1
// and j_k = (kbase & 1) ^ k.  While z0 = x0 + golden has no carry out of its
// low word for j_k <= 1, both z have the same high word, and so does the
// high word of z ^ (z >> 30); its share of the first product is computed
// once.  A pair whose low word would carry takes the plain function (one in
// about 2^31).  Of the last product r = q * C2 the even field needs bits
// 40..63 (the final z ^ (z >> 31) leaves them as they are) and the odd field
// bits 8..31 of r ^ (r >> 31).
__device__ __forceinline__ void dither4_top24(uint64_t kbase, uint32_t (&t)[4]) {
    constexpr uint64_t kC1 = 0xBF58476D1CE4E5B9ull;
    constexpr uint64_t kC2 = 0x94D049BB133111EBull;
    const uint64_t z0 = (kbase & ~1ull) + 0x9E3779B97F4A7C15ull;
    const uint32_t z0l = static_cast<uint32_t>(z0), zh = static_cast<uint32_t>(z0 >> 32);
    const uint32_t jb = static_cast<uint32_t>(kbase) & 1u;
    if (z0l == 0xFFFFFFFFu) {
        splitmix64_fields(kbase, t[0], t[1]);
        splitmix64_fields(kbase ^ 1ull, t[2], t[3]);
        return;
    }
    const uint32_t yh = zh ^ (zh >> 30);                               // high word of z ^ (z >> 30)
    const uint64_t yh_part = static_cast<uint64_t>(yh * static_cast<uint32_t>(kC1)) << 32;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t zl = z0l + (jb ^ static_cast<uint32_t>(k));
        const uint32_t yl = zl ^ __funnelshift_r(zl, zh, 30);              // low word of z ^ (z >> 30)
        const uint64_t p = static_cast<uint64_t>(yl) * kC1 + yh_part;      // (yh:yl) * C1 mod 2^64
        const uint64_t q = p ^ (p >> 27);
        const uint64_t r = q * kC2;
        const uint32_t rl = static_cast<uint32_t>(r), rh = static_cast<uint32_t>(r >> 32);
        t[2 * k] = rh >> 8;
        t[2 * k + 1] = (rl ^ __funnelshift_r(rl, rh, 31)) >> 8;
    }
}

// True when every value of the warp's bucket registers is +-0.
template <int ROUNDS>
__device__ __forceinline__ bool all_zero(const float4 (&v)[ROUNDS], int lane) {
    bool nz = false;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) nz |= (v[j].x != 0.0f) | (v[j].y != 0.0f) | (v[j].z != 0.0f) | (v[j].w != 0.0f);
    return !__any_sync(0xffffffffu, nz);
}

// One bucket of one worker, by one warp: the bucket's norm (written by lane
// 0), its codes (written), and -- when SUM -- every element's dequantised
// term added to sum[j][k] exactly as k_qsgd_dequant_sum adds it (one fma of
// the level with the signed norm * unit_scale), so that a fused pass over
// all workers equals the quantise calls followed by the dequant-sum.
// Programmatic dependent launch: the fix-up kernels are launched with the
// programmatic-serialisation attribute, so they can be scheduled while the
// main kernel's last CTAs drain instead of after a full launch gap.  The
// main kernel allows it at its start; the fix-up waits (griddepcontrol.wait)
// until the main grid has completed and its writes are visible before it
// reads a norm.  Launched without the attribute, the wait returns at once.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// A sum of squares below 2^-100 may have lost bits to underflow and one above
// 2^126 overflows: such buckets (subnormal-sized or huge gradients) are redone
// with every value scaled by the power of two that brings the bucket maximum
// to [0.5, 1), which is exact, and the norm scaled back.
template <int ROUNDS>
__device__ __forceinline__ float rescued_norm(const float4 (&v)[ROUNDS]) {
    float mx = 0.0f;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j)
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int ex = 0;
    frexpf(mx, &ex);
    float h2 = 0.0f, l2 = 0.0f;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
        acc_square(ldexpf(v[j].x, -ex), h2, l2);
        acc_square(ldexpf(v[j].y, -ex), h2, l2);
        acc_square(ldexpf(v[j].z, -ex), h2, l2);
        acc_square(ldexpf(v[j].w, -ex), h2, l2);
    }
    warp_sum2(h2, l2);
    return ldexpf(df_sqrt(h2, l2), ex);
}

// The four sign bits of a float4 at bit 7 of each byte (element k in byte k),
// set where the value is below zero: +0 is added first (packed), which turns
// -0 into +0 and leaves every other number as it is, then the top byte of
// each float is picked out.  (A NaN never reaches here: its bucket is flagged.)
__device__ __forceinline__ uint32_t sign_bytes(const float4 x) {
    const uint64_t p01 = add2(pack2(x.x, x.y), 0ull), p23 = add2(pack2(x.z, x.w), 0ull);
    const uint32_t lo = __byte_perm(static_cast<uint32_t>(p01), static_cast<uint32_t>(p01 >> 32), 0x0073);
    const uint32_t hi = __byte_perm(static_cast<uint32_t>(p23), static_cast<uint32_t>(p23 >> 32), 0x0073);
    return __byte_perm(lo, hi, 0x5410) & 0x80808080u;
}

// One bucket of one worker, by one warp: the bucket's norm (written by lane
// 0), its codes (written), and -- when SUM -- every element's dequantised
// term added to sum[j][k] exactly as k_qsgd_dequant_sum adds it (one fma of
// the level with the signed norm * unit_scale), so that a fused pass over
// all workers equals the quantise calls followed by the dequant-sum.
// RAGGED: the partial last bucket (bounds-checked loads and stores).
// FLAG: a bucket whose l2 norm needs the rescue above is not finished here:
// its norm is written as -1 (no norm is negative) and a second, small kernel
// redoes it with FLAG off.  Keeping the rare path out of the main kernel
// measured 10% faster than carrying it inline or as a call.
template <int ROUNDS, bool FOUR, bool MAXNORM, bool SUM, bool RAGGED, bool FLAG>
__device__ __forceinline__ void quantize_bucket_body(const QArgs& a, int64_t b, int lane, float unit_scale,
                                                     float (&sum)[ROUNDS][4]) {
    constexpr int D = 128 * ROUNDS;
    constexpr uint32_t kSignShift = FOUR ? 3 : 7;
    const float s_f = static_cast<float>(a.s);
    const uint32_t s_u = static_cast<uint32_t>(a.s);

    const int64_t b0 = b * D;
    float4 v[ROUNDS];
    if (!RAGGED) {
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j) v[j] = ld_stream_f4(a.v + b0 + 128 * j + 4 * lane);
    } else {
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j) {
            const int64_t e = b0 + 128 * j + 4 * lane;
            v[j].x = e < a.n ? a.v[e] : 0.0f;
            v[j].y = e + 1 < a.n ? a.v[e + 1] : 0.0f;
            v[j].z = e + 2 < a.n ? a.v[e + 2] : 0.0f;
            v[j].w = e + 3 < a.n ? a.v[e + 3] : 0.0f;
        }
    }
    float norm;
    if (MAXNORM) {
        // QSGD Knowl 8 max-norm scaling: the bucket's largest |v| (exact)
        float mx = 0.0f;
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j)
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        norm = mx;
    } else {
        // two double-float accumulators (even and odd elements) in packed fp32
        // pairs, joined by one TwoSum: the same accuracy as one accumulator
        uint64_t hi2 = 0ull, lo2 = 0ull;
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j) {
            acc_square2(pack2(v[j].x, v[j].y), hi2, lo2);
            acc_square2(pack2(v[j].z, v[j].w), hi2, lo2);
        }
        float ha, hb, la, lb, hi, e;
        unpack2(hi2, ha, hb);
        unpack2(lo2, la, lb);
        two_sum(ha, hb, hi, e);
        const float lo = __fadd_rn(__fadd_rn(la, lb), e);
        norm = warp_norm(hi, lo);
        const bool tiny = norm < 8.8817842e-16f;      // 2^-50: the sum of squares is below 2^-100
        const bool huge = !(norm < 9.2233720e18f);    // 2^63, or inf / NaN
        if (huge || (tiny && !all_zero(v, lane))) {   // warp-uniform
            if (FLAG)
                norm = -1.0f;
            else
                norm = rescued_norm<ROUNDS>(v);
        }
    }
    if (lane == 0) a.norms[b] = norm;
    // norm == 0 means every coordinate is +-0: sign bit 0, level 0, code 0
    // (a flagged norm of -1 gives level 0 everywhere; the codes are rewritten)
    const bool zero = !(norm > 0.0f);
    const float S = zero ? 0.0f : __fdiv_rn(s_f, norm);

#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
        const int64_t e = b0 + 128 * j + 4 * lane;
        // e is a multiple of 4: elements e, e + 1 share the key seed_w ^ (e / 2),
        // elements e + 2, e + 3 the key seed_w ^ (e / 2 + 1) == (seed_w ^ (e / 2)) ^ 1
        const uint64_t kbase = a.seed_w ^ static_cast<uint64_t>(e >> 1);
        const float xs[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        uint32_t lv[4] = {0u, 0u, 0u, 0u};
        if (!zero) {
            uint32_t t[4];
            dither4_top24(kbase, t);
#pragma unroll
            for (int k = 0; k < 4; ++k) lv[k] = qlevel(xs[k], S, s_u, t[k]);
        }
        if (SUM) {
            const float u = __fmul_rn(norm, unit_scale);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float lf = __uint_as_float(0x4B000000u | lv[k]) - 8388608.0f;
                sum[j][k] = __fmaf_rn(lf, xs[k] < 0.0f ? -u : u, sum[j][k]);
            }
        }
        if (FOUR) {
            uint32_t c[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) c[k] = ((xs[k] < 0.0f ? 1u : 0u) << kSignShift) | lv[k];
            const uint32_t lo2 = (c[0] << 4) | c[1];
            const uint32_t hi2 = (c[2] << 4) | c[3];
            if (!RAGGED) {
                *reinterpret_cast<uint16_t*>(a.codes + (e >> 1)) = static_cast<uint16_t>(lo2 | (hi2 << 8));
            } else {
                if (e < a.n) a.codes[e >> 1] = static_cast<uint8_t>(e + 1 < a.n ? lo2 : (c[0] << 4));
                if (e + 2 < a.n) a.codes[(e >> 1) + 1] = static_cast<uint8_t>(e + 3 < a.n ? hi2 : (c[2] << 4));
            }
        } else {
            // levels into bytes (element k in byte k), sign bits from the floats
            const uint32_t L = __byte_perm(__byte_perm(lv[0], lv[1], 0x0040), __byte_perm(lv[2], lv[3], 0x0040), 0x5410);
            const uint32_t word = L | sign_bytes(v[j]);
            if (!RAGGED) {
                *reinterpret_cast<uint32_t*>(a.codes + e) = word;
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (e + k < a.n) a.codes[e + k] = static_cast<uint8_t>(word >> (8 * k));
            }
        }
    }
}

// One warp per whole bucket; the grid covers the whole buckets.  For buckets
// of up to 512 the register bound allows 6 CTAs (48 warps) per SM with no
// spills: the quantiser is bound by instruction issue and the integer ALU
// pipe, and 6 measured ahead of 4 (56 registers) and of 8 (32 registers and
// spills).  The partial last bucket and flagged buckets: k_qsgd_fixup.
template <int ROUNDS, bool FOUR, bool MAXNORM>
__global__ void __launch_bounds__(kThreads, ROUNDS >= 8 ? 2 : 6)
k_qsgd_quantize(const QArgs a) {
    constexpr int D = 128 * ROUNDS;
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= a.n / D) return;
    float unused[ROUNDS][4];
    quantize_bucket_body<ROUNDS, FOUR, MAXNORM, false, false, !MAXNORM>(a, b, lane, 0.0f, unused);
}

// After k_qsgd_quantize: the first warp does the partial last bucket, then
// each warp scans 32 norms at a time and redoes, with the rescue, every
// bucket flagged there (norm -1).
template <int ROUNDS, bool FOUR, bool MAXNORM>
__global__ void __launch_bounds__(kThreads)
k_qsgd_fixup(const QArgs a) {
    constexpr int D = 128 * ROUNDS;
    const int lane = threadIdx.x & 31;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t nfull = a.n / D;
    float unused[ROUNDS][4];
    // the partial last bucket touches nothing the main kernel writes: done
    // before waiting for it
    if (gw == 0 && nfull * D < a.n)
        quantize_bucket_body<ROUNDS, FOUR, MAXNORM, false, true, false>(a, nfull, lane, 0.0f, unused);
    wait_for_primary();
    if (!MAXNORM) {
        for (int64_t g0 = gw * 32; g0 < nfull; g0 += nw * 32) {
            const int64_t b = g0 + lane;
            uint32_t m = __ballot_sync(0xffffffffu, b < nfull && a.norms[b] < 0.0f);
            while (m) {
                const int i = __ffs(m) - 1;
                m &= m - 1;
                quantize_bucket_body<ROUNDS, FOUR, false, false, false, false>(a, g0 + i, lane, 0.0f, unused);
            }
        }
    }
}

// Every worker's quantisation and the dequant-sum in one pass: one warp per
// bucket runs the W workers in order and keeps the sum in registers.
struct StepArgs {
    PtrTable<const float*> v;
    PtrTable<float*> norms;
    PtrTable<uint8_t*> codes;
    QArgs q;              // per-worker fields (v, seed_w, norms, codes) set in the loop
    int W;
    uint64_t seed;
    float unit_scale;
    float* out;
};

// All workers' quantisation of bucket b and the sum of their terms, written
// to out (FLAG and RAGGED as in quantize_bucket_body).
template <int ROUNDS, bool FOUR, bool MAXNORM, bool RAGGED, bool FLAG>
__device__ __forceinline__ void step_bucket(const StepArgs& a, int64_t b, int lane) {
    constexpr int D = 128 * ROUNDS;
    float sum[ROUNDS][4];
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) sum[j][k] = 0.0f;
    for (int w = 0; w < a.W; ++w) {
        QArgs q = a.q;
        q.v = a.v.p[w];
        q.seed_w = a.seed ^ (static_cast<uint64_t>(static_cast<uint32_t>(w)) << 48);
        q.norms = a.norms.p[w];
        q.codes = a.codes.p[w];
        quantize_bucket_body<ROUNDS, FOUR, MAXNORM, true, RAGGED, FLAG>(q, b, lane, a.unit_scale, sum);
    }
    const int64_t b0 = b * D;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
        const int64_t e = b0 + 128 * j + 4 * lane;
        const float4 o = make_float4(sum[j][0], sum[j][1], sum[j][2], sum[j][3]);
        if (!RAGGED) {
            st_stream_f4(a.out + e, o);
        } else {
            if (e < a.q.n) a.out[e] = o.x;
            if (e + 1 < a.q.n) a.out[e + 1] = o.y;
            if (e + 2 < a.q.n) a.out[e + 2] = o.z;
            if (e + 3 < a.q.n) a.out[e + 3] = o.w;
        }
    }
}

template <int ROUNDS, bool FOUR, bool MAXNORM>
__global__ void __launch_bounds__(kThreads, ROUNDS >= 8 ? 2 : 4)
k_qsgd_step(const StepArgs a) {
    constexpr int D = 128 * ROUNDS;
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= a.q.n / D) return;
    step_bucket<ROUNDS, FOUR, MAXNORM, false, !MAXNORM>(a, b, lane);
}

// After k_qsgd_step: the first warp does the partial last bucket, then every
// bucket in which some worker was flagged is redone for all workers (norms,
// codes and the sum).
template <int ROUNDS, bool FOUR, bool MAXNORM>
__global__ void __launch_bounds__(kThreads)
k_qsgd_step_fixup(const StepArgs a) {
    constexpr int D = 128 * ROUNDS;
    const int lane = threadIdx.x & 31;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t nfull = a.q.n / D;
    if (gw == 0 && nfull * D < a.q.n) step_bucket<ROUNDS, FOUR, MAXNORM, true, false>(a, nfull, lane);
    wait_for_primary();
    if (!MAXNORM) {
        for (int64_t g0 = gw * 32; g0 < nfull; g0 += nw * 32) {
            const int64_t b = g0 + lane;
            bool f = false;
            if (b < nfull)
                for (int w = 0; w < a.W; ++w) f |= a.norms.p[w][b] < 0.0f;
            uint32_t m = __ballot_sync(0xffffffffu, f);
            while (m) {
                const int i = __ffs(m) - 1;
                m &= m - 1;
                step_bucket<ROUNDS, FOUR, false, false, false>(a, g0 + i, lane);
            }
        }
    }
}

struct DArgs {
    PtrTable<const uint8_t*> codes;
    PtrTable<const float*> norms;
    int W;
    int64_t n;
    int64_t nbuckets;
    float unit_scale;     // scale / s, rounded once to fp32
    float* out;
};

// Raw code bits of elements e..e+3 (e a multiple of 4): 16 bits for 4-bit
// codes (byte e/2 in bits 0-7, byte e/2+1 in bits 8-15), 32 bits for 8-bit.
template <bool FOUR>
__device__ __forceinline__ uint32_t load_raw4(const uint8_t* codes, int64_t e, int64_t n, bool full) {
    if (FOUR) {
        if (full) return __ldg(reinterpret_cast<const uint16_t*>(codes + (e >> 1)));
        return (e < n ? codes[e >> 1] : 0u) | ((e + 2 < n ? codes[(e >> 1) + 1] : 0u) << 8);
    }
    if (full) return __ldg(reinterpret_cast<const uint32_t*>(codes + e));
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (e + k < n) w |= static_cast<uint32_t>(codes[e + k]) << (8 * k);
    return w;
}

// Code-to-level tables in shared memory, one row of 128 bytes per code byte c
// and a copy per lane so that a warp's table loads never meet in a bank:
// 8-bit codes: row c = 32 floats, the signed level (-1)^sign * level of c;
// 4-bit codes: row c = 16 float2, the signed levels of c's two codes (high
// nibble first), one copy per half-warp lane (a half-warp's 64-bit loads
// cover the 32 banks once).  Lane l reads entry c at lane_base(l) + 128 c.
constexpr int kLevelTableBytes = 256 * 128;

template <bool FOUR>
__device__ __forceinline__ void fill_level_table(float* tab) {
    for (int i = threadIdx.x; i < kLevelTableBytes / 4; i += blockDim.x) {
        const int c = i >> 5;
        const int code = FOUR ? ((i & 1) ? (c & 15) : (c >> 4)) : c;
        const float l = static_cast<float>(code & (FOUR ? 7 : 127));
        tab[i] = (code & (FOUR ? 8 : 128)) ? -l : l;
    }
}

template <bool FOUR>
__device__ __forceinline__ const char* level_lane_base(const float* tab, int lane) {
    return reinterpret_cast<const char*>(tab) + (FOUR ? 8 * (lane & 15) : 4 * lane);
}

// Signed levels of the four codes in `raw` (load_raw4's layout) as two
// float2 pairs (codes 0,1 and 2,3).
template <bool FOUR>
__device__ __forceinline__ void levels4(uint32_t raw, const char* lane_base, uint64_t& l01, uint64_t& l23) {
    if (FOUR) {
        l01 = *reinterpret_cast<const uint64_t*>(lane_base + ((raw & 255u) << 7));
        l23 = *reinterpret_cast<const uint64_t*>(lane_base + (((raw >> 8) & 255u) << 7));
    } else {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            v[k] = *reinterpret_cast<const float*>(lane_base + (__byte_perm(raw, 0u, 0x4440 | k) << 7));
        l01 = pack2(v[0], v[1]);
        l23 = pack2(v[2], v[3]);
    }
}

// Writes the sums of elements e..e+3 (e = b*D + 128j + 4*lane), clipped to n.
__device__ __forceinline__ void store_sum4(float* out, int64_t e, int64_t n, bool full, uint64_t s01, uint64_t s23) {
    float4 o;
    unpack2(s01, o.x, o.y);
    unpack2(s23, o.z, o.w);
    if (full) {
        st_stream_f4(out + e, o);
    } else {
        if (e < n) out[e] = o.x;
        if (e + 1 < n) out[e + 1] = o.y;
        if (e + 2 < n) out[e + 2] = o.z;
        if (e + 3 < n) out[e + 3] = o.w;
    }
}

// One bucket by one warp, codes read straight from global memory: every
// worker's code and norm loads issued together (WC at a time), then the
// sum.  Each element's sum runs in worker order, each term added by one fma
// of the signed level with norm * (scale / s) (packed: two elements per
// instruction, each rounded as alone).
template <int ROUNDS, bool FOUR>
__device__ __forceinline__ void dequant_bucket_direct(const DArgs& a, int64_t b, int lane, const char* lane_base) {
    constexpr int WC = ROUNDS >= 8 ? 2 : 4;
    constexpr int D = 128 * ROUNDS;
    uint64_t sum[ROUNDS][2];
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) sum[j][0] = sum[j][1] = 0ull;
    const bool full = (b + 1) * D <= a.n;
    for (int w0 = 0; w0 < a.W; w0 += WC) {
        uint32_t raw[WC][ROUNDS];
        float unit[WC];
#pragma unroll
        for (int q = 0; q < WC; ++q) {
            if (w0 + q < a.W) {
                unit[q] = __ldg(a.norms.p[w0 + q] + b);
#pragma unroll
                for (int j = 0; j < ROUNDS; ++j)
                    raw[q][j] = load_raw4<FOUR>(a.codes.p[w0 + q], b * D + 128 * j + 4 * lane, a.n, full);
            }
        }
#pragma unroll
        for (int q = 0; q < WC; ++q) {
            if (w0 + q < a.W) {
                const float u = __fmul_rn(unit[q], a.unit_scale);
                const uint64_t uu = pack2(u, u);
#pragma unroll
                for (int j = 0; j < ROUNDS; ++j) {
                    uint64_t l01, l23;
                    levels4<FOUR>(raw[q][j], lane_base, l01, l23);
                    sum[j][0] = fma2(l01, uu, sum[j][0]);
                    sum[j][1] = fma2(l23, uu, sum[j][1]);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) store_sum4(a.out, b * D + 128 * j + 4 * lane, a.n, full, sum[j][0], sum[j][1]);
}

// Persistent grid (as many CTAs as fit on the GPU at once): each warp strides
// over the buckets, so a CTA fills its level table once.
template <int ROUNDS, bool FOUR>
__global__ void __launch_bounds__(kThreads, ROUNDS >= 8 ? 2 : 4) k_qsgd_dequant_sum(const DArgs a) {
    __shared__ __align__(16) float s_tab[kLevelTableBytes / 4];
    fill_level_table<FOUR>(s_tab);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const char* lane_base = level_lane_base<FOUR>(s_tab, lane);
    const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; b < a.nbuckets; b += stride)
        dequant_bucket_direct<ROUNDS, FOUR>(a, b, lane, lane_base);
}

// Asynchronous 16- and 4-byte copies global -> shared (sm_80+ cp.async), in
// per-thread commit groups.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The pipelined dequant-sum: a warp's work is a sequence of units (bucket b,
// group of up to PipeWG workers); the codes and norms of unit u + kPipeStages
// - 1 are copied to the warp's shared stage while unit u is summed from its
// own.  Position is kept in running counters (no division).  Only whole
// buckets go through the pipeline; the ragged last one is summed directly.
constexpr int kPipeStages = 3;

template <int ROUNDS, bool FOUR>
__host__ __device__ constexpr int pipe_bytes_per_worker() { return FOUR ? 64 * ROUNDS : 128 * ROUNDS; }

// workers staged together: 4, or fewer so that a stage holds at most 2 KB of codes
template <int ROUNDS, bool FOUR>
__host__ __device__ constexpr int pipe_group() {
    return 4 * pipe_bytes_per_worker<ROUNDS, FOUR>() <= 2048 ? 4
           : (2048 / pipe_bytes_per_worker<ROUNDS, FOUR>() > 0 ? 2048 / pipe_bytes_per_worker<ROUNDS, FOUR>() : 1);
}

template <int ROUNDS, bool FOUR>
__host__ __device__ constexpr int pipe_smem_bytes() {
    return kLevelTableBytes +
           kWarpsPerBlock * kPipeStages * pipe_group<ROUNDS, FOUR>() * (pipe_bytes_per_worker<ROUNDS, FOUR>() + 4);
}

template <int ROUNDS, bool FOUR>
__global__ void __launch_bounds__(kThreads, ROUNDS >= 8 ? 2 : 4) k_qsgd_dequant_pipe(const DArgs a) {
    constexpr int D = 128 * ROUNDS;
    constexpr int BPW = pipe_bytes_per_worker<ROUNDS, FOUR>();
    constexpr int CH = BPW / 16;                                  // 16-byte copies per worker
    constexpr int S = kPipeStages, WG = pipe_group<ROUNDS, FOUR>();
    constexpr int IT = (WG * CH + 31) / 32;                       // copies per lane per unit
    extern __shared__ __align__(16) unsigned char dsm[];
    float* s_tab = reinterpret_cast<float*>(dsm);
    fill_level_table<FOUR>(s_tab);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned char* s_stage = dsm + kLevelTableBytes + warp * (S * WG * BPW);
    float* s_norm = reinterpret_cast<float*>(dsm + kLevelTableBytes + kWarpsPerBlock * S * WG * BPW) + warp * S * WG;
    const char* lane_base = level_lane_base<FOUR>(s_tab, lane);
    const int G = (a.W + WG - 1) / WG;
    const int64_t nfull = a.n / D;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    int64_t pb = wid;        // producer: next unit to copy
    int pg = 0, pst = 0;
    auto issue = [&]() {
        if (pb < nfull) {
            const int nq = a.W - pg * WG < WG ? a.W - pg * WG : WG;
            const int64_t boff = pb * BPW;
            unsigned char* dst = s_stage + pst * (WG * BPW);
#pragma unroll
            for (int it = 0; it < IT; ++it) {
                const int c = lane + 32 * it;
                const int q = c / CH, k = c % CH;
                if (q < nq) cp_async16(dst + q * BPW + 16 * k, a.codes.p[pg * WG + q] + boff + 16 * k);
            }
            if (lane < nq) cp_async4(s_norm + pst * WG + lane, a.norms.p[pg * WG + lane] + pb);
            if (++pg == G) {
                pg = 0;
                pb += nw;
            }
            pst = pst + 1 == S ? 0 : pst + 1;
        }
        cp_async_commit();     // an empty group past the end keeps the count uniform
    };
#pragma unroll
    for (int u = 0; u < S - 1; ++u) issue();
    uint64_t sum[ROUNDS][2];
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) sum[j][0] = sum[j][1] = 0ull;
    int cg = 0, cst = 0;     // consumer: the unit being summed
    for (int64_t cb = wid; cb < nfull;) {
        issue();
        cp_async_wait<S - 1>();     // this lane's copies of unit (cb, cg) have landed
        __syncwarp();               // ... and every lane's
        const int nq = a.W - cg * WG < WG ? a.W - cg * WG : WG;
        const unsigned char* sbuf = s_stage + cst * (WG * BPW);
#pragma unroll
        for (int q = 0; q < WG; ++q) {
            if (q < nq) {
                const float un = __fmul_rn(s_norm[cst * WG + q], a.unit_scale);
                const uint64_t uu = pack2(un, un);
#pragma unroll
                for (int j = 0; j < ROUNDS; ++j) {
                    const unsigned char* p = sbuf + q * BPW + (FOUR ? 64 * j + 2 * lane : 128 * j + 4 * lane);
                    const uint32_t raw = FOUR ? *reinterpret_cast<const uint16_t*>(p) : *reinterpret_cast<const uint32_t*>(p);
                    uint64_t l01, l23;
                    levels4<FOUR>(raw, lane_base, l01, l23);
                    sum[j][0] = fma2(l01, uu, sum[j][0]);
                    sum[j][1] = fma2(l23, uu, sum[j][1]);
                }
            }
        }
        if (++cg == G) {
#pragma unroll
            for (int j = 0; j < ROUNDS; ++j) {
                store_sum4(a.out, cb * D + 128 * j + 4 * lane, a.n, true, sum[j][0], sum[j][1]);
                sum[j][0] = sum[j][1] = 0ull;
            }
            cg = 0;
            cb += nw;
        }
        cst = cst + 1 == S ? 0 : cst + 1;
        __syncwarp();               // the stage is read before it is refilled
    }
    cp_async_wait<0>();
    if (nfull < a.nbuckets && wid == nfull % nw) dequant_bucket_direct<ROUNDS, FOUR>(a, nfull, lane, lane_base);
}

// Launches a fix-up kernel after the kernel just enqueued on s, as a
// programmatic dependent launch (see wait_for_primary).
template <typename Args>
cudaError_t launch_after(void (*kernel)(Args), unsigned grid, cudaStream_t s, const Args& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// The fix-up grid: one warp per 32 whole buckets (their norms scanned with
// one coalesced load), at most two CTAs per SM; one CTA when only the
// partial last bucket can need it (max-norm scaling flags nothing).
inline unsigned fixup_grid(int64_t nfull, bool flags) {
    if (!flags) return 1u;
    const int64_t want = (nfull / 32 + kWarpsPerBlock) / kWarpsPerBlock;
    const int64_t cap = grid_for(2) > 0 ? grid_for(2) : 1;
    return static_cast<unsigned>(want < cap ? want : cap);
}

template <int ROUNDS, bool FOUR, bool MAXNORM>
int launch_quantize_r(const QArgs& a, cudaStream_t s) {
    constexpr int D = 128 * ROUNDS;
    const int64_t nfull = a.n / D;
    if (nfull > 0) k_qsgd_quantize<ROUNDS, FOUR, MAXNORM><<<blocks_for_tiles(nfull), kThreads, 0, s>>>(a);
    if (!MAXNORM || nfull * D < a.n) {
        if (launch_after<QArgs>(k_qsgd_fixup<ROUNDS, FOUR, MAXNORM>, fixup_grid(nfull, !MAXNORM), s, a) != cudaSuccess)
            return GC_ERR_CUDA;
    }
    return launch_status();
}

template <bool FOUR, bool MAXNORM>
int launch_quantize(int rounds, const QArgs& a, cudaStream_t s) {
    switch (rounds) {
        case 1: return launch_quantize_r<1, FOUR, MAXNORM>(a, s);
        case 2: return launch_quantize_r<2, FOUR, MAXNORM>(a, s);
        case 4: return launch_quantize_r<4, FOUR, MAXNORM>(a, s);
        case 8: return launch_quantize_r<8, FOUR, MAXNORM>(a, s);
        case 16: return launch_quantize_r<16, FOUR, MAXNORM>(a, s);
        default: return GC_ERR_INVALID;
    }
}

template <int ROUNDS, bool FOUR, bool MAXNORM>
int launch_step_r(const StepArgs& a, cudaStream_t s) {
    constexpr int D = 128 * ROUNDS;
    const int64_t nfull = a.q.n / D;
    if (nfull > 0) k_qsgd_step<ROUNDS, FOUR, MAXNORM><<<blocks_for_tiles(nfull), kThreads, 0, s>>>(a);
    if (!MAXNORM || nfull * D < a.q.n) {
        if (launch_after<StepArgs>(k_qsgd_step_fixup<ROUNDS, FOUR, MAXNORM>, fixup_grid(nfull, !MAXNORM), s, a) !=
            cudaSuccess)
            return GC_ERR_CUDA;
    }
    return launch_status();
}

template <bool FOUR, bool MAXNORM>
int launch_step(int rounds, const StepArgs& a, cudaStream_t s) {
    switch (rounds) {
        case 1: return launch_step_r<1, FOUR, MAXNORM>(a, s);
        case 2: return launch_step_r<2, FOUR, MAXNORM>(a, s);
        case 4: return launch_step_r<4, FOUR, MAXNORM>(a, s);
        case 8: return launch_step_r<8, FOUR, MAXNORM>(a, s);
        case 16: return launch_step_r<16, FOUR, MAXNORM>(a, s);
        default: return GC_ERR_INVALID;
    }
}

constexpr int kMaxDevices = 64;

// The resident grid of the pipelined kernel on the current device; the first
// call on a device also raises the kernel's dynamic shared-memory limit there.
template <int ROUNDS, bool FOUR>
int pipe_resident_ctas(int64_t* resident) {
    static std::atomic<int64_t> cached[kMaxDevices];     // CTAs; 0 = not yet known
    constexpr int dyn = pipe_smem_bytes<ROUNDS, FOUR>();
    auto kern = k_qsgd_dequant_pipe<ROUNDS, FOUR>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GC_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) {
        const int64_t c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *resident = c;
            return GC_OK;
        }
    }
    int sms = 0, per_sm = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, dyn) != cudaSuccess)
        return GC_ERR_CUDA;
    *resident = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    if (dev >= 0 && dev < kMaxDevices) cached[dev].store(*resident, std::memory_order_relaxed);
    return GC_OK;
}

template <int ROUNDS, bool FOUR>
int launch_dequant_pipe(const DArgs& a, cudaStream_t s) {
    int64_t resident = 0;
    const int rc = pipe_resident_ctas<ROUNDS, FOUR>(&resident);
    if (rc != GC_OK) return rc;
    const int64_t want = blocks_for_tiles(a.nbuckets);
    k_qsgd_dequant_pipe<ROUNDS, FOUR><<<static_cast<unsigned>(want < resident ? want : resident), kThreads,
                                        pipe_smem_bytes<ROUNDS, FOUR>(), s>>>(a);
    return launch_status();
}

template <int ROUNDS, bool FOUR>
int launch_dequant_rounds(const DArgs& a, cudaStream_t s) {
    // 4-bit codes, and 8-bit codes of 8 or more workers, go through the
    // copy pipeline; 8-bit codes of fewer workers are read directly, which
    // keeps four CTAs per SM.  Measured on 61 M coordinates of 8-bit codes:
    // 4 workers, direct 83 us, pipeline 88 us; 8 workers, direct 134 us,
    // pipeline 116 us.
    if constexpr (FOUR) {
        return launch_dequant_pipe<ROUNDS, FOUR>(a, s);
    } else {
        if (a.W >= 8) return launch_dequant_pipe<ROUNDS, FOUR>(a, s);
        return launch_persistent(k_qsgd_dequant_sum<ROUNDS, FOUR>, blocks_for_tiles(a.nbuckets), s, a);
    }
}

template <bool FOUR>
int launch_dequant(int rounds, const DArgs& a, cudaStream_t s) {
    switch (rounds) {
        case 1: return launch_dequant_rounds<1, FOUR>(a, s);
        case 2: return launch_dequant_rounds<2, FOUR>(a, s);
        case 4: return launch_dequant_rounds<4, FOUR>(a, s);
        case 8: return launch_dequant_rounds<8, FOUR>(a, s);
        case 16: return launch_dequant_rounds<16, FOUR>(a, s);
        default: return GC_ERR_INVALID;
    }
}

bool valid_bucket(int bucket) {
    return bucket == 128 || bucket == 256 || bucket == 512 || bucket == 1024 || bucket == 2048;
}

}  // namespace
}  // namespace gc

using namespace gc;

extern "C" {

static int qsgd_quantize_impl(const float* grad, int64_t n, int bucket, int s_levels, uint64_t seed,
                              int worker, float* norms, uint8_t* codes, gc_stream_t stream, bool maxnorm) {
    if (n < 0 || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127 || worker < 0)
        return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!grad || !norms || !codes) return GC_ERR_INVALID;
    if (!aligned16(grad) || !aligned16(norms) || !aligned16(codes)) return GC_ERR_ALIGN;
    QArgs a;
    a.v = grad;
    a.n = n;
    a.nbuckets = (n + bucket - 1) / bucket;
    a.seed_w = seed ^ (static_cast<uint64_t>(static_cast<uint32_t>(worker)) << 48);
    a.s = s_levels;
    a.norms = norms;
    a.codes = codes;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (maxnorm)
        return s_levels <= 7 ? launch_quantize<true, true>(bucket / 128, a, s)
                             : launch_quantize<false, true>(bucket / 128, a, s);
    return s_levels <= 7 ? launch_quantize<true, false>(bucket / 128, a, s)
                         : launch_quantize<false, false>(bucket / 128, a, s);
}

int qsgd_quantize(const float* grad, int64_t n, int bucket, int s_levels, uint64_t seed, int worker,
                  float* norms, uint8_t* codes, gc_stream_t stream) {
    return qsgd_quantize_impl(grad, n, bucket, s_levels, seed, worker, norms, codes, stream, false);
}

int qsgd_quantize_maxnorm(const float* grad, int64_t n, int bucket, int s_levels, uint64_t seed, int worker,
                          float* scales, uint8_t* codes, gc_stream_t stream) {
    return qsgd_quantize_impl(grad, n, bucket, s_levels, seed, worker, scales, codes, stream, true);
}

int qsgd_dequant_sum(const uint8_t* const* codes, const float* const* norms, int W, int64_t n,
                     int bucket, int s_levels, float scale, float* out, gc_stream_t stream) {
    if (n < 0 || W < 1 || W > GC_MAX_WORKERS || !valid_bucket(bucket) || s_levels < 1 ||
        s_levels > 127 || !isfinite(scale))
        return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!codes || !norms || !out) return GC_ERR_INVALID;
    DArgs a;
    for (int w = 0; w < W; ++w) {
        if (!codes[w] || !norms[w]) return GC_ERR_INVALID;
        if (!aligned16(codes[w]) || !aligned16(norms[w])) return GC_ERR_ALIGN;
        a.codes.p[w] = codes[w];
        a.norms.p[w] = norms[w];
    }
    if (!aligned16(out)) return GC_ERR_ALIGN;
    a.W = W;
    a.n = n;
    a.nbuckets = (n + bucket - 1) / bucket;
    a.unit_scale = static_cast<float>(static_cast<double>(scale) / s_levels);
    a.out = out;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return s_levels <= 7 ? launch_dequant<true>(bucket / 128, a, s)
                         : launch_dequant<false>(bucket / 128, a, s);
}

int qsgd_step(const float* const* grads, int W, int64_t n, int bucket, int s_levels, uint64_t seed,
              int maxnorm, float* const* norms, uint8_t* const* codes, float scale, float* out,
              gc_stream_t stream) {
    if (n < 0 || W < 1 || W > GC_MAX_WORKERS || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127 ||
        !isfinite(scale) || (maxnorm != 0 && maxnorm != 1))
        return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!grads || !norms || !codes || !out) return GC_ERR_INVALID;
    StepArgs a;
    for (int w = 0; w < W; ++w) {
        if (!grads[w] || !norms[w] || !codes[w]) return GC_ERR_INVALID;
        if (!aligned16(grads[w]) || !aligned16(norms[w]) || !aligned16(codes[w])) return GC_ERR_ALIGN;
        a.v.p[w] = grads[w];
        a.norms.p[w] = norms[w];
        a.codes.p[w] = codes[w];
    }
    if (!aligned16(out)) return GC_ERR_ALIGN;
    a.q.v = nullptr;
    a.q.n = n;
    a.q.nbuckets = (n + bucket - 1) / bucket;
    a.q.seed_w = 0;
    a.q.s = s_levels;
    a.q.norms = nullptr;
    a.q.codes = nullptr;
    a.W = W;
    a.seed = seed;
    a.unit_scale = static_cast<float>(static_cast<double>(scale) / s_levels);
    a.out = out;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (maxnorm)
        return s_levels <= 7 ? launch_step<true, true>(bucket / 128, a, s)
                             : launch_step<false, true>(bucket / 128, a, s);
    return s_levels <= 7 ? launch_step<true, false>(bucket / 128, a, s)
                         : launch_step<false, false>(bucket / 128, a, s);
}

}  // extern "C"
