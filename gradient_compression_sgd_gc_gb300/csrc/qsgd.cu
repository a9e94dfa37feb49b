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
// quantisation.
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
__device__ __forceinline__ float df_sqrt(float hi, float lo) {
    const float X = __fadd_rn(hi, lo);
    const float Xl = __fsub_rn(lo, __fsub_rn(X, hi));
    if (!(X > 0.0f)) return 0.0f;
    const float r = __fsqrt_rn(X);
    const float rem = __fadd_rn(__fmaf_rn(-r, r, X), Xl);     // X + Xl - r^2
    return __fmaf_rn(rem, __fdiv_rn(0.5f, r), r);             // r + rem / (2r)
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
    const float X = __fadd_rn(hi, lo);
    const float Xl = __fsub_rn(lo, __fsub_rn(X, hi));
    if (!(X > 0.0f)) return 0.0f;
    const float r = __fsqrt_rn(X);
    const float rem = __fadd_rn(__fmaf_rn(-r, r, X), Xl);     // X + Xl - r^2
    return __fmaf_rn(rem, __fdiv_rn(0.5f, r), r);             // r + rem / (2r)
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

// level = min(floor(|v| * S + u), s) in fp32, u = top24(hash) * 2^-24.
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

// splitmix64_top24 of the four keys kbase ^ k (k = 0..3), sharing what the
// four have in common: they differ only in their low two bits, so
// x_k = x0 + j_k with x0 = kbase & ~3 and j_k = (kbase & 3) ^ k.  While
// z0 = x0 + golden has no carry out of its low word for j_k <= 3, the four z
// have the same high word, and so does the high word of z ^ (z >> 30); its
// share of the first product is computed once.  A group whose low word would
// carry takes the plain function (one group in about 2^30).
__device__ __forceinline__ void hash4_top24(uint64_t kbase, uint32_t (&t)[4]) {
    constexpr uint64_t kC1 = 0xBF58476D1CE4E5B9ull;
    constexpr uint64_t kC2 = 0x94D049BB133111EBull;
    const uint64_t z0 = (kbase & ~3ull) + 0x9E3779B97F4A7C15ull;
    const uint32_t z0l = static_cast<uint32_t>(z0), zh = static_cast<uint32_t>(z0 >> 32);
    const uint32_t jb = static_cast<uint32_t>(kbase) & 3u;
    if (z0l > 0xFFFFFFFCu) {
#pragma unroll
        for (int k = 0; k < 4; ++k) t[k] = splitmix64_top24(kbase ^ static_cast<uint64_t>(k));
        return;
    }
    const uint32_t yh = zh ^ (zh >> 30);                               // high word of z ^ (z >> 30)
    const uint64_t yh_part = static_cast<uint64_t>(yh * static_cast<uint32_t>(kC1)) << 32;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t zl = z0l + (jb ^ static_cast<uint32_t>(k));
        const uint32_t yl = zl ^ __funnelshift_r(zl, zh, 30);              // low word of z ^ (z >> 30)
        const uint64_t p = static_cast<uint64_t>(yl) * kC1 + yh_part;      // (yh:yl) * C1 mod 2^64
        const uint64_t q = p ^ (p >> 27);
        t[k] = static_cast<uint32_t>((q * kC2) >> 40);
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
template <int ROUNDS, bool FOUR, bool MAXNORM, bool SUM>
__device__ __forceinline__ void quantize_bucket(const QArgs& a, int64_t b, int lane, float unit_scale,
                                                float (&sum)[ROUNDS][4]) {
    constexpr int D = 128 * ROUNDS;
    constexpr uint32_t kSignShift = FOUR ? 3 : 7;
    const float s_f = static_cast<float>(a.s);
    const uint32_t s_u = static_cast<uint32_t>(a.s);

    const int64_t b0 = b * D;
    const bool full = b0 + D <= a.n;
    float4 v[ROUNDS];
    if (full) {
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
    // A sum of squares below 2^-100 may have lost bits to underflow and one
    // above 2^126 overflows: such buckets (subnormal-sized or huge gradients;
    // the test is warp-uniform) are redone with every value scaled by the
    // power of two that brings the bucket maximum to [0.5, 1), which is exact,
    // and the norm scaled back.
    const bool tiny = norm < 8.8817842e-16f;      // 2^-50: the sum of squares is below 2^-100
    const bool huge = !(norm < 9.2233720e18f);    // 2^63, or inf / NaN
    if (huge || (tiny && !all_zero(v, lane))) {
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
        norm = ldexpf(df_sqrt(h2, l2), ex);
    }
    }
    if (lane == 0) a.norms[b] = norm;
    // norm == 0 means every coordinate is +-0: sign bit 0, level 0, code 0
    const bool zero = !(norm > 0.0f);
    const float S = zero ? 0.0f : __fdiv_rn(s_f, norm);

#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
        const int64_t e = b0 + 128 * j + 4 * lane;
        // e is a multiple of 4, so seed_w ^ (e + k) == (seed_w ^ e) ^ k
        const uint64_t kbase = a.seed_w ^ static_cast<uint64_t>(e);
        const float xs[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        uint32_t c[4] = {0u, 0u, 0u, 0u};
        if (!zero) {
            uint32_t t[4];
            hash4_top24(kbase, t);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lvl = qlevel(xs[k], S, s_u, t[k]);
                c[k] = ((xs[k] < 0.0f ? 1u : 0u) << kSignShift) | lvl;
            }
        }
        if (SUM) {
            const float u = __fmul_rn(norm, unit_scale);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float lf = __uint_as_float(0x4B000000u | (c[k] & (FOUR ? 7u : 127u))) - 8388608.0f;
                sum[j][k] = __fmaf_rn(lf, (c[k] >> kSignShift) ? -u : u, sum[j][k]);
            }
        }
        if (FOUR) {
            const uint32_t lo2 = (c[0] << 4) | c[1];
            const uint32_t hi2 = (c[2] << 4) | c[3];
            if (full) {
                *reinterpret_cast<uint16_t*>(a.codes + (e >> 1)) = static_cast<uint16_t>(lo2 | (hi2 << 8));
            } else {
                if (e < a.n) a.codes[e >> 1] = static_cast<uint8_t>(e + 1 < a.n ? lo2 : (c[0] << 4));
                if (e + 2 < a.n) a.codes[(e >> 1) + 1] = static_cast<uint8_t>(e + 3 < a.n ? hi2 : (c[2] << 4));
            }
        } else {
            if (full) {
                *reinterpret_cast<uint32_t*>(a.codes + e) = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (e + k < a.n) a.codes[e + k] = static_cast<uint8_t>(c[k]);
            }
        }
    }
}

// One warp per bucket; the grid covers every bucket.  For buckets of up to
// 512 the register bound allows 6 CTAs (48 warps) per SM with no spills: the
// quantiser is bound by the integer ALU pipe and latency, and 6 measured
// ahead of 4 (56 registers) and of 8 (32 registers and spills).
template <int ROUNDS, bool FOUR, bool MAXNORM>
__global__ void __launch_bounds__(kThreads, ROUNDS >= 8 ? 2 : 6)
k_qsgd_quantize(const QArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= a.nbuckets) return;
    float unused[ROUNDS][4];
    quantize_bucket<ROUNDS, FOUR, MAXNORM, false>(a, b, lane, 0.0f, unused);
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

template <int ROUNDS, bool FOUR, bool MAXNORM>
__global__ void __launch_bounds__(kThreads, ROUNDS >= 8 ? 2 : 4)
k_qsgd_step(const StepArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= a.q.nbuckets) return;
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
        quantize_bucket<ROUNDS, FOUR, MAXNORM, true>(q, b, lane, a.unit_scale, sum);
    }
    const int64_t b0 = b * D;
    const bool full = b0 + D <= a.q.n;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
        const int64_t e = b0 + 128 * j + 4 * lane;
        const float4 o = make_float4(sum[j][0], sum[j][1], sum[j][2], sum[j][3]);
        if (full) {
            st_stream_f4(a.out + e, o);
        } else {
            if (e < a.q.n) a.out[e] = o.x;
            if (e + 1 < a.q.n) a.out[e + 1] = o.y;
            if (e + 2 < a.q.n) a.out[e + 2] = o.z;
            if (e + 3 < a.q.n) a.out[e + 3] = o.w;
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

// Code k (0..3) of the raw bits above.
template <bool FOUR>
__device__ __forceinline__ uint32_t code_of(uint32_t raw, int k) {
    if (FOUR) {
        // byte 0 = (c0 << 4) | c1, byte 1 = (c2 << 4) | c3
        const int shift = (k == 0) ? 4 : (k == 1) ? 0 : (k == 2) ? 12 : 8;
        return (raw >> shift) & 15u;
    }
    return (raw >> (8 * k)) & 255u;
}

// NB consecutive buckets by one warp (NB = 1 in use: a second bucket per warp
// measured slower).  Workers are taken WC at a time with every code and norm
// load of the group issued before any is decoded; each element's sum runs in
// worker order, every term added by one fma of the level with the signed unit
// norm * (scale / s).
template <int ROUNDS, bool FOUR, int NB>
__device__ __forceinline__ void dequant_buckets(const DArgs& a, int64_t b_first, int lane,
                                                const float* s_signed_level) {
    constexpr int WC = (ROUNDS * NB >= 8) ? 2 : 4;    // workers whose loads are issued together
    constexpr int D = 128 * ROUNDS;

    float sum[NB][ROUNDS][4];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb)
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) sum[bb][j][k] = 0.0f;
    bool full[NB];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) full[bb] = (b_first + bb + 1) * D <= a.n;

    for (int w0 = 0; w0 < a.W; w0 += WC) {
        uint32_t raw[WC][NB][ROUNDS];
        float unit[WC][NB];
#pragma unroll
        for (int q = 0; q < WC; ++q) {
            if (w0 + q < a.W) {
#pragma unroll
                for (int bb = 0; bb < NB; ++bb) {
                    const int64_t b = b_first + bb;
                    if (b < a.nbuckets) {
                        unit[q][bb] = __ldg(a.norms.p[w0 + q] + b);
#pragma unroll
                        for (int j = 0; j < ROUNDS; ++j)
                            raw[q][bb][j] = load_raw4<FOUR>(a.codes.p[w0 + q], b * D + 128 * j + 4 * lane, a.n,
                                                             full[bb]);
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < WC; ++q) {
            if (w0 + q < a.W) {
#pragma unroll
                for (int bb = 0; bb < NB; ++bb) {
                    if (b_first + bb >= a.nbuckets) continue;
                    const float u = __fmul_rn(unit[q][bb], a.unit_scale);
#pragma unroll
                    for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            // (+-level) * unit added with one rounding: the same
                            // value as level * (+-unit)
                            const uint32_t c = code_of<FOUR>(raw[q][bb][j], k);
                            sum[bb][j][k] = __fmaf_rn(s_signed_level[c], u, sum[bb][j][k]);
                        }
                }
            }
        }
    }
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
        const int64_t b = b_first + bb;
        if (b >= a.nbuckets) continue;
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j) {
            const int64_t e = b * D + 128 * j + 4 * lane;
            const float4 o = make_float4(sum[bb][j][0], sum[bb][j][1], sum[bb][j][2], sum[bb][j][3]);
            if (full[bb]) {
                st_stream_f4(a.out + e, o);
            } else {
                if (e < a.n) a.out[e] = o.x;
                if (e + 1 < a.n) a.out[e + 1] = o.y;
                if (e + 2 < a.n) a.out[e + 2] = o.z;
                if (e + 3 < a.n) a.out[e + 3] = o.w;
            }
        }
    }
}

// Persistent grid (as many CTAs as fit on the GPU at once): each warp strides
// over the buckets, so a CTA builds its code table once rather than once per
// 8 buckets (measured 8-15% faster than one CTA per 8 buckets).
template <int ROUNDS, bool FOUR, int NB>
__global__ void __launch_bounds__(kThreads, ROUNDS >= 8 ? 2 : 4)
k_qsgd_dequant_sum(const DArgs a) {
    // code -> signed level as an exact float: (-1)^sign * level; one table
    // load replaces the level extraction, its conversion and the sign select
    constexpr int kCodes = FOUR ? 16 : 256;
    __shared__ float s_signed_level[kCodes];
    for (int c = threadIdx.x; c < kCodes; c += blockDim.x) {
        const float l = static_cast<float>(c & (FOUR ? 7 : 127));
        s_signed_level[c] = (c & (FOUR ? 8 : 128)) ? -l : l;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t stride = ((static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) * NB;
    for (int64_t b_first = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * NB;
         b_first < a.nbuckets; b_first += stride)
        dequant_buckets<ROUNDS, FOUR, NB>(a, b_first, lane, s_signed_level);
}

template <bool FOUR, bool MAXNORM>
int launch_quantize(int rounds, const QArgs& a, unsigned grid, cudaStream_t s) {
    switch (rounds) {
        case 1: k_qsgd_quantize<1, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        case 2: k_qsgd_quantize<2, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        case 4: k_qsgd_quantize<4, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        case 8: k_qsgd_quantize<8, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        case 16: k_qsgd_quantize<16, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        default: return GC_ERR_INVALID;
    }
    return launch_status();
}

template <bool FOUR, bool MAXNORM>
int launch_step(int rounds, const StepArgs& a, unsigned grid, cudaStream_t s) {
    switch (rounds) {
        case 1: k_qsgd_step<1, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        case 2: k_qsgd_step<2, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        case 4: k_qsgd_step<4, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        case 8: k_qsgd_step<8, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        case 16: k_qsgd_step<16, FOUR, MAXNORM><<<grid, kThreads, 0, s>>>(a); break;
        default: return GC_ERR_INVALID;
    }
    return launch_status();
}

template <bool FOUR>
int launch_dequant(int rounds, const DArgs& a, cudaStream_t s) {
    const int64_t want = blocks_for_tiles(a.nbuckets);
    switch (rounds) {
        case 1: return launch_persistent(k_qsgd_dequant_sum<1, FOUR, 1>, want, s, a);
        case 2: return launch_persistent(k_qsgd_dequant_sum<2, FOUR, 1>, want, s, a);
        case 4: return launch_persistent(k_qsgd_dequant_sum<4, FOUR, 1>, want, s, a);
        case 8: return launch_persistent(k_qsgd_dequant_sum<8, FOUR, 1>, want, s, a);
        case 16: return launch_persistent(k_qsgd_dequant_sum<16, FOUR, 1>, want, s, a);
        default: return GC_ERR_INVALID;
    }
    return launch_status();
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
    const unsigned grid = blocks_for_tiles(a.nbuckets);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (maxnorm)
        return s_levels <= 7 ? launch_quantize<true, true>(bucket / 128, a, grid, s)
                             : launch_quantize<false, true>(bucket / 128, a, grid, s);
    return s_levels <= 7 ? launch_quantize<true, false>(bucket / 128, a, grid, s)
                         : launch_quantize<false, false>(bucket / 128, a, grid, s);
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
    const unsigned grid = blocks_for_tiles(a.q.nbuckets);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (maxnorm)
        return s_levels <= 7 ? launch_step<true, true>(bucket / 128, a, grid, s)
                             : launch_step<false, true>(bucket / 128, a, grid, s);
    return s_levels <= 7 ? launch_step<true, false>(bucket / 128, a, grid, s)
                         : launch_step<false, false>(bucket / 128, a, grid, s);
}

}  // extern "C"
