// twobit.cu -- 2-bit threshold quantisation with error feedback, its fused
// dequantise-sum + update, and the CD-SGD full-precision correction step.
//
// Sources: "2bit gradient compression" (MXNet PR #8662), sections "Two bit
// quantization", "Format of compressed gradient", "Local kvstore", "Dist
// kvstore"; "CD-SGD: Distributed Stochastic Gradient Descent with Compression
// and Delay Compensation", eq. 1, eq. 10, Algorithm 1, section 3.1; EASGD
// local update from the IMerge design notes.
//
// Layout in HBM: every buffer is a flat contiguous array.  A warp owns a
// "tile" of 512 consecutive elements = 32 packed code words; lane l reads the
// 16-byte vectors at tile offsets 4l, 128+4l, 256+4l, 384+4l, so every load
// and store instruction of the warp covers 512 contiguous bytes.
#include "gc_common.cuh"

namespace gc {
namespace {

constexpr int kTile = 512;            // elements per warp tile
constexpr int kWordsPerTile = kTile / 16;

// One element of the threshold rule; returns the 2-bit code and updates r.
// r + g, r - t and r + t are single fp32 round-to-nearest operations.
__device__ __forceinline__ uint32_t quantize1(float& r, float g, float t) {
    const float x = __fadd_rn(r, g);
    const bool pos = x >= t;
    const bool neg = x <= -t;
    r = pos ? __fsub_rn(x, t) : (neg ? __fadd_rn(x, t) : x);
    return pos ? 3u : (neg ? 2u : 0u);
}

// 4 consecutive elements -> 8 code bits, first element in the top two bits.
__device__ __forceinline__ uint32_t quantize4(float4& r, const float4 g, float t) {
    uint32_t c = quantize1(r.x, g.x, t) << 6;
    c |= quantize1(r.y, g.y, t) << 4;
    c |= quantize1(r.z, g.z, t) << 2;
    c |= quantize1(r.w, g.w, t);
    return c;
}

// Byte address (within the code buffer) of the 8 code bits of elements
// e0..e0+3, e0 a multiple of 4: word e0/16 holds them in byte 3 - (e0/4)%4
// of its little-endian representation (first element in the MSBs).
__device__ __forceinline__ int64_t code_byte(int64_t e0) {
    return 4 * (e0 >> 4) + (3 - ((e0 >> 2) & 3));
}

// Tail: elements [tile_base, n) of the last, partial tile, one warp.
template <typename LoadG>
__device__ void quantize_tail(LoadG loadg, float* __restrict__ r, uint8_t* __restrict__ cb,
                              int64_t tile_base, int64_t n, float t, int lane) {
    const int64_t nwords = (n + 15) >> 4;
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
        const int64_t e0 = tile_base + 128 * j + 4 * lane;
        uint32_t c = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t e = e0 + k;
            if (e < n) {
                float rr = r[e];
                c |= quantize1(rr, loadg(e), t) << (6 - 2 * k);
                r[e] = rr;
            }
        }
        if ((e0 >> 4) < nwords) cb[code_byte(e0)] = static_cast<uint8_t>(c);
    }
}

// K1, fp32 gradients.  One warp per 512-element tile and a grid that covers
// every tile: the block scheduler hands out tiles in address order, which
// keeps the set of tiles in flight a compact window of HBM (measured faster
// than a persistent grid-stride loop).  The warp whose tile is the partial
// last one takes the bounds-checked path.
__global__ void __launch_bounds__(kThreads)
k_2bit_quantize_f32(const float* __restrict__ g, float* __restrict__ r,
                    uint32_t* __restrict__ codes, int64_t n, float t) {
    const int lane = threadIdx.x & 31;
    const int64_t tile = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nfull = n / kTile;
    uint8_t* cb = reinterpret_cast<uint8_t*>(codes);
    if (tile < nfull) {
        const int64_t base = tile * kTile + 4 * lane;
        float4 gv[4], rv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            gv[j] = ld_stream_f4(g + base + 128 * j);
            rv[j] = ld_f4(r + base + 128 * j);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t c = quantize4(rv[j], gv[j], t);
            st_stream_f4(r + base + 128 * j, rv[j]);
            cb[code_byte(base + 128 * j)] = static_cast<uint8_t>(c);
        }
    } else if (tile == nfull && n % kTile != 0) {
        quantize_tail([g](int64_t e) { return g[e]; }, r, cb, nfull * kTile, n, t, lane);
    }
}

// K1, bf16 gradients: lane l of round j reads 8 bf16 (16 bytes) at tile
// offset 256j + 8l, i.e. two code bytes = one 16-bit half of a word.  Same
// launch shape as the fp32 kernel.
__global__ void __launch_bounds__(kThreads)
k_2bit_quantize_bf16(const uint16_t* __restrict__ g, float* __restrict__ r,
                     uint32_t* __restrict__ codes, int64_t n, float t) {
    const int lane = threadIdx.x & 31;
    const int64_t tile = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nfull = n / kTile;
    uint16_t* ch = reinterpret_cast<uint16_t*>(codes);
    if (tile < nfull) {
        const int64_t base = tile * kTile + 8 * lane;
        uint4 gv[2];
        float4 rv[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            gv[j] = ld_stream_u4(g + base + 256 * j);
            rv[2 * j] = ld_f4(r + base + 256 * j);
            rv[2 * j + 1] = ld_f4(r + base + 256 * j + 4);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float4 g0 = make_float4(bf16lo(gv[j].x), bf16hi(gv[j].x),
                                          bf16lo(gv[j].y), bf16hi(gv[j].y));
            const float4 g1 = make_float4(bf16lo(gv[j].z), bf16hi(gv[j].z),
                                          bf16lo(gv[j].w), bf16hi(gv[j].w));
            const uint32_t c = (quantize4(rv[2 * j], g0, t) << 8) | quantize4(rv[2 * j + 1], g1, t);
            st_stream_f4(r + base + 256 * j, rv[2 * j]);
            st_stream_f4(r + base + 256 * j + 4, rv[2 * j + 1]);
            // elements e..e+7 (e = 8 mod 16 or 0 mod 16) are the high half of
            // word e/16 when e % 16 == 0, its low half otherwise
            const int64_t e = base + 256 * j;
            ch[2 * (e >> 4) + 1 - ((e >> 3) & 1)] = static_cast<uint16_t>(c);
        }
    } else if (tile == nfull && n % kTile != 0) {
        quantize_tail([g](int64_t e) { return __uint_as_float(static_cast<uint32_t>(g[e]) << 16); },
                      r, reinterpret_cast<uint8_t*>(codes), nfull * kTile, n, t, lane);
    }
}

// ------------------------------------------------------------------ K1, batched

// B gradient buffers (workers, or the gradient tensors of one worker) of
// possibly different sizes quantised by one launch: the grid covers the
// concatenation of every buffer's 512-element tiles, and each warp finds its
// buffer in the tile prefix table.
struct BatchArgs {
    PtrTable<const void*> grads;
    PtrTable<float*> res;
    PtrTable<uint32_t*> codes;
    int64_t n[GC_MAX_WORKERS];
    int64_t tile_start[GC_MAX_WORKERS + 1];
    int B;
    float t;
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads)
k_2bit_quantize_batched(const BatchArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t T = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (T >= a.tile_start[a.B]) return;
    int lo = 0, hi = a.B - 1;           // last b with tile_start[b] <= T
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.tile_start[mid] <= T) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int64_t tile = T - a.tile_start[b];
    const int64_t n = a.n[b];
    float* __restrict__ r = a.res.p[b];
    const float t = a.t;
    const int64_t nfull = n / kTile;
    if (!BF16) {
        const float* __restrict__ g = static_cast<const float*>(a.grads.p[b]);
        uint8_t* cb = reinterpret_cast<uint8_t*>(a.codes.p[b]);
        if (tile < nfull) {
            const int64_t base = tile * kTile + 4 * lane;
            float4 gv[4], rv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                gv[j] = ld_stream_f4(g + base + 128 * j);
                rv[j] = ld_f4(r + base + 128 * j);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t c = quantize4(rv[j], gv[j], t);
                st_stream_f4(r + base + 128 * j, rv[j]);
                cb[code_byte(base + 128 * j)] = static_cast<uint8_t>(c);
            }
        } else {
            quantize_tail([g](int64_t e) { return g[e]; }, r, cb, nfull * kTile, n, t, lane);
        }
    } else {
        const uint16_t* __restrict__ g = static_cast<const uint16_t*>(a.grads.p[b]);
        uint16_t* ch = reinterpret_cast<uint16_t*>(a.codes.p[b]);
        if (tile < nfull) {
            const int64_t base = tile * kTile + 8 * lane;
            uint4 gv[2];
            float4 rv[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                gv[j] = ld_stream_u4(g + base + 256 * j);
                rv[2 * j] = ld_f4(r + base + 256 * j);
                rv[2 * j + 1] = ld_f4(r + base + 256 * j + 4);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float4 g0 = make_float4(bf16lo(gv[j].x), bf16hi(gv[j].x),
                                              bf16lo(gv[j].y), bf16hi(gv[j].y));
                const float4 g1 = make_float4(bf16lo(gv[j].z), bf16hi(gv[j].z),
                                              bf16lo(gv[j].w), bf16hi(gv[j].w));
                const uint32_t c = (quantize4(rv[2 * j], g0, t) << 8) | quantize4(rv[2 * j + 1], g1, t);
                st_stream_f4(r + base + 256 * j, rv[2 * j]);
                st_stream_f4(r + base + 256 * j + 4, rv[2 * j + 1]);
                const int64_t e = base + 256 * j;
                ch[2 * (e >> 4) + 1 - ((e >> 3) & 1)] = static_cast<uint16_t>(c);
            }
        } else {
            quantize_tail([g](int64_t e) { return __uint_as_float(static_cast<uint32_t>(g[e]) << 16); },
                          r, reinterpret_cast<uint8_t*>(a.codes.p[b]), nfull * kTile, n, t, lane);
        }
    }
}

// ------------------------------------------------------------------ K2

// Maps a code word to per-field (value + 1): 11 -> 2, 10 -> 0, 00/01 -> 1.
__device__ __forceinline__ uint32_t plus_one_fields(uint32_t c) {
    const uint32_t h = c >> 1;
    const uint32_t two = h & c & 0x55555555u;    // code 11
    const uint32_t one = ~h & 0x55555555u;       // code 0x
    return (two << 1) | one;
}

// Bytes (value+1 sums) for the four elements 4a..4a+3 of a word, from the
// four byte-lane accumulators (see k_2bit_dqsum).  Byte b of the result is
// element 4a+b.
template <int A>
__device__ __forceinline__ uint32_t pack_quad(uint32_t B0, uint32_t B1, uint32_t B2, uint32_t B3) {
    constexpr uint32_t sel = (3 - A) | ((7 - A) << 4);
    const uint32_t t1 = __byte_perm(B3, B1, sel);   // elements 4a, 4a+1
    const uint32_t t2 = __byte_perm(B2, B0, sel);   // elements 4a+2, 4a+3
    return __byte_perm(t1, t2, 0x5410);
}

struct DqArgs {
    PtrTable<const uint32_t*> codes;
    int W;
    int64_t n;
    float k_out;      // threshold / W                (NONE)
    float k_lr;       // lr * threshold / W           (SGD, EASGD)
    float alpha;      // EASGD
    const float* center;
    float* weights;
    float* out;
};

// Applies the update to 4 consecutive elements from their per-element
// (value + 1) sums packed in the bytes of R.  `w`/`c` are the already-loaded
// weight and center vectors (full tiles).
template <int KIND>
__device__ __forceinline__ void dq_apply_full(const DqArgs& a, int64_t e0, uint32_t R, float4 w, float4 c) {
    const float bias = 8388608.0f + static_cast<float>(a.W);
    float cnt[4];
#pragma unroll
    for (int b = 0; b < 4; ++b)
        cnt[b] = __uint_as_float(__byte_perm(R, 0x4B000000u, 0x7540u | b)) - bias;
    if (KIND == GC_UPD_NONE) {
        st_stream_f4(a.out + e0, make_float4(cnt[0] * a.k_out, cnt[1] * a.k_out,
                                             cnt[2] * a.k_out, cnt[3] * a.k_out));
    } else {
        float4 nw;
        nw.x = fmaf(-cnt[0], a.k_lr, w.x);
        nw.y = fmaf(-cnt[1], a.k_lr, w.y);
        nw.z = fmaf(-cnt[2], a.k_lr, w.z);
        nw.w = fmaf(-cnt[3], a.k_lr, w.w);
        if (KIND == GC_UPD_EASGD) {
            nw.x = fmaf(-a.alpha, w.x - c.x, nw.x);
            nw.y = fmaf(-a.alpha, w.y - c.y, nw.y);
            nw.z = fmaf(-a.alpha, w.z - c.z, nw.z);
            nw.w = fmaf(-a.alpha, w.w - c.w, nw.w);
        }
        st_stream_f4(a.weights + e0, nw);
    }
}

// Partial tile: element by element with bounds checks.
template <int KIND>
__device__ __forceinline__ void dq_apply_tail(const DqArgs& a, int64_t e0, uint32_t R) {
    const float bias = 8388608.0f + static_cast<float>(a.W);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int64_t e = e0 + b;
        if (e >= a.n) break;
        const float cnt = __uint_as_float(__byte_perm(R, 0x4B000000u, 0x7540u | b)) - bias;
        if (KIND == GC_UPD_NONE) {
            a.out[e] = cnt * a.k_out;
        } else {
            const float w = a.weights[e];
            float nw = fmaf(-cnt, a.k_lr, w);
            if (KIND == GC_UPD_EASGD) nw = fmaf(-a.alpha, w - a.center[e], nw);
            a.weights[e] = nw;
        }
    }
}

// Adds one code word's per-element (value + 1) to the 4-bit accumulators.
__device__ __forceinline__ void swar_add(uint32_t c, uint32_t& A0, uint32_t& A1) {
    const uint32_t m = plus_one_fields(c);
    A0 += m & 0x33333333u;
    A1 += (m >> 2) & 0x33333333u;
}

// Moves the 4-bit accumulators (<= 7 workers) into the 8-bit ones.
__device__ __forceinline__ void swar_spill(uint32_t A0, uint32_t A1, uint32_t& B0, uint32_t& B1,
                                           uint32_t& B2, uint32_t& B3) {
    B0 += A0 & 0x0F0F0F0Fu;
    B1 += (A0 >> 4) & 0x0F0F0F0Fu;
    B2 += A1 & 0x0F0F0F0Fu;
    B3 += (A1 >> 4) & 0x0F0F0F0Fu;
}

// K2: one warp per 512-element tile.  Lane m loads word m of the tile from
// every worker (128 contiguous bytes per worker) and sums, in SWAR form, the
// per-element (decoded value + 1) over the workers: 4-bit fields for up to 7
// workers at a time, then 8-bit fields (sums <= 2 * 64 fit a byte).  The
// per-element sums are regrouped through shared memory so that lane l then
// owns elements 128j + 4l .. +3 of the tile, matching the coalesced float4
// layout of the weights.  Every load of a tile (weights, center, up to 14
// code words) is issued before any of them is used.  One tile per warp; the
// grid covers every tile.
template <int KIND>
__global__ void __launch_bounds__(kThreads, KIND == GC_UPD_EASGD ? 3 : 4)
k_2bit_dqsum(const DqArgs a) {
    __shared__ uint4 stage[kWarpsPerBlock][32];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t nwords = (a.n + 15) >> 4;
    const int64_t ntiles = (a.n + kTile - 1) / kTile;
    const uint32_t* stage32 = reinterpret_cast<const uint32_t*>(&stage[wib][0]);

    const int64_t tile = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (tile < ntiles) {
        const bool full = (tile + 1) * kTile <= a.n;
        const int64_t ebase = tile * kTile + 4 * lane;
        float4 wv[4], cv[4];
        if (full && KIND != GC_UPD_NONE) {
#pragma unroll
            for (int j = 0; j < 4; ++j) wv[j] = ld_f4(a.weights + ebase + 128 * j);
            if (KIND == GC_UPD_EASGD) {
#pragma unroll
                for (int j = 0; j < 4; ++j) cv[j] = ld_stream_f4(a.center + ebase + 128 * j);
            }
        }
        const int64_t word = tile * kWordsPerTile + lane;
        const bool have_word = word < nwords;
        uint32_t B0 = 0, B1 = 0, B2 = 0, B3 = 0;
        for (int w0 = 0; w0 < a.W; w0 += 14) {
            uint32_t cw[14];
#pragma unroll
            for (int k = 0; k < 14; ++k)
                cw[k] = (w0 + k < a.W && have_word) ? __ldg(a.codes.p[w0 + k] + word) : 0u;
            uint32_t A0 = 0, A1 = 0;
#pragma unroll
            for (int k = 0; k < 7; ++k)
                if (w0 + k < a.W) swar_add(cw[k], A0, A1);
            swar_spill(A0, A1, B0, B1, B2, B3);
            if (w0 + 7 < a.W) {
                A0 = A1 = 0;
#pragma unroll
                for (int k = 7; k < 14; ++k)
                    if (w0 + k < a.W) swar_add(cw[k], A0, A1);
                swar_spill(A0, A1, B0, B1, B2, B3);
            }
        }
        stage[wib][lane] = make_uint4(pack_quad<0>(B0, B1, B2, B3), pack_quad<1>(B0, B1, B2, B3),
                                      pack_quad<2>(B0, B1, B2, B3), pack_quad<3>(B0, B1, B2, B3));
        __syncwarp();
        if (full) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dq_apply_full<KIND>(a, ebase + 128 * j, stage32[32 * j + lane], wv[j], cv[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t e0 = ebase + 128 * j;
                if (e0 < a.n) dq_apply_tail<KIND>(a, e0, stage32[32 * j + lane]);
            }
        }
    }
}

// ------------------------------------------------------------------ K1+K2 fused

// The whole 2-bit step of W workers held on this GPU in one pass: for every
// 512-element tile a warp quantises the tile of each worker in turn (codes
// and residuals written as gc_2bit_quantize does), keeps each element's
// decoded sum in registers instead of re-reading the codes, and applies the
// update as gc_2bit_dequant_sum_update does -- the outputs are bit-identical
// to those two calls.  Worker w+1's gradient and residual loads are issued
// before worker w's tile is processed.  With LOCAL, each worker's CD-SGD
// eq. 11 local weights W_loc = W - local_lr * g are written from the global
// weights as read before the update (as gc_2bit_quantize_local writes them).
struct StepArgs {
    PtrTable<const void*> grads;
    PtrTable<float*> res;
    PtrTable<uint32_t*> codes;
    PtrTable<float*> local;
    int W;
    int64_t n;
    float t;
    float k_out, k_lr, alpha, local_lr;
    const float* center;
    float* weights;
    float* out;
};

template <int KIND>
__device__ __forceinline__ void step_apply(const StepArgs& a, int64_t e0, const float (&cnt)[4], float4 w,
                                           float4 c) {
    if (KIND == GC_UPD_NONE) {
        st_stream_f4(a.out + e0, make_float4(cnt[0] * a.k_out, cnt[1] * a.k_out, cnt[2] * a.k_out,
                                             cnt[3] * a.k_out));
    } else {
        float4 nw;
        nw.x = fmaf(-cnt[0], a.k_lr, w.x);
        nw.y = fmaf(-cnt[1], a.k_lr, w.y);
        nw.z = fmaf(-cnt[2], a.k_lr, w.z);
        nw.w = fmaf(-cnt[3], a.k_lr, w.w);
        if (KIND == GC_UPD_EASGD) {
            nw.x = fmaf(-a.alpha, w.x - c.x, nw.x);
            nw.y = fmaf(-a.alpha, w.y - c.y, nw.y);
            nw.z = fmaf(-a.alpha, w.z - c.z, nw.z);
            nw.w = fmaf(-a.alpha, w.w - c.w, nw.w);
        }
        st_stream_f4(a.weights + e0, nw);
    }
}

// fp32 quantise of one float4 that also adds each element's decoded value
// + 1 (0, 1 or 2) to byte k of `cnt` (element k of the four); after W workers
// byte k holds (decoded sum + W) <= 2 * 64.
__device__ __forceinline__ uint32_t quantize4_count(float4& r, const float4 g, float t, uint32_t& cnt) {
    const uint32_t c0 = quantize1(r.x, g.x, t), c1 = quantize1(r.y, g.y, t);
    const uint32_t c2 = quantize1(r.z, g.z, t), c3 = quantize1(r.w, g.w, t);
    // code 11 -> 2, 10 -> 0, 00 -> 1: (c >> 1) ? (c & 1) * 2 : 1
    const uint32_t c = (c0 << 6) | (c1 << 4) | (c2 << 2) | c3;
    const uint32_t h = c >> 1;
    const uint32_t f = (((h & c & 0x55u) << 1) | (~h & 0x55u));   // four (value + 1) fields, element 0 on top
    cnt += ((f >> 6) & 3u) | (((f >> 4) & 3u) << 8) | (((f >> 2) & 3u) << 16) | ((f & 3u) << 24);
    return c;
}

// Element offset, within a lane's share of a full tile, of its q-th group of
// four consecutive elements (q = 0..3).  fp32: lane l owns 4l + 128q (one
// float4 per round, as the fp32 quantiser); bf16: lane l owns 8l + 256(q/2)
// + 4(q%2) (one 16-byte vector of 8 bf16 per round, as the bf16 quantiser).
template <bool BF16>
__device__ __forceinline__ int64_t step_group(int lane, int q) {
    return BF16 ? 8 * lane + 256 * (q >> 1) + 4 * (q & 1) : 4 * lane + 128 * q;
}

// One worker's gradient for a lane's 16 elements of a full tile, raw: four
// float4 (fp32) or two 16-byte vectors of 8 bf16 in the first two slots.
template <bool BF16>
__device__ __forceinline__ void step_load_grad(const void* g, int64_t tbase, int lane, uint4 (&raw)[4]) {
    if (BF16) {
        const uint16_t* gh = static_cast<const uint16_t*>(g) + tbase + 8 * lane;
        raw[0] = ld_stream_u4(gh);
        raw[1] = ld_stream_u4(gh + 256);
    } else {
        const float* gf = static_cast<const float*>(g) + tbase + 4 * lane;
#pragma unroll
        for (int q = 0; q < 4; ++q) raw[q] = ld_stream_u4(gf + 128 * q);
    }
}

// Gradient values of group q from the raw registers (bf16 widened exactly).
template <bool BF16>
__device__ __forceinline__ float4 step_grad(const uint4 (&raw)[4], int q) {
    if (BF16) {
        const uint4 u = raw[q >> 1];
        return (q & 1) ? make_float4(bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w))
                       : make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
    }
    return make_float4(__uint_as_float(raw[q].x), __uint_as_float(raw[q].y), __uint_as_float(raw[q].z),
                       __uint_as_float(raw[q].w));
}

// Registers bound the occupancy here: per lane the current and the next
// worker's gradient and residual (the next one's loads are in flight while
// the current one is quantised), the per-element counts packed four to a
// register, and -- only with LOCAL, which needs them in the loop -- the
// weights; otherwise weights and center are loaded after the worker loop.
template <int KIND, bool BF16, bool LOCAL>
__global__ void __launch_bounds__(kThreads, (BF16 && !LOCAL) ? 3 : 2)
k_2bit_step(const StepArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t tile = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nfull = a.n / kTile;
    if (tile < nfull) {
        const int64_t tbase = tile * kTile;
        float4 wv[4], cv[4];
        if (LOCAL) {
#pragma unroll
            for (int q = 0; q < 4; ++q) wv[q] = ld_f4(a.weights + tbase + step_group<BF16>(lane, q));
        }
        uint32_t cnt[4] = {0u, 0u, 0u, 0u};
        uint4 ga[4];
        float4 ra[4];
        step_load_grad<BF16>(a.grads.p[0], tbase, lane, ga);
#pragma unroll
        for (int q = 0; q < 4; ++q) ra[q] = ld_f4(a.res.p[0] + tbase + step_group<BF16>(lane, q));
        for (int w = 0; w < a.W; ++w) {
            uint4 gb[4];
            float4 rb[4];
            if (w + 1 < a.W) {
                step_load_grad<BF16>(a.grads.p[w + 1], tbase, lane, gb);
#pragma unroll
                for (int q = 0; q < 4; ++q) rb[q] = ld_f4(a.res.p[w + 1] + tbase + step_group<BF16>(lane, q));
            }
            float* r = a.res.p[w];
            uint32_t c[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t e = tbase + step_group<BF16>(lane, q);
                const float4 g = step_grad<BF16>(ga, q);
                if (LOCAL)
                    st_stream_f4(a.local.p[w] + e,
                                 make_float4(fmaf(-a.local_lr, g.x, wv[q].x), fmaf(-a.local_lr, g.y, wv[q].y),
                                             fmaf(-a.local_lr, g.z, wv[q].z), fmaf(-a.local_lr, g.w, wv[q].w)));
                c[q] = quantize4_count(ra[q], g, a.t, cnt[q]);
                st_stream_f4(r + e, ra[q]);
            }
            if (BF16) {
                // elements e..e+7 (e = tbase + 8 lane + 256 j) are the high half
                // of word e/16 when e % 16 == 0, its low half otherwise
                uint16_t* ch = reinterpret_cast<uint16_t*>(a.codes.p[w]);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int64_t e = tbase + 8 * lane + 256 * j;
                    ch[2 * (e >> 4) + 1 - ((e >> 3) & 1)] = static_cast<uint16_t>((c[2 * j] << 8) | c[2 * j + 1]);
                }
            } else {
                uint8_t* cb = reinterpret_cast<uint8_t*>(a.codes.p[w]);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    cb[code_byte(tbase + step_group<BF16>(lane, q))] = static_cast<uint8_t>(c[q]);
            }
            if (w + 1 < a.W) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ga[q] = gb[q];
                    ra[q] = rb[q];
                }
            }
        }
        if (KIND != GC_UPD_NONE && !LOCAL) {
#pragma unroll
            for (int q = 0; q < 4; ++q) wv[q] = ld_f4(a.weights + tbase + step_group<BF16>(lane, q));
        }
        if (KIND == GC_UPD_EASGD) {
#pragma unroll
            for (int q = 0; q < 4; ++q) cv[q] = ld_stream_f4(a.center + tbase + step_group<BF16>(lane, q));
        }
        const float bias = static_cast<float>(a.W);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float cf[4] = {static_cast<float>(cnt[q] & 255u) - bias,
                                 static_cast<float>((cnt[q] >> 8) & 255u) - bias,
                                 static_cast<float>((cnt[q] >> 16) & 255u) - bias,
                                 static_cast<float>(cnt[q] >> 24) - bias};
            step_apply<KIND>(a, tbase + step_group<BF16>(lane, q), cf, wv[q], cv[q]);
        }
    } else if (tile == nfull && a.n % kTile != 0) {
        // partial last tile: element by element
        const int64_t nwords = (a.n + 15) >> 4;
        for (int j = 0; j < 4; ++j) {
            const int64_t e0 = nfull * kTile + 128 * j + 4 * lane;
            int cnt[4] = {0, 0, 0, 0};
            for (int w = 0; w < a.W; ++w) {
                float* r = a.res.p[w];
                uint32_t cbits = 0;
                for (int k = 0; k < 4; ++k) {
                    const int64_t e = e0 + k;
                    if (e < a.n) {
                        const float gval = BF16 ? __uint_as_float(static_cast<uint32_t>(
                                                      static_cast<const uint16_t*>(a.grads.p[w])[e]) << 16)
                                                : static_cast<const float*>(a.grads.p[w])[e];
                        if (LOCAL) a.local.p[w][e] = fmaf(-a.local_lr, gval, a.weights[e]);
                        float rr = r[e];
                        const uint32_t c = quantize1(rr, gval, a.t);
                        r[e] = rr;
                        cbits |= c << (6 - 2 * k);
                        cnt[k] += (c == 3u) - (c == 2u);
                    }
                }
                if ((e0 >> 4) < nwords) reinterpret_cast<uint8_t*>(a.codes.p[w])[code_byte(e0)] = static_cast<uint8_t>(cbits);
            }
            for (int k = 0; k < 4; ++k) {
                const int64_t e = e0 + k;
                if (e >= a.n) break;
                const float cf = static_cast<float>(cnt[k]);
                if (KIND == GC_UPD_NONE) {
                    a.out[e] = cf * a.k_out;
                } else {
                    const float wo = a.weights[e];
                    float nw = fmaf(-cf, a.k_lr, wo);
                    if (KIND == GC_UPD_EASGD) nw = fmaf(-a.alpha, wo - a.center[e], nw);
                    a.weights[e] = nw;
                }
            }
        }
    }
}

template <bool BF16, bool LOCAL>
void launch_step(gc_update kind, unsigned grid, cudaStream_t s, const StepArgs& a) {
    switch (kind) {
        case GC_UPD_NONE: k_2bit_step<GC_UPD_NONE, BF16, LOCAL><<<grid, kThreads, 0, s>>>(a); break;
        case GC_UPD_SGD: k_2bit_step<GC_UPD_SGD, BF16, LOCAL><<<grid, kThreads, 0, s>>>(a); break;
        default: k_2bit_step<GC_UPD_EASGD, BF16, LOCAL><<<grid, kThreads, 0, s>>>(a); break;
    }
}

// ------------------------------------------------------------------ K1 (+K2 NONE) over S steps

// S successive steps of one worker in one launch: step s quantises gradient
// g_s into codes_s with the residual carried from step s-1 and, when out is
// given, writes the dequantised values out_s (+t, -t, 0).  The residual stays
// in registers between steps and is read and written once.  Bit-identical to
// S calls of gc_2bit_quantize (+ gc_2bit_dequant_sum_update NONE with W = 1).
struct StepsArgs {
    PtrTable<const void*> grads;
    PtrTable<uint32_t*> codes;
    PtrTable<float*> out;
    float* res;
    int S;
    bool has_out;
    int64_t n;
    float t;
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads)
k_2bit_steps(const StepsArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t tile = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nfull = a.n / kTile;
    if (tile < nfull) {
        const int64_t tbase = tile * kTile;
        float4 ra[4];
        uint4 ga[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) ra[q] = ld_f4(a.res + tbase + step_group<BF16>(lane, q));
        // the gradients of the next two steps are in flight while a step is
        // coded (one step ahead measured 8% slower at 2^20 elements, where
        // 13 warps per SM carry all the loads)
        uint4 gb[4];
        step_load_grad<BF16>(a.grads.p[0], tbase, lane, ga);
        if (a.S > 1) step_load_grad<BF16>(a.grads.p[1], tbase, lane, gb);
        for (int st = 0; st < a.S; ++st) {
            uint4 gn[4];
            if (st + 2 < a.S) step_load_grad<BF16>(a.grads.p[st + 2], tbase, lane, gn);
            uint32_t c[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                int d[4];
                const float4 g = step_grad<BF16>(ga, q);
                uint32_t cnt = 0u;
                c[q] = quantize4_count(ra[q], g, a.t, cnt);
                d[0] = static_cast<int>(cnt & 255u) - 1;
                d[1] = static_cast<int>((cnt >> 8) & 255u) - 1;
                d[2] = static_cast<int>((cnt >> 16) & 255u) - 1;
                d[3] = static_cast<int>(cnt >> 24) - 1;
                if (a.has_out)
                    st_stream_f4(a.out.p[st] + tbase + step_group<BF16>(lane, q),
                                 make_float4(static_cast<float>(d[0]) * a.t, static_cast<float>(d[1]) * a.t,
                                             static_cast<float>(d[2]) * a.t, static_cast<float>(d[3]) * a.t));
            }
            if (BF16) {
                uint16_t* ch = reinterpret_cast<uint16_t*>(a.codes.p[st]);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int64_t e = tbase + 8 * lane + 256 * j;
                    ch[2 * (e >> 4) + 1 - ((e >> 3) & 1)] = static_cast<uint16_t>((c[2 * j] << 8) | c[2 * j + 1]);
                }
            } else {
                uint8_t* cb = reinterpret_cast<uint8_t*>(a.codes.p[st]);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    cb[code_byte(tbase + step_group<BF16>(lane, q))] = static_cast<uint8_t>(c[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                ga[q] = gb[q];
                gb[q] = gn[q];
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            st_stream_f4(a.res + tbase + step_group<BF16>(lane, q), ra[q]);
    } else if (tile == nfull && a.n % kTile != 0) {
        const int64_t nwords = (a.n + 15) >> 4;
        float* r = a.res;
        for (int j = 0; j < 4; ++j) {
            const int64_t e0 = nfull * kTile + 128 * j + 4 * lane;
            float rr[4];
            for (int k = 0; k < 4; ++k) rr[k] = e0 + k < a.n ? r[e0 + k] : 0.0f;
            for (int st = 0; st < a.S; ++st) {
                uint32_t cbits = 0;
                for (int k = 0; k < 4; ++k) {
                    const int64_t e = e0 + k;
                    if (e < a.n) {
                        const float gval = BF16 ? __uint_as_float(static_cast<uint32_t>(
                                                      static_cast<const uint16_t*>(a.grads.p[st])[e]) << 16)
                                                : static_cast<const float*>(a.grads.p[st])[e];
                        const uint32_t c = quantize1(rr[k], gval, a.t);
                        cbits |= c << (6 - 2 * k);
                        if (a.has_out) a.out.p[st][e] = static_cast<float>((c == 3u) - (c == 2u)) * a.t;
                    }
                }
                if ((e0 >> 4) < nwords) reinterpret_cast<uint8_t*>(a.codes.p[st])[code_byte(e0)] = static_cast<uint8_t>(cbits);
            }
            for (int k = 0; k < 4; ++k)
                if (e0 + k < a.n) r[e0 + k] = rr[k];
        }
    }
}

// ------------------------------------------------------------------ K1 + CD-SGD local update

// CD-SGD eq. 11: while worker w's gradient is in registers for the 2-bit
// quantiser, its local weights W_loc[w] = W - local_lr * g are written too
// (W = the global weights, shared by all workers).  The grid visits the B
// workers of one tile on adjacent warps, so the B reads of a W tile meet in L2.
struct LocalArgs {
    PtrTable<const void*> grads;
    PtrTable<float*> res;
    PtrTable<uint32_t*> codes;
    PtrTable<float*> local;
    const float* weights;
    int B;
    int64_t n;
    float t, local_lr;
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads)
k_2bit_quantize_local(const LocalArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t T = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t ntiles = (a.n + kTile - 1) / kTile;
    if (T >= ntiles * a.B) return;
    const int64_t tile = T / a.B;
    const int b = static_cast<int>(T - tile * a.B);
    const int64_t nfull = a.n / kTile;
    float* __restrict__ r = a.res.p[b];
    float* __restrict__ wl = a.local.p[b];
    const float t = a.t, lr = a.local_lr;
    if (tile < nfull) {
        const int64_t base = tile * kTile + (BF16 ? 8 : 4) * lane;
        if (!BF16) {
            const float* __restrict__ g = static_cast<const float*>(a.grads.p[b]);
            uint8_t* cb = reinterpret_cast<uint8_t*>(a.codes.p[b]);
            float4 gv[4], rv[4], wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                gv[j] = ld_stream_f4(g + base + 128 * j);
                rv[j] = ld_f4(r + base + 128 * j);
                wv[j] = __ldg(reinterpret_cast<const float4*>(a.weights + base + 128 * j));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                st_stream_f4(wl + base + 128 * j,
                             make_float4(fmaf(-lr, gv[j].x, wv[j].x), fmaf(-lr, gv[j].y, wv[j].y),
                                         fmaf(-lr, gv[j].z, wv[j].z), fmaf(-lr, gv[j].w, wv[j].w)));
                const uint32_t c = quantize4(rv[j], gv[j], t);
                st_stream_f4(r + base + 128 * j, rv[j]);
                cb[code_byte(base + 128 * j)] = static_cast<uint8_t>(c);
            }
        } else {
            const uint16_t* __restrict__ g = static_cast<const uint16_t*>(a.grads.p[b]);
            uint16_t* ch = reinterpret_cast<uint16_t*>(a.codes.p[b]);
            uint4 gv[2];
            float4 rv[4], wv[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                gv[j] = ld_stream_u4(g + base + 256 * j);
                rv[2 * j] = ld_f4(r + base + 256 * j);
                rv[2 * j + 1] = ld_f4(r + base + 256 * j + 4);
                wv[2 * j] = __ldg(reinterpret_cast<const float4*>(a.weights + base + 256 * j));
                wv[2 * j + 1] = __ldg(reinterpret_cast<const float4*>(a.weights + base + 256 * j + 4));
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float4 g0 = make_float4(bf16lo(gv[j].x), bf16hi(gv[j].x), bf16lo(gv[j].y), bf16hi(gv[j].y));
                const float4 g1 = make_float4(bf16lo(gv[j].z), bf16hi(gv[j].z), bf16lo(gv[j].w), bf16hi(gv[j].w));
                st_stream_f4(wl + base + 256 * j,
                             make_float4(fmaf(-lr, g0.x, wv[2 * j].x), fmaf(-lr, g0.y, wv[2 * j].y),
                                         fmaf(-lr, g0.z, wv[2 * j].z), fmaf(-lr, g0.w, wv[2 * j].w)));
                st_stream_f4(wl + base + 256 * j + 4,
                             make_float4(fmaf(-lr, g1.x, wv[2 * j + 1].x), fmaf(-lr, g1.y, wv[2 * j + 1].y),
                                         fmaf(-lr, g1.z, wv[2 * j + 1].z), fmaf(-lr, g1.w, wv[2 * j + 1].w)));
                const uint32_t c = (quantize4(rv[2 * j], g0, t) << 8) | quantize4(rv[2 * j + 1], g1, t);
                st_stream_f4(r + base + 256 * j, rv[2 * j]);
                st_stream_f4(r + base + 256 * j + 4, rv[2 * j + 1]);
                const int64_t e = base + 256 * j;
                ch[2 * (e >> 4) + 1 - ((e >> 3) & 1)] = static_cast<uint16_t>(c);
            }
        }
    } else {
        // partial last tile
        const int64_t t0 = nfull * kTile;
        const int64_t nwords = (a.n + 15) >> 4;
        uint8_t* cb = reinterpret_cast<uint8_t*>(a.codes.p[b]);
        for (int j = 0; j < 4; ++j) {
            const int64_t e0 = t0 + 128 * j + 4 * lane;
            uint32_t cbits = 0;
            for (int k = 0; k < 4; ++k) {
                const int64_t e = e0 + k;
                if (e < a.n) {
                    const float gval = BF16 ? __uint_as_float(static_cast<uint32_t>(
                                                  static_cast<const uint16_t*>(a.grads.p[b])[e]) << 16)
                                            : static_cast<const float*>(a.grads.p[b])[e];
                    wl[e] = fmaf(-lr, gval, a.weights[e]);
                    float rr = r[e];
                    cbits |= quantize1(rr, gval, t) << (6 - 2 * k);
                    r[e] = rr;
                }
            }
            if ((e0 >> 4) < nwords) cb[code_byte(e0)] = static_cast<uint8_t>(cbits);
        }
    }
}

// ------------------------------------------------------------------ K3

struct CompArgs {
    PtrTable<const void*> grads;
    PtrTable<float*> res;
    int W;
    int64_t n;
    float k_lr;     // lr / W
    float* weights;
};

// 8 consecutive gradient values of worker w starting at e (full vectors).
template <bool BF16>
__device__ __forceinline__ void load_grad8(const void* g, int64_t e, float (&v)[8]) {
    if (BF16) {
        const uint4 u = ld_stream_u4(static_cast<const uint16_t*>(g) + e);
        v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
        v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
    } else {
        const float* gf = static_cast<const float*>(g) + e;
        const float4 a = ld_stream_f4(gf), b = ld_stream_f4(gf + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

template <bool BF16>
__device__ __forceinline__ float load_grad1(const void* g, int64_t e) {
    if (BF16) return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(g)[e]) << 16);
    return static_cast<const float*>(g)[e];
}

// K3: one warp per 256-element tile, lane l owns 8 consecutive elements (one
// 16-byte bf16 vector, or two fp32 vectors); for every worker it forms
// m = r + g in fp32, adds it to the running sum in worker order, and writes
// the residual back as zero.  The weights get w -= (lr/W) * sum.
template <bool BF16>
__global__ void __launch_bounds__(kThreads, 2)
k_compensated(const CompArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t tile = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nfull = a.n / 256;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tile < nfull) {
        const int64_t e = tile * 256 + 8 * lane;
        const float4 w0 = ld_f4(a.weights + e), w1 = ld_f4(a.weights + e + 4);
        float s[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) s[k] = 0.0f;
        for (int q0 = 0; q0 < a.W; q0 += 4) {
            float gv[4][8];
            float4 r0[4], r1[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (q0 + q < a.W) {
                    load_grad8<BF16>(a.grads.p[q0 + q], e, gv[q]);
                    r0[q] = ld_f4(a.res.p[q0 + q] + e);
                    r1[q] = ld_f4(a.res.p[q0 + q] + e + 4);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (q0 + q < a.W) {
                    s[0] = __fadd_rn(s[0], __fadd_rn(r0[q].x, gv[q][0]));
                    s[1] = __fadd_rn(s[1], __fadd_rn(r0[q].y, gv[q][1]));
                    s[2] = __fadd_rn(s[2], __fadd_rn(r0[q].z, gv[q][2]));
                    s[3] = __fadd_rn(s[3], __fadd_rn(r0[q].w, gv[q][3]));
                    s[4] = __fadd_rn(s[4], __fadd_rn(r1[q].x, gv[q][4]));
                    s[5] = __fadd_rn(s[5], __fadd_rn(r1[q].y, gv[q][5]));
                    s[6] = __fadd_rn(s[6], __fadd_rn(r1[q].z, gv[q][6]));
                    s[7] = __fadd_rn(s[7], __fadd_rn(r1[q].w, gv[q][7]));
                    st_stream_f4(a.res.p[q0 + q] + e, zero);
                    st_stream_f4(a.res.p[q0 + q] + e + 4, zero);
                }
            }
        }
        st_stream_f4(a.weights + e, make_float4(fmaf(-s[0], a.k_lr, w0.x), fmaf(-s[1], a.k_lr, w0.y),
                                                fmaf(-s[2], a.k_lr, w0.z), fmaf(-s[3], a.k_lr, w0.w)));
        st_stream_f4(a.weights + e + 4, make_float4(fmaf(-s[4], a.k_lr, w1.x), fmaf(-s[5], a.k_lr, w1.y),
                                                    fmaf(-s[6], a.k_lr, w1.z), fmaf(-s[7], a.k_lr, w1.w)));
    } else if (tile == nfull) {
        // tail: elements [nfull*256, n), one per lane, 8 rounds
        for (int k = lane; nfull * 256 + k < a.n; k += 32) {
            const int64_t i = nfull * 256 + k;
            float s = 0.0f;
            for (int q = 0; q < a.W; ++q) {
                s = __fadd_rn(s, __fadd_rn(a.res.p[q][i], load_grad1<BF16>(a.grads.p[q], i)));
                a.res.p[q][i] = 0.0f;
            }
            a.weights[i] = fmaf(-s, a.k_lr, a.weights[i]);
        }
    }
}

}  // namespace
}  // namespace gc

using namespace gc;

extern "C" {

const char* gc_status_string(int status) {
    switch (status) {
        case GC_OK: return "GC_OK";
        case GC_ERR_INVALID: return "GC_ERR_INVALID: invalid argument";
        case GC_ERR_ALIGN: return "GC_ERR_ALIGN: data pointer not 16-byte aligned";
        case GC_ERR_CUDA: return "GC_ERR_CUDA: CUDA launch or runtime error";
        case GC_ERR_CAPACITY: return "GC_ERR_CAPACITY: more masked entries than capacity";
        case GC_ERR_TIMEOUT: return "GC_ERR_TIMEOUT: bounded device wait ran out";
        case GC_ERR_CORRUPT: return "GC_ERR_CORRUPT: coded stream does not decode";
        default: return "unknown status";
    }
}

int gc_version(void) { return (1 << 16) | 0; }

int gc_2bit_quantize(const void* grad, gc_dtype dtype, float* residual, uint32_t* codes,
                     int64_t n, float threshold, gc_stream_t stream) {
    if (n < 0 || !finite_pos(threshold) || (dtype != GC_F32 && dtype != GC_BF16)) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!grad || !residual || !codes) return GC_ERR_INVALID;
    if (!aligned16(grad) || !aligned16(residual) || !aligned16(codes)) return GC_ERR_ALIGN;
    const unsigned grid = blocks_for_tiles((n + 511) / 512);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == GC_F32)
        k_2bit_quantize_f32<<<grid, kThreads, 0, s>>>(static_cast<const float*>(grad), residual,
                                                      codes, n, threshold);
    else
        k_2bit_quantize_bf16<<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(grad), residual,
                                                       codes, n, threshold);
    return launch_status();
}

int gc_2bit_quantize_batched(const void* const* grads, gc_dtype dtype, float* const* residuals,
                             uint32_t* const* codes, const int64_t* n, int B, float threshold,
                             gc_stream_t stream) {
    if (B < 1 || B > GC_MAX_WORKERS || !finite_pos(threshold) || (dtype != GC_F32 && dtype != GC_BF16))
        return GC_ERR_INVALID;
    if (!grads || !residuals || !codes || !n) return GC_ERR_INVALID;
    BatchArgs a;
    a.B = B;
    a.t = threshold;
    a.tile_start[0] = 0;
    for (int b = 0; b < B; ++b) {
        if (n[b] < 0) return GC_ERR_INVALID;
        if (n[b] > 0) {
            if (!grads[b] || !residuals[b] || !codes[b]) return GC_ERR_INVALID;
            if (!aligned16(grads[b]) || !aligned16(residuals[b]) || !aligned16(codes[b])) return GC_ERR_ALIGN;
        }
        a.grads.p[b] = grads[b];
        a.res.p[b] = residuals[b];
        a.codes.p[b] = codes[b];
        a.n[b] = n[b];
        a.tile_start[b + 1] = a.tile_start[b] + (n[b] + 511) / 512;
    }
    if (a.tile_start[B] == 0) return GC_OK;
    const unsigned grid = blocks_for_tiles(a.tile_start[B]);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == GC_F32)
        k_2bit_quantize_batched<false><<<grid, kThreads, 0, s>>>(a);
    else
        k_2bit_quantize_batched<true><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

int gc_2bit_dequant_sum_update(const uint32_t* const* codes, int W, int64_t n, float threshold,
                               gc_update kind, float lr, float alpha, const float* center,
                               float* weights, float* out, gc_stream_t stream) {
    if (n < 0 || W < 1 || W > GC_MAX_WORKERS || !finite_pos(threshold)) return GC_ERR_INVALID;
    if (kind != GC_UPD_NONE && kind != GC_UPD_SGD && kind != GC_UPD_EASGD) return GC_ERR_INVALID;
    if (!isfinite(lr) || !isfinite(alpha)) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!codes) return GC_ERR_INVALID;
    DqArgs a;
    for (int w = 0; w < W; ++w) {
        if (!codes[w]) return GC_ERR_INVALID;
        if (!aligned16(codes[w])) return GC_ERR_ALIGN;
        a.codes.p[w] = codes[w];
    }
    if (kind == GC_UPD_NONE) {
        if (!out) return GC_ERR_INVALID;
        if (!aligned16(out)) return GC_ERR_ALIGN;
    } else {
        if (!weights) return GC_ERR_INVALID;
        if (!aligned16(weights)) return GC_ERR_ALIGN;
        if (kind == GC_UPD_EASGD) {
            if (!center) return GC_ERR_INVALID;
            if (!aligned16(center)) return GC_ERR_ALIGN;
        }
    }
    a.W = W;
    a.n = n;
    a.k_out = static_cast<float>(static_cast<double>(threshold) / W);
    a.k_lr = static_cast<float>(static_cast<double>(lr) * threshold / W);
    a.alpha = alpha;
    a.center = center;
    a.weights = weights;
    a.out = out;
    const unsigned grid = blocks_for_tiles((n + 511) / 512);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (kind) {
        case GC_UPD_NONE: k_2bit_dqsum<GC_UPD_NONE><<<grid, kThreads, 0, s>>>(a); break;
        case GC_UPD_SGD: k_2bit_dqsum<GC_UPD_SGD><<<grid, kThreads, 0, s>>>(a); break;
        default: k_2bit_dqsum<GC_UPD_EASGD><<<grid, kThreads, 0, s>>>(a); break;
    }
    return launch_status();
}

}  // extern "C"

namespace {

int step_entry(const void* const* grads, gc_dtype dtype, float* const* residuals, uint32_t* const* codes,
               float* const* local_weights, float local_lr, int W, int64_t n, float threshold,
               gc_update kind, float lr, float alpha, const float* center, float* weights, float* out,
               gc_stream_t stream) {
    const bool local = local_weights != nullptr;
    if (n < 0 || W < 1 || W > GC_MAX_WORKERS || !finite_pos(threshold)) return GC_ERR_INVALID;
    if (dtype != GC_F32 && dtype != GC_BF16) return GC_ERR_INVALID;
    if (kind != GC_UPD_NONE && kind != GC_UPD_SGD && kind != GC_UPD_EASGD) return GC_ERR_INVALID;
    if (!isfinite(lr) || !isfinite(alpha) || !isfinite(local_lr)) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!grads || !residuals || !codes) return GC_ERR_INVALID;
    StepArgs a;
    for (int w = 0; w < W; ++w) {
        if (!grads[w] || !residuals[w] || !codes[w] || (local && !local_weights[w])) return GC_ERR_INVALID;
        if (!aligned16(grads[w]) || !aligned16(residuals[w]) || !aligned16(codes[w])) return GC_ERR_ALIGN;
        if (local && !aligned16(local_weights[w])) return GC_ERR_ALIGN;
        a.grads.p[w] = grads[w];
        a.res.p[w] = residuals[w];
        a.codes.p[w] = codes[w];
        a.local.p[w] = local ? local_weights[w] : nullptr;
    }
    if (kind == GC_UPD_NONE) {
        if (!out) return GC_ERR_INVALID;
        if (!aligned16(out)) return GC_ERR_ALIGN;
    }
    if (kind != GC_UPD_NONE || local) {
        if (!weights) return GC_ERR_INVALID;
        if (!aligned16(weights)) return GC_ERR_ALIGN;
    }
    if (kind == GC_UPD_EASGD) {
        if (!center) return GC_ERR_INVALID;
        if (!aligned16(center)) return GC_ERR_ALIGN;
    }
    a.W = W;
    a.n = n;
    a.t = threshold;
    a.k_out = static_cast<float>(static_cast<double>(threshold) / W);
    a.k_lr = static_cast<float>(static_cast<double>(lr) * threshold / W);
    a.alpha = alpha;
    a.local_lr = local_lr;
    a.center = center;
    a.weights = weights;
    a.out = out;
    const unsigned grid = blocks_for_tiles((n + 511) / 512);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == GC_BF16) {
        if (local) launch_step<true, true>(kind, grid, s, a); else launch_step<true, false>(kind, grid, s, a);
    } else {
        if (local) launch_step<false, true>(kind, grid, s, a); else launch_step<false, false>(kind, grid, s, a);
    }
    return launch_status();
}

}  // namespace

extern "C" {

int gc_2bit_step(const void* const* grads, gc_dtype dtype, float* const* residuals, uint32_t* const* codes,
                 int W, int64_t n, float threshold, gc_update kind, float lr, float alpha,
                 const float* center, float* weights, float* out, gc_stream_t stream) {
    return step_entry(grads, dtype, residuals, codes, nullptr, 0.0f, W, n, threshold, kind, lr, alpha, center,
                      weights, out, stream);
}

int gc_2bit_step_local(const void* const* grads, gc_dtype dtype, float* const* residuals,
                       uint32_t* const* codes, float* const* local_weights, float local_lr, int W, int64_t n,
                       float threshold, gc_update kind, float lr, float alpha, const float* center,
                       float* weights, float* out, gc_stream_t stream) {
    if (!local_weights) return GC_ERR_INVALID;
    return step_entry(grads, dtype, residuals, codes, local_weights, local_lr, W, n, threshold, kind, lr, alpha,
                      center, weights, out, stream);
}

int gc_2bit_quantize_steps(const void* const* grads, gc_dtype dtype, float* residual, uint32_t* const* codes,
                           float* const* out, int S, int64_t n, float threshold, gc_stream_t stream) {
    if (n < 0 || S < 1 || S > GC_MAX_WORKERS || !finite_pos(threshold)) return GC_ERR_INVALID;
    if (dtype != GC_F32 && dtype != GC_BF16) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!grads || !residual || !codes) return GC_ERR_INVALID;
    if (!aligned16(residual)) return GC_ERR_ALIGN;
    StepsArgs a;
    for (int st = 0; st < S; ++st) {
        if (!grads[st] || !codes[st] || (out && !out[st])) return GC_ERR_INVALID;
        if (!aligned16(grads[st]) || !aligned16(codes[st]) || (out && !aligned16(out[st]))) return GC_ERR_ALIGN;
        a.grads.p[st] = grads[st];
        a.codes.p[st] = codes[st];
        a.out.p[st] = out ? out[st] : nullptr;
    }
    a.res = residual;
    a.S = S;
    a.has_out = out != nullptr;
    a.n = n;
    a.t = threshold;
    const unsigned grid = blocks_for_tiles((n + 511) / 512);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == GC_BF16)
        k_2bit_steps<true><<<grid, kThreads, 0, s>>>(a);
    else
        k_2bit_steps<false><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

int gc_2bit_quantize_local(const void* const* grads, gc_dtype dtype, float* const* residuals,
                           uint32_t* const* codes, const float* weights, float* const* local_weights,
                           int B, int64_t n, float threshold, float local_lr, gc_stream_t stream) {
    if (n < 0 || B < 1 || B > GC_MAX_WORKERS || !finite_pos(threshold) || !isfinite(local_lr) ||
        (dtype != GC_F32 && dtype != GC_BF16))
        return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!grads || !residuals || !codes || !weights || !local_weights) return GC_ERR_INVALID;
    if (!aligned16(weights)) return GC_ERR_ALIGN;
    LocalArgs a;
    for (int b = 0; b < B; ++b) {
        if (!grads[b] || !residuals[b] || !codes[b] || !local_weights[b]) return GC_ERR_INVALID;
        if (!aligned16(grads[b]) || !aligned16(residuals[b]) || !aligned16(codes[b]) || !aligned16(local_weights[b]))
            return GC_ERR_ALIGN;
        a.grads.p[b] = grads[b];
        a.res.p[b] = residuals[b];
        a.codes.p[b] = codes[b];
        a.local.p[b] = local_weights[b];
    }
    a.weights = weights;
    a.B = B;
    a.n = n;
    a.t = threshold;
    a.local_lr = local_lr;
    const unsigned grid = blocks_for_tiles((n + 511) / 512 * B);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == GC_F32)
        k_2bit_quantize_local<false><<<grid, kThreads, 0, s>>>(a);
    else
        k_2bit_quantize_local<true><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

int gc_compensated_sum_update(const void* const* grads, gc_dtype dtype, float* const* residuals,
                              int W, int64_t n, float lr, float* weights, gc_stream_t stream) {
    if (n < 0 || W < 1 || W > GC_MAX_WORKERS || !isfinite(lr)) return GC_ERR_INVALID;
    if (dtype != GC_F32 && dtype != GC_BF16) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!grads || !residuals || !weights) return GC_ERR_INVALID;
    CompArgs a;
    for (int w = 0; w < W; ++w) {
        if (!grads[w] || !residuals[w]) return GC_ERR_INVALID;
        if (!aligned16(grads[w]) || !aligned16(residuals[w])) return GC_ERR_ALIGN;
        a.grads.p[w] = grads[w];
        a.res.p[w] = residuals[w];
    }
    if (!aligned16(weights)) return GC_ERR_ALIGN;
    a.W = W;
    a.n = n;
    a.k_lr = static_cast<float>(static_cast<double>(lr) / W);
    a.weights = weights;
    // one warp per 256-element tile, plus one for the partial last tile
    const unsigned grid = blocks_for_tiles(n / 256 + 1);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == GC_BF16)
        k_compensated<true><<<grid, kThreads, 0, s>>>(a);
    else
        k_compensated<false><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

}  // extern "C"
