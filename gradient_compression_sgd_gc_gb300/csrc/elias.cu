// elias.cu -- lossless Elias-omega coding of QSGD's quantised tuple.
//
// "QSGD: Communication-Efficient SGD via Gradient Quantization and Encoding",
// Knowl 2, dense regime: the bucket's norm as a 32-bit float, then every
// coordinate in turn as Elias'(level) = Elias-omega(level + 1), followed by
// its sign bit when the level is not zero.  Stream layout: 32-bit words, most
// significant bit first; every bucket starts on a word boundary and its last
// word is padded with zero bits; offsets[b] is bucket b's first word and
// offsets[nbuckets] the stream's length, so that buckets decode in parallel.
//
// Encode = one launch reading the codes once.  Each CTA takes a chunk of up
// to 64 buckets (a ticket, so chunks go out in the order CTAs start) and
// stages all of it in shared memory: its warps assemble the buckets (a
// 256-entry table turns a code byte into its codeword bits and length; one
// warp scan of bit lengths per 32 code words, then shared-memory atomicOr of
// at most three words per lane); the chunk's word count is published, its
// first word taken from a decoupled look-back over the chunks before it, and
// the chunk stored with coalesced 32-bit writes.
// Decode: one thread per bucket (or per quarter or half bucket, from the
// quarter marks) walks its stream with a 64-bit window; an 11-bit (4-bit
// codes) or 12-bit (8-bit codes) lookahead table, built by the compiler,
// decodes up to 8 or 4 whole codewords per step, and an 8-bit one the rest;
// each CTA first copies its buckets' words to shared memory.
#include <atomic>

#include "gc_common.cuh"
#include "../../include/gc_gb300_testing.h"

namespace gc {
namespace {

constexpr int kChunk = 64;                          // buckets per encoding CTA, at most
constexpr int kEncodeStageWords = 9216;             // the dense encoder's staging per CTA, at most
constexpr int kSparseStageWords = 9600;             // the sparse encoder's staging per CTA, at most
constexpr size_t kTicketBytes = 16;

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool valid_bucket(int bucket) {
    return bucket == 128 || bucket == 256 || bucket == 512 || bucket == 1024 || bucket == 2048;
}

// Longest codeword + sign a code of the given width can produce: level 7
// (omega(8) = 7 bits, + sign) for 4-bit codes, level 127 (omega(128) = 14
// bits, + sign) for 8-bit codes.  The bound holds for any code content.
inline int max_code_bits(bool four) { return four ? 8 : 15; }

inline int64_t bucket_max_words(int64_t len, bool four) {
    return 1 + div_up(len * max_code_bits(four), 32);
}

// ---------------------------------------------------------------- codewords

// Elias omega of N >= 1 (Elias 1975): the terminating 0, preceded by the
// binary form of N, preceded by that of (digits of N) - 1, and so on while
// the number is above 1.  Returns the length; *pat holds the bits
// right-aligned.
__device__ __forceinline__ int omega(uint32_t N, uint32_t* pat) {
    uint32_t p = 0;
    int len = 1;
    while (N > 1) {
        const int L = 32 - __clz(N);
        p |= N << len;
        len += L;
        N = static_cast<uint32_t>(L - 1);
    }
    *pat = p;
    return len;
}

// One code's stream bits, packed as (pattern << 5) | length.
__device__ __forceinline__ uint32_t code_entry(uint32_t sign, uint32_t level) {
    uint32_t pat;
    int len = omega(level + 1u, &pat);
    if (level) {
        pat = (pat << 1) | sign;
        ++len;
    }
    return (pat << 5) | static_cast<uint32_t>(len);
}

// Table entry of a code byte: two 4-bit codes (high nibble first) or one
// 8-bit code, at most 16 bits of stream.
template <bool FOUR>
__device__ __forceinline__ uint32_t byte_entry(uint32_t byte) {
    if (FOUR) {
        const uint32_t hi = code_entry((byte >> 7) & 1u, (byte >> 4) & 7u);
        const uint32_t lo = code_entry((byte >> 3) & 1u, byte & 7u);
        const uint32_t llo = lo & 31u;
        return ((((hi >> 5) << llo) | (lo >> 5)) << 5) | ((hi & 31u) + llo);
    }
    return code_entry(byte >> 7, byte & 127u);
}

template <bool FOUR>
__device__ __forceinline__ void build_lut(uint32_t* lut) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) lut[i] = byte_entry<FOUR>(static_cast<uint32_t>(i));
}

// The bytes of code word k of a bucket (k counts 32-bit words from the
// bucket's first byte): how many are valid and whether the last valid one
// holds only its high nibble (odd-length last bucket with 4-bit codes).
struct BucketBytes {
    const uint8_t* base;   // first code byte of the bucket (64-byte aligned)
    int valid;             // code bytes of the bucket
    bool half;             // the last byte carries one 4-bit code
};

template <bool FOUR>
__device__ __forceinline__ BucketBytes bucket_bytes(const uint8_t* codes, int64_t n, int d, int64_t b) {
    const int64_t lo = b * d;
    const int len = static_cast<int>((n - lo < d ? n - lo : static_cast<int64_t>(d)));
    BucketBytes bb;
    bb.base = codes + (FOUR ? lo / 2 : lo);
    bb.valid = FOUR ? (len + 1) / 2 : len;
    bb.half = FOUR && (len & 1);
    return bb;
}

// The stream bits of code word k of a bucket, right-aligned in acc (at most
// 64 bits: four bytes of at most 16 bits each).
template <bool FOUR>
__device__ __forceinline__ int word_bits(const BucketBytes& bb, int k, const uint32_t* lut, uint64_t& acc) {
    acc = 0;
    const int b0 = 4 * k;
    if (b0 >= bb.valid) return 0;
    const int nv = min(4, bb.valid - b0);
    uint32_t w;
    if (nv == 4) {
        w = __ldg(reinterpret_cast<const uint32_t*>(bb.base) + k);
    } else {
        w = 0;
        for (int j = 0; j < nv; ++j) w |= static_cast<uint32_t>(__ldg(bb.base + b0 + j)) << (8 * j);
    }
    int len = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j < nv) {
            const uint32_t byte = (w >> (8 * j)) & 255u;
            uint32_t e;
            if (FOUR && bb.half && b0 + j == bb.valid - 1) {
                // only the high nibble is a code: drop the low nibble's level-0 bit
                e = lut[byte & 0xF0u];
                e = ((e >> 6) << 5) | ((e & 31u) - 1u);
            } else {
                e = lut[byte];
            }
            const int l = static_cast<int>(e & 31u);
            acc = (acc << l) | (e >> 5);
            len += l;
        }
    }
    return len;
}

__device__ __forceinline__ int warp_incl_sum(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Bits `len` (right-aligned in acc, len <= 64) OR-ed into the bucket's
// staging words at bit position pos (most significant bit first).
__device__ __forceinline__ void emit(uint32_t* stage, uint32_t pos, uint64_t acc, int len) {
    if (len == 0) return;
    const uint64_t A = acc << (64 - len);
    const uint32_t w0 = pos >> 5, sh = pos & 31u;
    const uint32_t x0 = static_cast<uint32_t>(A >> (32 + sh));
    const uint32_t x1 = static_cast<uint32_t>(A >> sh);
    const uint32_t x2 = sh ? static_cast<uint32_t>(A << (32 - sh)) : 0u;
    if (x0) atomicOr(stage + w0, x0);
    if (x1) atomicOr(stage + w0 + 1, x1);
    if (x2) atomicOr(stage + w0 + 2, x2);
}

// ---------------------------------------------------------------- full buckets

// A full bucket is Bb = d/2 (4-bit) or d (8-bit) code bytes, a multiple of
// 64, read as P = Bb/16 pieces of 16 bytes.  G = min(P, 32) consecutive
// lanes share a bucket; a warp covers 32/G buckets per pass and a bucket
// takes P/G rounds.
struct Geometry {
    int Bb, P, G;
};

template <bool FOUR>
__device__ __forceinline__ Geometry geometry(int d) {
    Geometry g;
    g.Bb = FOUR ? d / 2 : d;
    g.P = g.Bb / 16;
    g.G = g.P < 32 ? g.P : 32;
    return g;
}

// ---------------------------------------------------------------- encode

// The encoder's workspace: a 16-byte header (the device status, then the
// CTA ticket) and one look-back state word per chunk of buckets (its word
// count, then its inclusive prefix).
struct EncodeWs {
    int* status;
    uint32_t* ticket;
    uint64_t* state;    // [nchunks] (at most nbuckets)
};

inline size_t encode_ws_bytes(int64_t nbuckets) {
    return kTicketBytes + static_cast<size_t>(div_up(nbuckets * 8, 16) * 16);
}

EncodeWs encode_ws(void* ws) {
    char* p = static_cast<char*>(ws);
    return EncodeWs{reinterpret_cast<int*>(p), reinterpret_cast<uint32_t*>(p + 4),
                    reinterpret_cast<uint64_t*>(p + kTicketBytes)};
}

// Once every bucket of the CTA's chunk is staged (s_nw[lb] = its words), by
// warp 0: publishes the chunk's word count, takes the chunk's first word from
// the look-back over the chunks before it (Merrill and Garland's decoupled
// look-back, bounded: a wait that runs out records GC_ERR_TIMEOUT in the
// workspace), then its inclusive prefix; writes each bucket's first word to
// offsets and to s_nw, the stream's length when this is the last chunk, and
// the chunk's end to *s_end.  At most 64 buckets per chunk.
__device__ __forceinline__ void chunk_offsets(const EncodeWs& ws, int64_t chunk, int64_t b0, int nbc,
                                              int64_t nbuckets, uint32_t* offsets, uint32_t* s_nw,
                                              uint32_t* s_end, uint64_t wait_ns, int64_t withhold, int lane) {
    const uint32_t c0 = 2 * lane < nbc ? s_nw[2 * lane] : 0u;
    const uint32_t c1 = 2 * lane + 1 < nbc ? s_nw[2 * lane + 1] : 0u;
    const uint32_t incl = static_cast<uint32_t>(warp_incl_sum(static_cast<int>(c0 + c1), lane));
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    const bool publish = chunk != withhold;
    if (lane == 0 && publish) st_state(ws.state + chunk, (chunk == 0 ? kFlagPrefix : kFlagAgg) | total);
    bool timed_out = false;
    const uint64_t base = chunk == 0 ? 0 : lookback_exclusive(ws.state, chunk, lane, wait_ns, 0u, timed_out);
    if (lane == 0) {
        if (chunk != 0 && publish) st_state(ws.state + chunk, kFlagPrefix | (base + total));
        if (timed_out) atomicExch(ws.status, GC_ERR_TIMEOUT);
        if (b0 + nbc == nbuckets) offsets[nbuckets] = static_cast<uint32_t>(base) + total;
        *s_end = static_cast<uint32_t>(base) + total;
    }
    const uint32_t o0 = static_cast<uint32_t>(base) + incl - c0 - c1;
    if (2 * lane < nbc) {
        s_nw[2 * lane] = o0;
        offsets[b0 + 2 * lane] = o0;
    }
    if (2 * lane + 1 < nbc) {
        s_nw[2 * lane + 1] = o0 + c0;
        offsets[b0 + 2 * lane + 1] = o0 + c0;
    }
}

// Writes the chunk's staged buckets to the stream: warp w takes buckets w,
// w + 8, ..., each from its first word (s_nw) to the next bucket's, coalesced.
__device__ __forceinline__ void write_chunk(const uint32_t* stages, int stride, const uint32_t* s_nw,
                                            uint32_t chunk_end, int nbc, uint32_t* words, int warp, int lane) {
    for (int lb = warp; lb < nbc; lb += kWarpsPerBlock) {
        const uint32_t off = s_nw[lb];
        const uint32_t nw = (lb + 1 < nbc ? s_nw[lb + 1] : chunk_end) - off;
        const uint32_t* st = stages + lb * stride;
        uint32_t* dst = words + off;
        for (uint32_t k = lane; k < nw; k += 32) dst[k] = st[k];
    }
}


struct EncodeArgs {
    const uint8_t* codes;
    const float* norms;
    int64_t n;
    int d;
    int64_t nbuckets;
    uint32_t* words;
    uint32_t* offsets;
    int stage_stride;   // staging words per bucket
    int slots;          // buckets per warp and pass (32 / G)
    uint16_t* marks;    // quarter marks [3 * nbuckets], or null
    EncodeWs ws;
    uint64_t wait_ns;   // bound on each look-back wait
    int64_t withhold;   // test hook: this chunk never publishes (-1: none)
    int chunk;          // buckets per CTA (<= kChunk), all staged at once
};


// The stream bits of 16 code bytes (table entries e[]) OR-ed into the
// staging words from bit position `start`: the entries are joined two at a
// time (at most 16 + 16 bits), and a 64-bit shift register (hi:lo) collects
// the pairs and hands over every completed word (at most one per pair).
__device__ __forceinline__ void emit_piece(uint32_t* stage, uint32_t start, const uint32_t (&e)[16]) {
    uint32_t wi = start >> 5;
    int nacc = static_cast<int>(start & 31u);
    uint32_t hi = 0u, lo = 0u;
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        const int l1 = static_cast<int>(e[j + 1] & 31u);
        const int l = static_cast<int>(e[j] & 31u) + l1;                 // <= 32
        const uint32_t pat = ((e[j] >> 5) << l1) | (e[j + 1] >> 5);
        hi = __funnelshift_lc(lo, hi, l);
        lo = __funnelshift_lc(0u, lo, l) | pat;
        nacc += l;
        if (nacc >= 32) {
            atomicOr(stage + wi, __funnelshift_r(lo, hi, nacc - 32));
            ++wi;
            nacc -= 32;
        }
    }
    if (nacc > 0) atomicOr(stage + wi, lo << (32 - nacc));
}

// Register bound for 5 CTAs per SM (48 registers, no spills).  Every bucket
// of the CTA's chunk is staged at once (chunk x stage_stride words), so the
// chunk's word count is known when its encoding ends: it is published then,
// and the look-back over the chunks before it rarely waits.
template <bool FOUR>
__global__ void __launch_bounds__(kThreads, 5) k_elias_encode(EncodeArgs a) {
    extern __shared__ uint32_t smem[];
    __shared__ uint32_t s_chunk, s_end;
    __shared__ uint32_t s_nw[kChunk];             // words of each bucket, then its first word
    uint32_t* lut = smem;
    uint32_t* stages = smem + 256;                // [chunk][stage_stride]
    build_lut<FOUR>(lut);
    const int nstage = a.chunk * a.stage_stride;
    for (int i = threadIdx.x; i < nstage; i += kThreads) stages[i] = 0u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // Chunks are taken in the order CTAs start (a ticket), so every chunk a
    // look-back waits for belongs to a CTA already running: the waits end.
    if (threadIdx.x == 0) s_chunk = atomicAdd(a.ws.ticket, 1u);
    __syncthreads();
    const int64_t chunk = s_chunk;
    const int64_t b0 = chunk * a.chunk;
    const Geometry g = geometry<FOUR>(a.d);
    const int nbc = static_cast<int>(a.nbuckets - b0 < a.chunk ? a.nbuckets - b0 : a.chunk);
    const bool ragged = (a.n % a.d) != 0 && b0 + nbc == a.nbuckets;
    const int nfull = nbc - (ragged ? 1 : 0);
    const int grp = lane / g.G, gl = lane % g.G;
    const uint4* src = reinterpret_cast<const uint4*>(a.codes + b0 * g.Bb);
    // Items = (bucket pass j, round r), r < R (1, 2 or 4), counted without
    // division; the next item's 16 bytes and norm are loaded while the
    // current one is coded.
    const int R = g.P / g.G;
    const int first = warp * a.slots, step = kWarpsPerBlock * a.slots;
    const int passes = nfull > first ? (nfull - first + step - 1) / step : 0;
    const int items = passes * R;
    auto load_item = [&](int lb, int r, uint4& v, float& nrm) {
        if (lb < nfull) {
            v = __ldg(src + lb * g.P + r * g.G + gl);
            nrm = __ldg(a.norms + b0 + lb);
        }
    };
    uint4 vn = make_uint4(0u, 0u, 0u, 0u);
    float nn = 0.0f;
    if (items) load_item(first + grp, 0, vn, nn);
    uint32_t pos = 32;
    int r = 0, lb = first + grp;                  // the current item
    for (int it = 0; it < items; ++it) {
        const bool active = lb < nfull;
        uint32_t* stage = stages + lb * a.stage_stride;
        const uint4 v = vn;
        const float nrm = nn;
        const bool last_round = r + 1 == R;
        const int nlb = last_round ? lb + step : lb, nr = last_round ? 0 : r + 1;
        if (it + 1 < items) load_item(nlb, nr, vn, nn);
        if (r == 0) {
            pos = 32;
            if (active && gl == 0) stage[0] = __float_as_uint(nrm);
        }
        uint32_t e[16];
        uint32_t len = 0;
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                e[4 * i + j] = lut[(w[i] >> (8 * j)) & 255u];
                len += e[4 * i + j] & 31u;
            }
        if (!active) len = 0;
        uint32_t incl = len;
        for (int o = 1; o < g.G; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (gl >= o) incl += t;
        }
        if (active) emit_piece(stage, pos + incl - len, e);
        if (a.marks && active) {
            // a piece that starts a quarter of the bucket records its start bit
            // (a quarter, d / 4, is a power of two)
            const int c = (r * g.G + gl) * (FOUR ? 32 : 16);
            const int qs = __ffs(a.d) - 3;
            if (c > 0 && (c & ((1 << qs) - 1)) == 0)
                a.marks[3 * (b0 + lb) + (c >> qs) - 1] = static_cast<uint16_t>(pos + incl - len);
        }
        pos += __shfl_sync(0xffffffffu, incl, grp * g.G + g.G - 1);
        if (last_round && active && gl == 0) s_nw[lb] = (pos + 31) >> 5;
        lb = nlb;
        r = nr;
    }
    if (ragged && warp == kWarpsPerBlock - 1) {
        // the ragged last bucket, by one warp
        const int lb = nfull;
        const int64_t b = b0 + lb;
        const BucketBytes bb = bucket_bytes<FOUR>(a.codes, a.n, a.d, b);
        const int nw_in = (bb.valid + 3) >> 2;
        uint32_t* st0 = stages + lb * a.stage_stride;
        if (lane == 0) st0[0] = __float_as_uint(__ldg(a.norms + b));
        uint32_t pos = 32;
        const int q = a.d / 4;
        const int blen = static_cast<int>(a.n - b * a.d);
        for (int k0 = 0; k0 < nw_in; k0 += 32) {
            uint64_t acc;
            const int len = word_bits<FOUR>(bb, k0 + lane, lut, acc);
            const int incl = warp_incl_sum(len, lane);
            emit(st0, pos + static_cast<uint32_t>(incl - len), acc, len);
            if (a.marks) {
                const int c = (k0 + lane) * (FOUR ? 8 : 4);
                if (c > 0 && c < blen && c % q == 0)
                    a.marks[3 * b + c / q - 1] = static_cast<uint16_t>(pos + static_cast<uint32_t>(incl - len));
            }
            pos += static_cast<uint32_t>(__shfl_sync(0xffffffffu, incl, 31));
        }
        // quarters that start past the short bucket's end: the end
        if (a.marks && lane < 3 && (lane + 1) * q >= blen) a.marks[3 * b + lane] = static_cast<uint16_t>(pos);
        if (lane == 0) s_nw[lb] = (pos + 31) >> 5;
    }
    __syncthreads();
    if (warp == 0)
        chunk_offsets(a.ws, chunk, b0, nbc, a.nbuckets, a.offsets, s_nw, &s_end, a.wait_ns, a.withhold, lane);
    __syncthreads();
    write_chunk(stages, a.stage_stride, s_nw, s_end, nbc, a.words, warp, lane);
}

// ---------------------------------------------------------------- decode

// One launch decodes W streams (blockIdx.y = stream): a decoding thread owns
// one bucket, so a single stream of 61 M coordinates fills only about a
// quarter of the GPU's warp slots; W streams fill W times more.
struct DecodeArgs {
    PtrTable<const uint32_t*> words;
    PtrTable<const uint32_t*> offsets;
    PtrTable<uint8_t*> codes;
    PtrTable<float*> norms;
    int64_t n;
    int d;
    int64_t nbuckets;
    int s;
    int* status;
    uint32_t stage_cap;   // shared words for the staged stream words (at most stage_cap - 3 of them)
    const uint16_t* marks;   // quarter marks of stream 0 (segmented decode), else null
    int bpc;              // buckets per CTA (at most its threads / parts; balanced_bpc)
};

// Lookahead bits of the multi-codeword table: 11 for 4-bit codes, 12 for
// 8-bit ones (measured fastest of 10-12 on the QSGD workloads).
template <bool FOUR>
__host__ __device__ constexpr int win_bits() { return FOUR ? 11 : 12; }

// The codeword (+ sign) at the top of a W-bit window x, as
// (level << 5) | (sign << 4) | length, or 0 when it does not end inside the
// window.  W = 8 gives the single-codeword table; evaluable at compile time.
template <int W>
__host__ __device__ constexpr uint32_t window_entry(uint32_t x) {
    constexpr uint32_t kMask = (1u << W) - 1u;
    int pos = 0;
    uint32_t N = 1;
    for (;;) {
        if (pos >= W) return 0u;
        const uint32_t bit = (x >> (W - 1 - pos)) & 1u;
        ++pos;
        if (!bit) break;
        if (pos + static_cast<int>(N) > W) return 0u;
        const uint32_t v = ((x << (pos - 1)) & kMask) >> (W - (N + 1));
        pos += static_cast<int>(N);
        N = v;
    }
    const uint32_t level = N - 1u;
    uint32_t sign = 0u;
    if (level) {
        if (pos >= W) return 0u;
        sign = (x >> (W - 1 - pos)) & 1u;
        ++pos;
    }
    return (level << 5) | (sign << 4) | static_cast<uint32_t>(pos);
}

// Multi-codeword table entry: every whole codeword (+ sign) at the front of a
// win_bits()-bit window, up to KMAX of them (the codes that fill 32 bits) and
// stopping before a level the code width cannot hold.  Bits 0-3: bits used;
// 4-7: codeword count (0 when the first codeword is longer than the window);
// 8-14: the largest level (checked against s at run time); 32-63: the codes
// in the output layout, first one most significant.
template <bool FOUR>
__host__ __device__ constexpr uint64_t multi_window_entry(uint32_t x) {
    constexpr uint32_t KMAX = FOUR ? 8 : 4;
    constexpr uint32_t kMaxLevel = FOUR ? 7 : 127;
    constexpr int W = win_bits<FOUR>();
    constexpr uint32_t kMask = (1u << W) - 1u;
    uint32_t used = 0, k = 0, packed = 0, top = 0;
    while (k < KMAX && used < static_cast<uint32_t>(W)) {
        const uint32_t t = window_entry<W>((x << used) & kMask);
        const uint32_t len = t & 15u;
        if (!t || used + len > static_cast<uint32_t>(W)) break;
        const uint32_t level = t >> 5, sign = (t >> 4) & 1u;
        if (level > kMaxLevel) break;
        packed = FOUR ? (packed << 4) | (sign << 3) | level : (packed << 8) | (sign << 7) | level;
        top = level > top ? level : top;
        used += len;
        ++k;
    }
    return (static_cast<uint64_t>(packed) << 32) | (top << 8) | (k << 4) | used;
}

template <bool FOUR>
struct MultiTable {
    uint64_t e[1 << win_bits<FOUR>()];
};

template <bool FOUR>
constexpr MultiTable<FOUR> make_multi_table() {
    MultiTable<FOUR> t{};
    for (uint32_t x = 0; x < (1u << win_bits<FOUR>()); ++x) t.e[x] = multi_window_entry<FOUR>(x);
    return t;
}

// Built by the compiler; each decoding CTA copies its table to shared memory.
__device__ const MultiTable<true> kMulti4 = make_multi_table<true>();
__device__ const MultiTable<false> kMulti8 = make_multi_table<false>();

// Output side of the decoder: codes arrive in units of 4 or 8 bits, first
// code most significant, and leave as 16-byte stores.
template <bool FOUR>
struct CodeWriter {
    static constexpr int kUnit = FOUR ? 4 : 8;
    static constexpr int kPerWord = 32 / kUnit;
    uint32_t ahi = 0, alo = 0;   // pending units, right-aligned
    int pend = 0;
    uint32_t b0 = 0, b1 = 0, b2 = 0, b3 = 0;   // completed words, newest in b3
    int nbuf = 0;
    uint32_t* out;               // 16-byte aligned

    __device__ __forceinline__ void put(uint32_t packed, int k) {
        const int sh = k * kUnit;                    // <= 32
        ahi = __funnelshift_lc(alo, ahi, sh);
        alo = __funnelshift_lc(0u, alo, sh) | packed;
        pend += k;
        if (pend >= kPerWord) {
            pend -= kPerWord;
            const uint32_t w = __funnelshift_r(alo, ahi, pend * kUnit);
            b0 = b1;
            b1 = b2;
            b2 = b3;
            b3 = __byte_perm(w, 0u, 0x0123);
            if (++nbuf == 4) {
                *reinterpret_cast<uint4*>(out) = make_uint4(b0, b1, b2, b3);
                out += 4;
                nbuf = 0;
            }
        }
    }

    __device__ __forceinline__ void finish() {
        if (nbuf == 3) {
            out[0] = b1;
            out[1] = b2;
            out[2] = b3;
        } else if (nbuf == 2) {
            out[0] = b2;
            out[1] = b3;
        } else if (nbuf == 1) {
            out[0] = b3;
        }
        if (pend) {
            const uint32_t w = __byte_perm(alo << (32 - pend * kUnit), 0u, 0x0123);
            uint8_t* tail = reinterpret_cast<uint8_t*>(out + nbuf);
            const int nbytes = (pend * kUnit + 7) / 8;
            for (int j = 0; j < nbytes; ++j) tail[j] = static_cast<uint8_t>(w >> (8 * j));
        }
    }
};

// One thread per bucket: its stream is walked with a 64-bit window (whi:wlo,
// `have` valid bits from the top, the next word waiting in `pre`).
// S > 1: each thread decodes 1/S of a bucket (S = 2 or 4), from the
// bucket's quarter marks (qsgd_elias_decode_quarters).  A CTA covers
// DecodeArgs::bpc buckets, at most its threads / S.
// The CTA's NT tasks in order of stream length: a counting sort on `key`
// (the task's word count, capped at 255), so that the threads of a warp walk
// streams of about the same length instead of idling on the warp's longest
// one.  Returns the task (a thread index of the CTA) this thread takes.
template <int NT>
__device__ __forceinline__ int task_by_length(uint32_t key) {
    static_assert(NT % 256 == 0 && NT <= 1024, "256 bins, scanned by the first 8 warps");
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_wsum[8];
    __shared__ uint16_t s_order[NT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < 256) s_hist[threadIdx.x] = 0u;
    __syncthreads();
    const uint32_t pos = atomicAdd(s_hist + key, 1u);
    __syncthreads();
    const uint32_t h = threadIdx.x < 256 ? s_hist[threadIdx.x] : 0u;
    const int incl = warp_incl_sum(static_cast<int>(h), lane);
    if (threadIdx.x < 256 && lane == 31) s_wsum[warp] = static_cast<uint32_t>(incl);
    __syncthreads();
    uint32_t start = static_cast<uint32_t>(incl) - h;
#pragma unroll
    for (int w = 0; w < 8; ++w) start += w < warp ? s_wsum[w] : 0u;
    __syncthreads();
    if (threadIdx.x < 256) s_hist[threadIdx.x] = start;     // bin starts
    __syncthreads();
    s_order[s_hist[key] + pos] = static_cast<uint16_t>(threadIdx.x);
    __syncthreads();
    return s_order[threadIdx.x];
}

// A decoding CTA's copy of the nst words at g (16-byte aligned buffer,
// g = words + base) to shared memory in 16-byte pieces: the words before the
// first 16-byte boundary (`lead`, at most 3), the vectors, and the words after
// the last one (`tail`, at most 3).  stage_issue loads the first R x NT
// vectors and the edge words into registers at the start of the CTA, so that
// those loads are in flight during its other set-up; stage_store writes them
// and copies any further vectors.  Word i goes to s[i], where s = the shared
// array + (base & 3), so that the vectors land on 16-byte boundaries: the
// array holds nst + 3 words.  Every load lies inside g[0, nst).
struct StageSplit {
    uint32_t lead, nv, tail;
};

__device__ __forceinline__ StageSplit stage_split(uint32_t base, uint32_t nst) {
    StageSplit p;
    const uint32_t a0 = (4u - (base & 3u)) & 3u;
    p.lead = a0 < nst ? a0 : nst;
    p.nv = (nst - p.lead) >> 2;
    p.tail = nst - p.lead - 4u * p.nv;
    return p;
}

// Thread t < lead holds word t, thread 4 + t < 4 + tail the t-th word after the vectors.
__device__ __forceinline__ bool edge_word(const StageSplit& p, uint32_t& i) {
    const uint32_t t = threadIdx.x;
    if (t < p.lead) {
        i = t;
        return true;
    }
    if (t >= 4u && t - 4u < p.tail) {
        i = p.lead + 4u * p.nv + (t - 4u);
        return true;
    }
    return false;
}

template <int NT, int R>
__device__ __forceinline__ void stage_issue(const uint32_t* g, const StageSplit& p, uint4 (&v)[R], uint32_t& edge) {
    const uint4* gv = reinterpret_cast<const uint4*>(g + p.lead);
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const uint32_t i = threadIdx.x + j * NT;
        if (i < p.nv) v[j] = __ldg(gv + i);
    }
    uint32_t i;
    edge = edge_word(p, i) ? __ldg(g + i) : 0u;
}

template <int NT, int R>
__device__ __forceinline__ void stage_store(const uint32_t* g, const StageSplit& p, const uint4 (&v)[R],
                                            uint32_t edge, uint32_t* s) {
    uint4* sv = reinterpret_cast<uint4*>(s + p.lead);
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const uint32_t i = threadIdx.x + j * NT;
        if (i < p.nv) sv[i] = v[j];
    }
    uint32_t i;
    if (edge_word(p, i)) s[i] = edge;
    const uint4* gv = reinterpret_cast<const uint4*>(g + p.lead);
    for (uint32_t k = threadIdx.x + R * NT; k < p.nv; k += 4 * NT) {
        uint4 w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (k + j * NT < p.nv) w[j] = __ldg(gv + k + j * NT);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (k + j * NT < p.nv) sv[k + j * NT] = w[j];
    }
}

// Threads per decoding CTA and the resident CTAs per SM its shared staging
// is sized for.  Each CTA copies the codeword tables (19 KB for 4-bit codes,
// 35 KB for 8-bit codes) to shared memory, so fewer, larger CTAs leave more
// of it for staging stream words.  4-bit codes: 256 threads, 4 CTAs per SM a
// bucket per thread (one stream of 61 M coordinates fills them in one wave
// at 197 buckets a CTA, balanced_bpc), 6 with a part of a bucket per thread;
// 512- or 1024-thread CTAs measured no faster.  8-bit codes: one 1024-thread
// CTA per SM a bucket per thread (all its words staged),
// three 512-thread CTAs a part per thread (72 -> 70 us, 85 -> 76 us with L2
// flushed).
template <bool FOUR, int S>
__host__ __device__ constexpr int decode_threads() { return FOUR ? 256 : (S == 1 ? 1024 : 512); }
template <bool FOUR, int S>
__host__ __device__ constexpr int decode_ctas_per_sm() { return FOUR ? (S > 1 ? 6 : 4) : (S == 1 ? 1 : 3); }

// Parts per bucket in qsgd_elias_decode_quarters: 4-bit codes, a thread per
// half bucket (the middle mark); 8-bit codes, whose streams are about twice
// as long, a thread per quarter.
constexpr int kPartsFour = 2, kPartsEight = 4;

template <bool FOUR, int S>
__global__ void __launch_bounds__((decode_threads<FOUR, S>()), (decode_ctas_per_sm<FOUR, S>()))
k_elias_decode(DecodeArgs a) {
    constexpr int NT = decode_threads<FOUR, S>();
    static_assert(NT % 256 == 0 && NT <= 1024, "the length sort has 256 bins");
    extern __shared__ __align__(16) uint32_t s_words[];   // a.stage_cap words
    static_assert(S == 1 || S == 2 || S == 4, "a bucket splits at its quarter marks");
    constexpr int QS = 4 / S;               // quarters per task
    constexpr int KMAX = FOUR ? 8 : 4;
    constexpr int W = win_bits<FOUR>();
    // vectors of the staging held in registers through the set-up
    constexpr int RS = S == 1 ? 4 : 2;
    __shared__ __align__(16) uint64_t multi[1 << W];
    __shared__ uint32_t single[256];
    const uint32_t smax = static_cast<uint32_t>(a.s);
    const int stream = blockIdx.y;
    const uint32_t* offsets = a.offsets.p[stream];
    const int bpc = a.bpc;                  // <= NT / S
    // The CTA's words, offsets[b0] .. offsets[b0 + cnt) (at most stage_cap - 3
    // of them), are copied to shared memory, so that the walks below read from
    // there; their loads are issued first.  Every word of that range lies
    // inside the range of one of the CTA's buckets, whatever the offsets: the
    // copy reads nothing a bucket would not.
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * bpc;
    const int64_t cnt = a.nbuckets - b0 < bpc ? a.nbuckets - b0 : bpc;
    const uint32_t base = offsets[b0], wend = offsets[b0 + cnt];
    const uint32_t cap = a.stage_cap > 3u ? a.stage_cap - 3u : 0u;
    const uint32_t nst = wend > base ? (wend - base < cap ? wend - base : cap) : 0u;
    const uint32_t* gwords = a.words.p[stream];
    const StageSplit sp = stage_split(base, nst);
    uint4 sv[RS];
    uint32_t sedge;
    stage_issue<NT, RS>(gwords + base, sp, sv, sedge);
    uint32_t* staged_words = s_words + (base & 3u);
    {
        // A window holding a level above s gets count 0, which sends it to
        // the one-codeword path (where that level is flagged): the main loop
        // then tests only the count.  Entries are (packed << 32) | meta, meta
        // = (max level << 8) | (count << 4) | bits; the shared copy drops the
        // max level, so that the count is meta >> 4.  All of a thread's
        // loads are issued before its stores.
        constexpr int kTv = (1 << W) / 2;    // 16-byte pieces of the table
        constexpr int kTi = (kTv + NT - 1) / NT;
        const uint4* src = reinterpret_cast<const uint4*>(FOUR ? kMulti4.e : kMulti8.e);
        uint4* dst = reinterpret_cast<uint4*>(multi);
        uint4 tv[kTi];
#pragma unroll
        for (int j = 0; j < kTi; ++j) {
            const int i = static_cast<int>(threadIdx.x) + j * NT;
            if (i < kTv) tv[j] = __ldg(src + i);
        }
#pragma unroll
        for (int j = 0; j < kTi; ++j) {
            const int i = static_cast<int>(threadIdx.x) + j * NT;
            if (i < kTv) {
                uint4 v = tv[j];
                v.x = ((v.x >> 8) & 127u) > smax ? (v.x & 15u) : (v.x & 255u);
                v.z = ((v.z >> 8) & 127u) > smax ? (v.z & 15u) : (v.z & 255u);
                dst[i] = v;
            }
        }
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x) single[i] = window_entry<8>(static_cast<uint32_t>(i));
    const int64_t bb = static_cast<int64_t>(blockIdx.x) * bpc + threadIdx.x / S;
    uint32_t key = 255u;
    if (static_cast<int>(threadIdx.x) / S < bpc && bb < a.nbuckets) {
        uint32_t nw = offsets[bb + 1] - offsets[bb];
        if (S > 1) {
            const int k = threadIdx.x % S;
            const uint32_t sb = k ? a.marks[3 * bb + k * QS - 1] : 32u;
            const uint32_t eb = k < S - 1 ? a.marks[3 * bb + (k + 1) * QS - 1] : 32u * nw;
            nw = eb > sb ? (eb - sb + 31u) / 32u : 0u;
        }
        key = nw < 255u ? nw : 255u;
    }
    const int task = task_by_length<NT>(key);
    stage_store<NT, RS>(gwords + base, sp, sv, sedge, staged_words);
    __syncthreads();
    if (task / S >= bpc) return;                // a thread past the CTA's buckets
    const int64_t b = b0 + task / S;
    if (b >= a.nbuckets) return;
    const int kq = task % S;                    // the task's part of the bucket
    const int64_t blo = b * a.d;
    const int blen = static_cast<int>(a.n - blo < a.d ? a.n - blo : static_cast<int64_t>(a.d));
    const int q = a.d / S;
    const int c0 = kq * q;                      // first coordinate of the task
    if (c0 >= blen && kq > 0) return;           // a part past a short bucket's end
    const int64_t lo = blo + c0;
    const int len = min(blen - c0, q);
    const uint32_t w_lo = offsets[b], w_hi = offsets[b + 1];
    // a bucket wholly inside the staged words reads shared memory (through a
    // generic pointer), any other bucket global memory
    const bool staged = w_lo - base <= nst && w_hi - base <= nst;
    const uint32_t* src = staged ? staged_words + (w_lo - base) : gwords + w_lo;
    const int64_t avail = w_hi > w_lo ? static_cast<int64_t>(w_hi - w_lo) : 0;
    bool bad = avail == 0;
    auto word = [&](int64_t i) { return i < avail ? src[i] : 0u; };
    if (kq == 0) a.norms.p[stream][b] = __uint_as_float(word(0));
    // the task's first bit (after the norm, or its quarter mark)
    const uint32_t sb = kq ? a.marks[3 * b + kq * QS - 1] : 32u;
    const int64_t w0 = sb >> 5;
    uint32_t whi = word(w0), wlo = word(w0 + 1), pre = word(w0 + 2);
    int64_t next = w0 + 3;
    int have = 64;
    CodeWriter<FOUR> wr;
    wr.out = reinterpret_cast<uint32_t*>(a.codes.p[stream] + (FOUR ? lo / 2 : lo));
    auto shift_out = [&](int l) {
        whi = __funnelshift_l(wlo, whi, l);
        wlo <<= l;
        have -= l;
    };
    auto refill = [&]() {
        if (have <= 32) {
            whi |= __funnelshift_rc(pre, 0u, have);
            wlo |= pre << (32 - have);
            have += 32;
            pre = word(next);
            ++next;
        }
    };
    auto consume = [&](int l) {
        shift_out(l);
        refill();
    };
    // A codeword longer than 8 bits in a valid stream is omega(N) for N of
    // k = 5..8 binary digits: the groups "10" and binary(k - 1) = "1xx", then
    // N itself, the final 0 and the sign bit (k + 7 bits in all).  Anything
    // else at this point -- or a level above s -- is not the encoder's
    // output: it is flagged, and decoding goes on with a clamped level.
    auto long_code = [&](uint32_t& code, int& l) {
        const uint32_t top5 = whi >> 27;
        const uint32_t k = 5u + (top5 & 3u);
        const uint32_t N = (whi >> (27u - k)) & ((1u << k) - 1u);
        uint32_t level = N - 1u;
        const uint32_t sign = (whi >> (25u - k)) & 1u;
        const bool ok = (top5 >> 2) == 5u && ((whi >> (26u - k)) & 1u) == 0u && (N >> (k - 1u)) == 1u &&
                        level <= smax;
        if (!ok) {
            bad = true;
            level = level < smax ? level : smax;
        }
        code = FOUR ? (sign << 3) | (level & 7u) : (sign << 7) | level;
        l = static_cast<int>(k) + 7;
    };
    // One codeword through the 8-bit table, or the long-codeword formula.  A
    // level above s is flagged and written as s; its codeword's own length is
    // consumed, so that the codes after it still decode in step.
    auto one_code = [&](uint32_t& code, int& l) {
        const uint32_t t = single[whi >> 24];
        if (t) {
            l = static_cast<int>(t & 15u);
            uint32_t level = t >> 5;
            const uint32_t sign = level ? (t >> 4) & 1u : 0u;
            if (level > smax) {
                bad = true;
                level = smax;
            }
            code = FOUR ? (sign << 3) | level : (sign << 7) | level;
        } else {
            long_code(code, l);
        }
    };
    if (sb & 31u) consume(static_cast<int>(sb & 31u));
    int e = 0;
    auto table_step = [&]() {
        const uint64_t t = multi[whi >> (32 - W)];
        int k = static_cast<int>(static_cast<uint32_t>(t) >> 4);
        int l = static_cast<int>(t & 15u);
        uint32_t packed = static_cast<uint32_t>(t >> 32);
        if (k == 0) {
            // a codeword longer than the window, or a level above s
            one_code(packed, l);
            k = 1;
        }
        shift_out(l);
        wr.put(packed, k);
        e += k;
    };
    // After a refill the window holds more than 32 bits and a step takes at
    // most 15 (the longest codeword with its sign), so two steps share one
    // refill: the second still sees at least 18 valid bits.
    while (len - e >= 2 * KMAX) {
        table_step();
        table_step();
        refill();
    }
    while (len - e >= KMAX) {
        table_step();
        refill();
    }
    for (; e < len; ++e) {
        uint32_t code;
        int l;
        one_code(code, l);
        consume(l);
        wr.put(code, 1);
    }
    wr.finish();
    // bits consumed: the words fetched (norm included, `pre` not) minus those still in the window
    const int64_t used = 32 * (next - 1) - have;
    if (used > 32 * avail) bad = true;
    // a part must end where the next one starts; the bucket's last part (of
    // a short bucket: the last one holding coordinates) must end at the start
    // mark of every part after it, which the encoder sets to the bucket's end
    if (S > 1) {
        if (c0 + q < blen) {
            if (used != a.marks[3 * b + (kq + 1) * QS - 1]) bad = true;
        } else {
            for (int k = kq + 1; k < S; ++k)
                if (used != a.marks[3 * b + k * QS - 1]) bad = true;
        }
    }
    if (bad && a.status) *a.status = GC_ERR_CORRUPT;
}

constexpr int kMaxDevices = 64;

// Stream words a CTA of `kernel` stages: the shared memory left, after its
// static tables and the per-CTA reservation, when `ctas` CTAs share an SM.
// Computed once per device (cache[device] = words + 1), which also raises the
// kernel's dynamic shared-memory limit there.
template <typename Kernel>
int stage_cap_for(Kernel kernel, int ctas, std::atomic<uint32_t>* cache, uint32_t* cap) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GC_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevices) {
        const uint32_t c = cache[dev].load(std::memory_order_relaxed);
        if (c) {
            *cap = c - 1;
            return GC_OK;
        }
    }
    int per_sm = 0, reserved = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, kernel) != cudaSuccess)
        return GC_ERR_CUDA;
    int64_t bytes = static_cast<int64_t>(per_sm) / ctas - reserved - static_cast<int64_t>(fa.sharedSizeBytes);
    bytes = bytes > 0 ? bytes & ~static_cast<int64_t>(15) : 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
        cudaSuccess)
        return GC_ERR_CUDA;
    *cap = static_cast<uint32_t>(bytes / sizeof(uint32_t));
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(*cap + 1, std::memory_order_relaxed);
    return GC_OK;
}

template <bool FOUR, int S>
int decode_stage_words(uint32_t* cap) {
    static std::atomic<uint32_t> cached[kMaxDevices];
    return stage_cap_for(k_elias_decode<FOUR, S>, decode_ctas_per_sm<FOUR, S>(), cached, cap);
}

// Buckets per CTA (even_buckets_per_cta) for the current device's SMs, with
// `ctas` CTAs of at most maxb buckets resident per SM.  At 61.1 M coordinates
// (119,338 buckets): 197 buckets in each of 606 CTAs of 256 threads (4-bit
// codes, four per SM) where full CTAs left ten SMs 1024 buckets against 768
// elsewhere, and 786 in each of 152 CTAs of 1024 (8-bit codes) where full
// CTAs left 35 SMs idle.
int balanced_bpc(int64_t nb, int W, int ctas, int maxb, int* bpc) {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1)
        return GC_ERR_CUDA;
    *bpc = static_cast<int>(even_buckets_per_cta(nb, W, static_cast<int64_t>(nsm) * ctas, maxb));
    return GC_OK;
}

// ================================================================ sparse regimes
//
// QSGD Knowl 2, items 1 (s >= 2) and 1' (s = 1): only the non-zero
// coordinates are sent.  Per bucket: the 32 norm bits, then for each
// coordinate i (0-based within the bucket) whose level is not 0, in order,
// Elias-omega(i - p) (p the previous such i, or -1), one sign bit and, when
// s >= 2, Elias-omega(level); then Elias-omega(len - p) closes the bucket.
// Same stream conventions as the dense code above (most significant bit
// first, buckets on word boundaries, an offsets table).
//
// Encode = one launch, as the dense code (chunks by ticket, a chunk-level
// look-back): one warp per bucket, lane l owning coordinates
// [l d/32, (l+1) d/32); a lane's distances need the last non-zero coordinate
// before its range, which a warp max-scan supplies.  Decode: one thread per
// bucket, after its CTA has zeroed the code bytes of its buckets.


// Elias-omega codewords of 1..255 as (pattern << 5) | length (at most 14
// bits), built per CTA in shared memory; longer values take omega().
constexpr int kOmegaLut = 256;

__device__ __forceinline__ void build_omega_lut(uint32_t* lut) {
    for (int i = threadIdx.x; i < kOmegaLut; i += blockDim.x) {
        uint32_t pat = 0;
        const int len = i ? omega(static_cast<uint32_t>(i), &pat) : 0;
        lut[i] = (pat << 5) | static_cast<uint32_t>(len);
    }
}


__device__ __forceinline__ int omega_lut(const uint32_t* lut, uint32_t N, uint32_t* pat) {
    if (N < kOmegaLut) {
        const uint32_t e = lut[N];
        *pat = e >> 5;
        return static_cast<int>(e & 31u);
    }
    return omega(N, pat);
}

// Words of a sparse-coded bucket of len coordinates, whatever its codes: 32
// norm bits and at most 18 bits per coordinate (the distances sum to len and
// |omega(g)| <= g + 2; one sign bit; omega(level) <= 14 bits) plus 2.
inline int64_t sparse_bucket_max_words(int64_t len) { return 1 + div_up(18 * len + 2, 32); }

template <bool FOUR>
__device__ __forceinline__ void code_at(const uint8_t* codes, int64_t i, uint32_t& sign, uint32_t& level) {
    if (FOUR) {
        const uint32_t byte = __ldg(codes + (i >> 1));
        const uint32_t c = (i & 1) ? (byte & 15u) : (byte >> 4);
        sign = c >> 3;
        level = c & 7u;
    } else {
        const uint32_t c = __ldg(codes + i);
        sign = c >> 7;
        level = c & 127u;
    }
}

// Walks the codes of coordinates [c0, c1) of the bucket starting at
// coordinate lo.  A whole bucket's range is read a word (or, for 2-byte
// ranges, a half-word) at a time: word(k, w, nz) gets the word's first
// coordinate k (relative to c0), the word with element e in field e (low
// field first) and the mask of its non-zero fields (bit 0 of each 4-bit
// field, bit 7 of each byte); the ragged last bucket is read byte by byte,
// so that nothing past the codes is touched, and code(c) is called for each
// of its non-zero coordinates.
template <bool FOUR, typename Fw, typename Fc>
__device__ __forceinline__ void for_nonzero_words(const uint8_t* codes, int64_t lo, int c0, int c1, bool whole,
                                                  Fw word, Fc code) {
    if (!whole) {
        for (int c = c0; c < c1; ++c) {
            uint32_t sg, lv;
            code_at<FOUR>(codes, lo + c, sg, lv);
            if (lv) code(c);
        }
        return;
    }
    constexpr int kPerWord = FOUR ? 8 : 4;
    const int ncodes = c1 - c0;
    const uint8_t* base = codes + (FOUR ? (lo + c0) / 2 : lo + c0);
    for (int k = 0; k < ncodes; k += kPerWord) {
        uint32_t w;
        if (FOUR && ncodes < 8) w = __ldg(reinterpret_cast<const uint16_t*>(base));   // 4 codes, 2 bytes
        else w = __ldg(reinterpret_cast<const uint32_t*>(base) + k / kPerWord);
        uint32_t nz;
        if (FOUR) {
            // element e of the word in nibble e (low nibble first): swap the
            // nibbles of each byte (the first code of a byte is its high nibble)
            w = ((w >> 4) & 0x0F0F0F0Fu) | ((w & 0x0F0F0F0Fu) << 4);
            nz = (w | (w >> 1) | (w >> 2)) & 0x11111111u;
        } else {
            nz = ((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) & 0x80808080u;
        }
        word(k, w, nz);
    }
}

// Calls f(c, sign, level) for each coordinate c in [c0, c1) of the bucket
// starting at coordinate lo whose level is not 0, in order.
template <bool FOUR, typename F>
__device__ __forceinline__ void for_nonzero(const uint8_t* codes, int64_t lo, int c0, int c1, bool whole, F f) {
    for_nonzero_words<FOUR>(
        codes, lo, c0, c1, whole,
        [&](int k, uint32_t w, uint32_t nz) {
            while (nz) {
                const int bit = __ffs(nz) - 1;
                nz &= nz - 1;
                const int e = FOUR ? (bit >> 2) : (bit >> 3);
                const uint32_t cd = FOUR ? (w >> (4 * e)) & 15u : (w >> (8 * e)) & 255u;
                f(c0 + k + e, FOUR ? cd >> 3 : cd >> 7, FOUR ? cd & 7u : cd & 127u);
            }
        },
        [&](int c) {
            uint32_t sg, lv;
            code_at<FOUR>(codes, lo + c, sg, lv);
            f(c, sg, lv);
        });
}

// Non-zero codes among coordinates [c0, c1) of the bucket at lo: one
// population count per code word of a whole bucket.
template <bool FOUR>
__device__ __forceinline__ int count_nonzero(const uint8_t* codes, int64_t lo, int c0, int c1, bool whole) {
    int cnt = 0;
    for_nonzero_words<FOUR>(codes, lo, c0, c1, whole, [&](int, uint32_t, uint32_t nz) { cnt += __popc(nz); },
                            [&](int) { ++cnt; });
    return cnt;
}

struct SparseArgs {
    const uint8_t* codes;
    const float* norms;
    int64_t n;
    int d;
    int64_t nbuckets;
    bool levels;          // s >= 2
    uint32_t* words;
    uint32_t* offsets;
    int stage_words;      // staging words per bucket
    int chunk;            // buckets per CTA (<= kChunk), all staged at once
    EncodeWs ws;
    uint64_t wait_ns;     // bound on each look-back wait
};

// Encode, one launch: each CTA takes a chunk of buckets by ticket and the
// chunk goes out after a look-back over the chunks before it, as in the dense
// encoder.  A warp codes one bucket at a time, spreading its non-zero
// coordinates over the lanes: each lane counts those in its range of d/32
// coordinates (a population count per code word), a warp scan ranks them,
// and each lane writes its (coordinate, code) entries to the warp's list in
// shared memory in order; then rounds of 32 entries, one per lane, take
// their distance from the entry before, their codeword bits from the table,
// their bit position from a warp scan of the lengths, and are OR-ed into the
// bucket's staging words.
template <bool FOUR>
__global__ void __launch_bounds__(kThreads) k_elias_sparse_encode(SparseArgs a) {
    extern __shared__ uint32_t smem[];
    __shared__ uint32_t s_chunk, s_end;
    __shared__ uint32_t s_nw[kChunk];             // words of each bucket, then its first word
    uint32_t* lut = smem;                         // [kOmegaLut]
    uint32_t* stages = smem + kOmegaLut;          // [chunk][stage_words]
    uint32_t* lists = stages + a.chunk * a.stage_words;   // [kWarpsPerBlock][d]: (coordinate << 16) | code
    build_omega_lut(lut);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < a.chunk * a.stage_words; i += kThreads) stages[i] = 0u;
    if (threadIdx.x == 0) s_chunk = atomicAdd(a.ws.ticket, 1u);
    __syncthreads();
    const int64_t chunk = s_chunk;
    const int64_t b0 = chunk * a.chunk;
    const int nbc = static_cast<int>(a.nbuckets - b0 < a.chunk ? a.nbuckets - b0 : a.chunk);
    uint32_t* list = lists + warp * a.d;
    const int cpl = a.d / 32;
    for (int lb = warp; lb < nbc; lb += kWarpsPerBlock) {
        uint32_t* stage = stages + lb * a.stage_words;
        const int64_t b = b0 + lb;
        const int64_t lo = b * a.d;
        const int len = static_cast<int>(a.n - lo < a.d ? a.n - lo : static_cast<int64_t>(a.d));
        const bool whole = len == a.d;
        const int c0 = min(len, lane * cpl), c1 = min(len, c0 + cpl);
        // rank the non-zero coordinates, then list them in order
        const int cnt = count_nonzero<FOUR>(a.codes, lo, c0, c1, whole);
        const int incl = warp_incl_sum(cnt, lane);
        const int K = __shfl_sync(0xffffffffu, incl, 31);
        int r = incl - cnt;
        for_nonzero<FOUR>(a.codes, lo, c0, c1, whole, [&](int c, uint32_t sg, uint32_t lv) {
            list[r++] = (static_cast<uint32_t>(c) << 16) | (sg << 8) | lv;
        });
        __syncwarp();
        if (lane == 0) stage[0] = __float_as_uint(__ldg(a.norms + b));
        uint32_t pos = 32;
        for (int r0 = 0; r0 < K; r0 += 32) {
            const int k = r0 + lane;
            uint64_t piece = 0;
            int plen = 0;
            if (k < K) {
                const uint32_t ent = list[k];
                const int c = static_cast<int>(ent >> 16);
                const int prev = k ? static_cast<int>(list[k - 1] >> 16) : -1;
                uint32_t gpat, lpat = 0;
                const int glen = omega_lut(lut, static_cast<uint32_t>(c - prev), &gpat);
                const int llen = a.levels ? omega_lut(lut, ent & 255u, &lpat) : 0;
                piece = (((static_cast<uint64_t>(gpat) << 1) | ((ent >> 8) & 1u)) << llen) | lpat;
                plen = glen + 1 + llen;                      // <= 34
            }
            const int pin = warp_incl_sum(plen, lane);
            emit(stage, pos + static_cast<uint32_t>(pin - plen), piece, plen);
            pos += static_cast<uint32_t>(__shfl_sync(0xffffffffu, pin, 31));
        }
        if (lane == 0) {
            const int last = K ? static_cast<int>(list[K - 1] >> 16) : -1;
            uint32_t tpat;
            const int tlen = omega_lut(lut, static_cast<uint32_t>(len - last), &tpat);
            emit(stage, pos, tpat, tlen);
            s_nw[lb] = (pos + static_cast<uint32_t>(tlen) + 31u) >> 5;
        }
        __syncwarp();
    }
    __syncthreads();
    if (warp == 0)
        chunk_offsets(a.ws, chunk, b0, nbc, a.nbuckets, a.offsets, s_nw, &s_end, a.wait_ns, -1, lane);
    __syncthreads();
    write_chunk(stages, a.stage_words, s_nw, s_end, nbc, a.words, warp, lane);
}

// Decode: a thread per bucket, in the dense decoder's way.  The CTA zeroes
// the code bytes of its buckets (coalesced), hands its buckets to its threads
// in order of stream length, and copies its stream words to shared memory;
// each thread then walks its bucket with a 64-bit window (the next word
// waiting in a register) and assembles the 32-bit code words that hold
// non-zero coordinates, each stored once.  A stream this encoder did not
// write -- a distance past the bucket's end, a read past its words, a level
// above s or an impossible codeword -- sets the status to GC_ERR_CORRUPT.
// Elias-omega codewords that end inside a 12-bit window (values up to 63),
// looked up as (value << 4) | length, 0 when the codeword is longer.
constexpr int kOmegaWin = 12;

__device__ __forceinline__ uint32_t omega_window_entry(uint32_t x) {
    int pos = 0;
    uint32_t N = 1;
    for (;;) {
        if (pos >= kOmegaWin) return 0u;
        const uint32_t bit = (x >> (kOmegaWin - 1 - pos)) & 1u;
        ++pos;
        if (!bit) break;
        if (pos + static_cast<int>(N) > kOmegaWin) return 0u;
        const uint32_t v = (x >> (kOmegaWin - pos - static_cast<int>(N))) & ((1u << N) - 1u);
        pos += static_cast<int>(N);
        N = (1u << N) | v;
    }
    return (N << 4) | static_cast<uint32_t>(pos);
}

constexpr int kSparseDecodeCtasPerSm = 4;

template <bool FOUR>
__global__ void __launch_bounds__(kThreads, kSparseDecodeCtasPerSm) k_elias_decode_sparse(DecodeArgs a) {
    extern __shared__ __align__(16) uint32_t s_words[];   // a.stage_cap words
    __shared__ uint16_t otab[1 << kOmegaWin];
    const int stream = blockIdx.y;
    const int bpc = a.bpc;                  // <= kThreads
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * bpc;
    const int64_t cnt = a.nbuckets - b0 < bpc ? a.nbuckets - b0 : bpc;
    // the CTA's words (at most stage_cap - 3) to shared memory: loads first
    const uint32_t* offsets = a.offsets.p[stream];
    const uint32_t base = offsets[b0], wend = offsets[b0 + cnt];
    const uint32_t cap = a.stage_cap > 3u ? a.stage_cap - 3u : 0u;
    const uint32_t nst = wend > base ? (wend - base < cap ? wend - base : cap) : 0u;
    const uint32_t* gwords = a.words.p[stream];
    const StageSplit sp = stage_split(base, nst);
    uint4 sv[2];
    uint32_t sedge;
    stage_issue<kThreads, 2>(gwords + base, sp, sv, sedge);
    uint32_t* staged_words = s_words + (base & 3u);
    for (int i = threadIdx.x; i < (1 << kOmegaWin); i += kThreads)
        otab[i] = static_cast<uint16_t>(omega_window_entry(static_cast<uint32_t>(i)));
    uint8_t* codes = a.codes.p[stream];
    const int64_t total = FOUR ? (a.n + 1) / 2 : a.n;      // code bytes
    {
        const int64_t bpb = FOUR ? a.d / 2 : a.d;           // bytes per whole bucket (>= 64)
        const int64_t start = b0 * bpb;
        int64_t end = (b0 + cnt) * bpb;
        if (end > total) end = total;
        const int64_t nvec = (end - start) / 16;
        uint4* v = reinterpret_cast<uint4*>(codes + start);
        for (int64_t i = threadIdx.x; i < nvec; i += kThreads) v[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int64_t i = start + nvec * 16 + threadIdx.x; i < end; i += kThreads) codes[i] = 0;
    }
    const int64_t bb = b0 + threadIdx.x;
    uint32_t key = 255u;
    if (static_cast<int>(threadIdx.x) < bpc && bb < a.nbuckets) {
        const uint32_t nw = offsets[bb + 1] - offsets[bb];
        key = nw < 255u ? nw : 255u;
    }
    // (its barriers also order the zero fill before the code words below)
    const int task = task_by_length<kThreads>(key);
    stage_store<kThreads, 2>(gwords + base, sp, sv, sedge, staged_words);
    __syncthreads();
    if (task >= bpc) return;                    // a thread past the CTA's buckets
    const int64_t b = b0 + task;
    if (b >= a.nbuckets) return;
    const uint32_t w_lo = offsets[b], w_hi = offsets[b + 1];
    const bool staged = w_lo - base <= nst && w_hi - base <= nst;
    const uint32_t* src = staged ? staged_words + (w_lo - base) : gwords + w_lo;
    const int64_t avail = w_hi > w_lo ? static_cast<int64_t>(w_hi - w_lo) : 0;
    auto word = [&](int64_t i) { return i < avail ? src[i] : 0u; };
    const int64_t lo = b * a.d;
    const int len = static_cast<int>(a.n - lo < a.d ? a.n - lo : static_cast<int64_t>(a.d));
    bool bad = avail == 0;
    a.norms.p[stream][b] = __uint_as_float(word(0));
    // window: `have` valid bits from the top of win, the next word in `pre`
    uint64_t win = (static_cast<uint64_t>(word(1)) << 32) | word(2);
    int have = 64;
    uint32_t pre = word(3);
    int64_t next = 4;
    auto refill = [&]() {
        if (have <= 32) {
            win |= static_cast<uint64_t>(pre) << (32 - have);
            have += 32;
            pre = word(next);
            ++next;
        }
    };
    auto consume = [&](int l) {
        win <<= l;
        have -= l;
    };
    auto take = [&](int k) -> uint32_t {       // k in 1..31
        refill();
        const uint32_t v = static_cast<uint32_t>(win >> (64 - k));
        consume(k);
        return v;
    };
    // a codeword longer than the table's window, bit by bit
    auto omega_slow = [&]() -> uint32_t {
        uint32_t N = 1;
        while (take(1)) {
            if (N > 16) {                      // no distance or level of a valid stream is this long
                bad = true;
                return 0u;
            }
            N = (1u << N) | take(static_cast<int>(N));
        }
        return N;
    };
    // bits after the norm word consumed so far; beyond its last word the
    // stream is corrupt (the window may hold zero words read past it)
    const int64_t limit = avail > 0 ? 32 * (avail - 1) : 0;
    auto used = [&]() { return 32 * (next - 2) - have; };
    // the code word (8 codes of 4 bits or 4 of 8) being assembled
    uint32_t* out = reinterpret_cast<uint32_t*>(codes + (FOUR ? lo / 2 : lo));
    const int64_t out_bytes = total - (FOUR ? lo / 2 : lo);
    uint32_t cw = 0xFFFFFFFFu, cv = 0u;
    auto flush = [&]() {
        if (cw == 0xFFFFFFFFu) return;
        if (4 * static_cast<int64_t>(cw) + 4 <= out_bytes) {
            out[cw] = cv;
        } else {                               // the last word of a ragged buffer
            uint8_t* ob = reinterpret_cast<uint8_t*>(out + cw);
            for (int j = 0; j < 4; ++j)
                if (4 * static_cast<int64_t>(cw) + j < out_bytes) ob[j] = static_cast<uint8_t>(cv >> (8 * j));
        }
    };
    const uint32_t smax = static_cast<uint32_t>(a.s);
    int64_t p = -1;
    for (int guard = 0; guard <= len && !bad; ++guard) {
        // After a refill the window holds more than 32 bits: a distance from
        // the table (at most 12), the sign and a level from the table (at
        // most 12) need no refill in between.
        refill();
        uint32_t g;
        const uint32_t e1 = otab[static_cast<uint32_t>(win >> (64 - kOmegaWin))];
        if (e1) {
            g = e1 >> 4;
            consume(static_cast<int>(e1 & 15u));
        } else {
            g = omega_slow();
            if (bad) break;
            refill();
        }
        p += g;
        if (p >= len) {
            bad |= p > len;
            break;
        }
        const uint32_t sign = static_cast<uint32_t>(win >> 63);
        consume(1);
        uint32_t level = 1u;
        if (a.s >= 2) {
            const uint32_t e2 = otab[static_cast<uint32_t>(win >> (64 - kOmegaWin))];
            if (e2) {
                level = e2 >> 4;
                consume(static_cast<int>(e2 & 15u));
            } else {
                level = omega_slow();
                if (bad) break;
            }
        }
        if (level > smax) {             // written as s; the walk stops after it
            bad = true;
            level = smax;
        }
        if (used() > limit) {           // read past the bucket's words
            bad = true;
            break;
        }
        const uint32_t pp = static_cast<uint32_t>(p);
        const uint32_t wi = FOUR ? pp >> 3 : pp >> 2;
        if (wi != cw) {
            flush();
            cw = wi;
            cv = 0u;
        }
        // element e of a word: byte e / 2, high nibble for even e (4-bit
        // codes); byte e (8-bit codes)
        if (FOUR)
            cv |= ((sign << 3) | level) << (8 * ((pp & 7u) >> 1) + 4 * (1u - (pp & 1u)));
        else
            cv |= ((sign << 7) | level) << (8 * (pp & 3u));
    }
    flush();
    bad |= used() > limit;
    if (bad && a.status) *a.status = GC_ERR_CORRUPT;
}

}  // namespace
// Raises the sparse encoder's dynamic shared-memory limit to `bytes` when
// it is above the default 48 KB (large buckets).
template <bool FOUR>
int sparse_encode_smem(size_t bytes) {
    if (bytes <= 48 * 1024) return GC_OK;
    return cudaFuncSetAttribute(k_elias_sparse_encode<FOUR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes)) == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

template <bool FOUR>
int sparse_stage_words(uint32_t* cap) {
    static std::atomic<uint32_t> cached[kMaxDevices];
    return stage_cap_for(k_elias_decode_sparse<FOUR>, kSparseDecodeCtasPerSm, cached, cap);
}

}  // namespace gc

using namespace gc;

extern "C" {

uint64_t qsgd_elias_max_words(int64_t n, int bucket, int s_levels) {
    if (n < 0 || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127) return 0;
    const bool four = s_levels <= 7;
    const int64_t full = n / bucket, rest = n % bucket;
    return static_cast<uint64_t>(full * bucket_max_words(bucket, four) +
                                 (rest ? bucket_max_words(rest, four) : 0));
}

size_t qsgd_elias_workspace_bytes(int64_t n, int bucket) {
    if (n < 0 || !valid_bucket(bucket)) return 0;
    return encode_ws_bytes(div_up(n, bucket));
}

}  // extern "C"

namespace {

int encode_dense(const uint8_t* codes, const float* norms, int64_t n, int bucket, int s_levels, uint32_t* words,
                 uint64_t capacity_words, uint32_t* offsets, uint16_t* marks, void* workspace, size_t ws_bytes,
                 int64_t withhold, uint64_t wait_ns, gc_stream_t stream) {
    if (n < 0 || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127) return GC_ERR_INVALID;
    if (!offsets || (n > 0 && (!codes || !norms || !words || !workspace))) return GC_ERR_INVALID;
    const uint64_t need = qsgd_elias_max_words(n, bucket, s_levels);
    if (need > 0xFFFFFFFFull) return GC_ERR_INVALID;    // offsets are 32-bit word indices
    if (capacity_words < need) return GC_ERR_CAPACITY;
    if (ws_bytes < qsgd_elias_workspace_bytes(n, bucket)) return GC_ERR_INVALID;
    if ((codes && !aligned16(codes)) || (norms && !aligned16(norms)) || (words && !aligned16(words)) ||
        !aligned16(offsets) || (workspace && !aligned16(workspace)))
        return GC_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (workspace && cudaMemsetAsync(workspace, 0, kTicketBytes, s) != cudaSuccess) return GC_ERR_CUDA;
        return cudaMemsetAsync(offsets, 0, sizeof(uint32_t), s) == cudaSuccess ? GC_OK : GC_ERR_CUDA;
    }
    const bool four = s_levels <= 7;
    const int64_t nb = div_up(n, bucket);
    const int P = (four ? bucket / 2 : bucket) / 16;
    const int stride = static_cast<int>(bucket_max_words(bucket, four)) + 2;
    // buckets per CTA: 64, halved while their staging would pass 36 KB (so
    // that five CTAs share an SM)
    int chunk = kChunk;
    while (chunk > 8 && chunk * stride > kEncodeStageWords) chunk /= 2;
    const int64_t nchunks = div_up(nb, chunk);
    // status, ticket and the look-back states start at zero
    if (cudaMemsetAsync(workspace, 0, kTicketBytes + static_cast<size_t>(nchunks) * 8, s) != cudaSuccess)
        return GC_ERR_CUDA;
    EncodeArgs ea{codes, norms, n, bucket, nb, words, offsets, stride, P < 32 ? 32 / P : 1, marks,
                  encode_ws(workspace), wait_ns, withhold < 0 ? -1 : withhold / chunk, chunk};
    const size_t smem = sizeof(uint32_t) * (256 + static_cast<size_t>(chunk) * stride);
    const unsigned grid = static_cast<unsigned>(nchunks);
    if (four)
        k_elias_encode<true><<<grid, kThreads, smem, s>>>(ea);
    else
        k_elias_encode<false><<<grid, kThreads, smem, s>>>(ea);
    return launch_status();
}

constexpr uint64_t kEncodeWaitNs = 1000000000ull;   // 1 s: only a fault elsewhere makes a wait that long

}  // namespace

extern "C" {

int qsgd_elias_encode(const uint8_t* codes, const float* norms, int64_t n, int bucket, int s_levels,
                      uint32_t* words, uint64_t capacity_words, uint32_t* offsets, void* workspace,
                      size_t ws_bytes, gc_stream_t stream) {
    return encode_dense(codes, norms, n, bucket, s_levels, words, capacity_words, offsets, nullptr, workspace,
                        ws_bytes, -1, kEncodeWaitNs, stream);
}

int qsgd_elias_encode_marked(const uint8_t* codes, const float* norms, int64_t n, int bucket, int s_levels,
                             uint32_t* words, uint64_t capacity_words, uint32_t* offsets, uint16_t* marks,
                             void* workspace, size_t ws_bytes, gc_stream_t stream) {
    if (n > 0 && !marks) return GC_ERR_INVALID;
    if (marks && !aligned16(marks)) return GC_ERR_ALIGN;
    return encode_dense(codes, norms, n, bucket, s_levels, words, capacity_words, offsets, marks, workspace,
                        ws_bytes, -1, kEncodeWaitNs, stream);
}

int gc_testing_qsgd_elias_encode_withhold(const uint8_t* codes, const float* norms, int64_t n, int bucket,
                                          int s_levels, uint32_t* words, uint64_t capacity_words, uint32_t* offsets,
                                          void* workspace, size_t ws_bytes, int64_t withhold_bucket, uint64_t wait_ns,
                                          gc_stream_t stream) {
    if (wait_ns < 1 || wait_ns > kEncodeWaitNs || withhold_bucket < 0) return GC_ERR_INVALID;
    return encode_dense(codes, norms, n, bucket, s_levels, words, capacity_words, offsets, nullptr, workspace,
                        ws_bytes, withhold_bucket, wait_ns, stream);
}

int qsgd_elias_decode_batched(const uint32_t* const* words, const uint32_t* const* offsets, int W,
                              int64_t n, int bucket, int s_levels, uint8_t* const* codes,
                              float* const* norms, int* d_status, gc_stream_t stream) {
    if (n < 0 || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127 || W < 1 || W > GC_MAX_WORKERS)
        return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!words || !offsets || !codes || !norms) return GC_ERR_INVALID;
    if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return GC_ERR_ALIGN;
    DecodeArgs a;
    for (int w = 0; w < W; ++w) {
        if (!words[w] || !offsets[w] || !codes[w] || !norms[w]) return GC_ERR_INVALID;
        if (!aligned16(words[w]) || !aligned16(offsets[w]) || !aligned16(codes[w]) || !aligned16(norms[w]))
            return GC_ERR_ALIGN;
        a.words.p[w] = words[w];
        a.offsets.p[w] = offsets[w];
        a.codes.p[w] = codes[w];
        a.norms.p[w] = norms[w];
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nb = div_up(n, bucket);
    a.n = n;
    a.d = bucket;
    a.nbuckets = nb;
    a.s = s_levels;
    a.status = d_status;
    a.marks = nullptr;
    const bool four = s_levels <= 7;
    const int nt = four ? decode_threads<true, 1>() : decode_threads<false, 1>();
    int rc = balanced_bpc(nb, W, four ? decode_ctas_per_sm<true, 1>() : decode_ctas_per_sm<false, 1>(), nt, &a.bpc);
    if (rc != GC_OK) return rc;
    const dim3 grid(static_cast<unsigned>(div_up(nb, a.bpc)), static_cast<unsigned>(W));
    rc = four ? decode_stage_words<true, 1>(&a.stage_cap) : decode_stage_words<false, 1>(&a.stage_cap);
    if (rc != GC_OK) return rc;
    const size_t dyn = static_cast<size_t>(a.stage_cap) * sizeof(uint32_t);
    if (four)
        k_elias_decode<true, 1><<<grid, nt, dyn, s>>>(a);
    else
        k_elias_decode<false, 1><<<grid, nt, dyn, s>>>(a);
    return launch_status();
}

int qsgd_elias_decode(const uint32_t* words, const uint32_t* offsets, int64_t n, int bucket, int s_levels,
                      uint8_t* codes, float* norms, int* d_status, gc_stream_t stream) {
    return qsgd_elias_decode_batched(&words, &offsets, 1, n, bucket, s_levels, &codes, &norms, d_status, stream);
}

int qsgd_elias_decode_quarters(const uint32_t* words, const uint32_t* offsets, const uint16_t* marks, int64_t n,
                               int bucket, int s_levels, uint8_t* codes, float* norms, int* d_status,
                               gc_stream_t stream) {
    if (n < 0 || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!words || !offsets || !marks || !codes || !norms) return GC_ERR_INVALID;
    if (!aligned16(words) || !aligned16(offsets) || !aligned16(marks) || !aligned16(codes) || !aligned16(norms))
        return GC_ERR_ALIGN;
    if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return GC_ERR_ALIGN;
    DecodeArgs a;
    a.words.p[0] = words;
    a.offsets.p[0] = offsets;
    a.codes.p[0] = codes;
    a.norms.p[0] = norms;
    a.n = n;
    a.d = bucket;
    a.nbuckets = div_up(n, bucket);
    a.s = s_levels;
    a.status = d_status;
    a.marks = marks;
    const bool four = s_levels <= 7;
    const int S = four ? kPartsFour : kPartsEight;
    const int nt = four ? decode_threads<true, kPartsFour>() : decode_threads<false, kPartsEight>();
    // Full CTAs: with a part of a bucket per thread the grid is two or more
    // waves already, and the extra CTAs of an even spread cost more in
    // per-CTA set-up (table copy, length sort) than the spread saves.
    a.bpc = nt / S;
    const dim3 grid(static_cast<unsigned>(div_up(a.nbuckets, a.bpc)), 1u);
    const int rc = four ? decode_stage_words<true, kPartsFour>(&a.stage_cap)
                        : decode_stage_words<false, kPartsEight>(&a.stage_cap);
    if (rc != GC_OK) return rc;
    const size_t dyn = static_cast<size_t>(a.stage_cap) * sizeof(uint32_t);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (four)
        k_elias_decode<true, kPartsFour><<<grid, nt, dyn, s>>>(a);
    else
        k_elias_decode<false, kPartsEight><<<grid, nt, dyn, s>>>(a);
    return launch_status();
}

uint64_t qsgd_elias_sparse_max_words(int64_t n, int bucket) {
    if (n < 0 || !valid_bucket(bucket)) return 0;
    const int64_t full = n / bucket, rest = n % bucket;
    return static_cast<uint64_t>(full * sparse_bucket_max_words(bucket) +
                                 (rest ? sparse_bucket_max_words(rest) : 0));
}

int qsgd_elias_encode_sparse(const uint8_t* codes, const float* norms, int64_t n, int bucket, int s_levels,
                             uint32_t* words, uint64_t capacity_words, uint32_t* offsets, void* workspace,
                             size_t ws_bytes, gc_stream_t stream) {
    if (n < 0 || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127) return GC_ERR_INVALID;
    if (!offsets || (n > 0 && (!codes || !norms || !words || !workspace))) return GC_ERR_INVALID;
    const uint64_t need = qsgd_elias_sparse_max_words(n, bucket);
    if (need > 0xFFFFFFFFull) return GC_ERR_INVALID;
    if (capacity_words < need) return GC_ERR_CAPACITY;
    if (ws_bytes < qsgd_elias_workspace_bytes(n, bucket)) return GC_ERR_INVALID;
    if ((codes && !aligned16(codes)) || (norms && !aligned16(norms)) || (words && !aligned16(words)) ||
        !aligned16(offsets) || (workspace && !aligned16(workspace)))
        return GC_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (workspace && cudaMemsetAsync(workspace, 0, kTicketBytes, s) != cudaSuccess) return GC_ERR_CUDA;
        return cudaMemsetAsync(offsets, 0, sizeof(uint32_t), s) == cudaSuccess ? GC_OK : GC_ERR_CUDA;
    }
    const bool four = s_levels <= 7;
    const int64_t nb = div_up(n, bucket);
    const int stride = static_cast<int>(sparse_bucket_max_words(bucket)) + 2;
    // buckets per CTA: as many as 37.5 KB of staging holds, at most 64
    const int chunk = static_cast<int>(kSparseStageWords / stride < kChunk ? kSparseStageWords / stride : kChunk);
    const int64_t nchunks = div_up(nb, chunk);
    if (cudaMemsetAsync(workspace, 0, kTicketBytes + static_cast<size_t>(nchunks) * 8, s) != cudaSuccess)
        return GC_ERR_CUDA;
    SparseArgs a{codes, norms, n, bucket, nb, s_levels >= 2, words, offsets, stride, chunk, encode_ws(workspace),
                 kEncodeWaitNs};
    // the table, the chunk's staging, and each warp's list of non-zero coordinates
    const size_t smem = sizeof(uint32_t) * (kOmegaLut + static_cast<size_t>(chunk) * stride +
                                            static_cast<size_t>(kWarpsPerBlock) * bucket);
    const int rc = four ? sparse_encode_smem<true>(smem) : sparse_encode_smem<false>(smem);
    if (rc != GC_OK) return rc;
    const unsigned grid = static_cast<unsigned>(nchunks);
    if (four)
        k_elias_sparse_encode<true><<<grid, kThreads, smem, s>>>(a);
    else
        k_elias_sparse_encode<false><<<grid, kThreads, smem, s>>>(a);
    return launch_status();
}

int qsgd_elias_decode_sparse(const uint32_t* words, const uint32_t* offsets, int64_t n, int bucket, int s_levels,
                             uint8_t* codes, float* norms, int* d_status, gc_stream_t stream) {
    if (n < 0 || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!words || !offsets || !codes || !norms) return GC_ERR_INVALID;
    if (!aligned16(words) || !aligned16(offsets) || !aligned16(codes) || !aligned16(norms)) return GC_ERR_ALIGN;
    if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return GC_ERR_ALIGN;
    DecodeArgs a;
    a.words.p[0] = words;
    a.offsets.p[0] = offsets;
    a.codes.p[0] = codes;
    a.norms.p[0] = norms;
    a.n = n;
    a.d = bucket;
    a.nbuckets = div_up(n, bucket);
    a.s = s_levels;
    a.status = d_status;
    a.marks = nullptr;
    int rc = balanced_bpc(a.nbuckets, 1, kSparseDecodeCtasPerSm, kThreads, &a.bpc);
    if (rc != GC_OK) return rc;
    const dim3 grid(static_cast<unsigned>(div_up(a.nbuckets, a.bpc)), 1u);
    const bool four = s_levels <= 7;
    rc = four ? sparse_stage_words<true>(&a.stage_cap) : sparse_stage_words<false>(&a.stage_cap);
    if (rc != GC_OK) return rc;
    const size_t dyn = static_cast<size_t>(a.stage_cap) * sizeof(uint32_t);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (four)
        k_elias_decode_sparse<true><<<grid, kThreads, dyn, s>>>(a);
    else
        k_elias_decode_sparse<false><<<grid, kThreads, dyn, s>>>(a);
    return launch_status();
}

}  // extern "C"
