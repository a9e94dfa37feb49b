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
// Encode = two launches.  k_elias_count: one warp per bucket sums the coded
// lengths (a 256-entry table turns one code byte into its codeword bits and
// length), writes each bucket's word count, and the last CTA to finish turns
// the per-CTA totals into an exclusive prefix (a ticket counter, no waiting).
// k_elias_encode: every CTA scans its 64 buckets' counts from that prefix,
// and each warp assembles one bucket at a time in shared memory (one warp
// scan of bit lengths per 32 code words, then shared-memory atomicOr of at
// most three words per lane) and stores it with coalesced 32-bit writes.
// Decode: one thread per bucket walks its stream with a 64-bit window; an
// 8-bit lookahead table decodes every codeword of up to 8 bits (all of them
// for 4-bit codes) in one step.
#include "gc_common.cuh"

namespace gc {
namespace {

constexpr int kChunk = 64;                          // buckets per CTA
constexpr int kBucketsPerWarp = kChunk / kWarpsPerBlock;
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

struct Ws {
    uint32_t* ticket;
    uint32_t* chunk;    // [nchunks + 1]: per-CTA word totals, then their exclusive prefix
    uint32_t* counts;   // [nbuckets]: words of each bucket
};

inline size_t chunk_bytes(int64_t nchunks) {
    return static_cast<size_t>(div_up((nchunks + 1) * 4, 16) * 16);
}

Ws ws_layout(void* ws, int64_t nchunks) {
    char* p = static_cast<char*>(ws);
    Ws w;
    w.ticket = reinterpret_cast<uint32_t*>(p);
    w.chunk = reinterpret_cast<uint32_t*>(p + kTicketBytes);
    w.counts = reinterpret_cast<uint32_t*>(p + kTicketBytes + chunk_bytes(nchunks));
    return w;
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

// ---------------------------------------------------------------- count

struct CountArgs {
    const uint8_t* codes;
    int64_t n;
    int d;
    int64_t nbuckets;
    Ws ws;
};

template <bool FOUR>
__global__ void __launch_bounds__(kThreads) k_elias_count(CountArgs a) {
    __shared__ uint32_t lut[256];
    __shared__ uint32_t wsum[kWarpsPerBlock];
    __shared__ uint32_t scan_carry;
    __shared__ bool is_last;
    build_lut<FOUR>(lut);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t warp_words = 0;
    for (int j = 0; j < kBucketsPerWarp; ++j) {
        const int64_t b = static_cast<int64_t>(blockIdx.x) * kChunk + warp * kBucketsPerWarp + j;
        if (b >= a.nbuckets) break;
        const BucketBytes bb = bucket_bytes<FOUR>(a.codes, a.n, a.d, b);
        const int nw_in = (bb.valid + 3) >> 2;
        int bits = 0;
        for (int k = lane; k < nw_in; k += 32) {
            uint64_t acc;
            bits += word_bits<FOUR>(bb, k, lut, acc);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) bits += __shfl_xor_sync(0xffffffffu, bits, o);
        const uint32_t nw = static_cast<uint32_t>((32 + bits + 31) >> 5);
        if (lane == 0) a.ws.counts[b] = nw;
        warp_words += nw;
    }
    if (lane == 0) wsum[warp] = warp_words;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < kWarpsPerBlock; ++w) t += wsum[w];
        a.ws.chunk[blockIdx.x] = t;
        __threadfence();
        is_last = atomicAdd(a.ws.ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!is_last) return;
    // The last CTA: exclusive prefix of the per-CTA totals, in place, and
    // the grand total after them.  Every other CTA fenced its total before
    // taking its ticket; the totals are read from L2.
    __threadfence();
    const int nchunks = static_cast<int>(gridDim.x);
    if (threadIdx.x == 0) scan_carry = 0;
    __syncthreads();
    for (int base = 0; base < nchunks; base += kThreads) {
        const int i = base + threadIdx.x;
        const uint32_t v = i < nchunks ? __ldcg(a.ws.chunk + i) : 0u;
        const int incl = warp_incl_sum(static_cast<int>(v), lane);
        if (lane == 31) wsum[warp] = static_cast<uint32_t>(incl);
        __syncthreads();
        uint32_t before = scan_carry;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        if (i < nchunks) a.ws.chunk[i] = before + static_cast<uint32_t>(incl) - v;
        __syncthreads();
        if (threadIdx.x == kThreads - 1) scan_carry = before + static_cast<uint32_t>(incl);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.ws.chunk[nchunks] = scan_carry;
        *a.ws.ticket = 0u;
    }
}

// ---------------------------------------------------------------- encode

struct EncodeArgs {
    const uint8_t* codes;
    const float* norms;
    int64_t n;
    int d;
    int64_t nbuckets;
    Ws ws;
    uint32_t* words;
    uint32_t* offsets;
    int stage_stride;   // staging words per warp
};

template <bool FOUR>
__global__ void __launch_bounds__(kThreads) k_elias_encode(EncodeArgs a) {
    extern __shared__ uint32_t smem[];
    uint32_t* lut = smem;
    uint32_t* offs = smem + 256;                       // [kChunk]
    uint32_t* stage_all = smem + 256 + kChunk;
    build_lut<FOUR>(lut);
    for (int i = threadIdx.x; i < kWarpsPerBlock * a.stage_stride; i += kThreads) stage_all[i] = 0u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * kChunk;
    if (warp == 0) {
        const int64_t ba = b0 + 2 * lane, bb = ba + 1;
        const uint32_t c0 = ba < a.nbuckets ? a.ws.counts[ba] : 0u;
        const uint32_t c1 = bb < a.nbuckets ? a.ws.counts[bb] : 0u;
        const int incl = warp_incl_sum(static_cast<int>(c0 + c1), lane);
        const uint32_t o0 = a.ws.chunk[blockIdx.x] + static_cast<uint32_t>(incl) - c0 - c1;
        offs[2 * lane] = o0;
        offs[2 * lane + 1] = o0 + c0;
        if (ba < a.nbuckets) a.offsets[ba] = o0;
        if (bb < a.nbuckets) a.offsets[bb] = o0 + c0;
        if (blockIdx.x == gridDim.x - 1 && lane == 0) a.offsets[a.nbuckets] = a.ws.chunk[gridDim.x];
    }
    __syncthreads();
    uint32_t* stage = stage_all + warp * a.stage_stride;
    for (int j = 0; j < kBucketsPerWarp; ++j) {
        const int local = warp * kBucketsPerWarp + j;
        const int64_t b = b0 + local;
        if (b >= a.nbuckets) break;
        const BucketBytes bb = bucket_bytes<FOUR>(a.codes, a.n, a.d, b);
        const int nw_in = (bb.valid + 3) >> 2;
        if (lane == 0) stage[0] = __float_as_uint(__ldg(a.norms + b));
        uint32_t pos = 32;
        for (int k0 = 0; k0 < nw_in; k0 += 32) {
            uint64_t acc;
            const int len = word_bits<FOUR>(bb, k0 + lane, lut, acc);
            const int incl = warp_incl_sum(len, lane);
            emit(stage, pos + static_cast<uint32_t>(incl - len), acc, len);
            pos += static_cast<uint32_t>(__shfl_sync(0xffffffffu, incl, 31));
        }
        __syncwarp();
        const int nw = static_cast<int>((pos + 31) >> 5);
        uint32_t* dst = a.words + offs[local];
        for (int k = lane; k < nw; k += 32) {
            dst[k] = stage[k];
            stage[k] = 0u;
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------- decode

struct DecodeArgs {
    const uint32_t* words;
    const uint32_t* offsets;
    int64_t n;
    int d;
    int64_t nbuckets;
    int s;
    uint8_t* codes;
    float* norms;
    int* status;
};

// Lookahead table: the codeword (+ sign) at the top of an 8-bit window, as
// (level << 5) | (sign << 4) | length, or 0 when it does not end inside the
// window.
__device__ __forceinline__ uint32_t decode_entry(uint32_t x) {
    int pos = 0;
    uint32_t N = 1;
    for (;;) {
        if (pos >= 8) return 0u;
        const uint32_t bit = (x >> (7 - pos)) & 1u;
        ++pos;
        if (!bit) break;
        if (pos + static_cast<int>(N) > 8) return 0u;
        const uint32_t v = ((x << (pos - 1)) & 255u) >> (8 - (N + 1));
        pos += static_cast<int>(N);
        N = v;
    }
    const uint32_t level = N - 1u;
    uint32_t sign = 0u;
    if (level) {
        if (pos >= 8) return 0u;
        sign = (x >> (7 - pos)) & 1u;
        ++pos;
    }
    return (level << 5) | (sign << 4) | static_cast<uint32_t>(pos);
}

template <bool FOUR>
__global__ void __launch_bounds__(kThreads) k_elias_decode(DecodeArgs a) {
    __shared__ uint32_t lut[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) lut[i] = decode_entry(static_cast<uint32_t>(i));
    __syncthreads();
    const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (b >= a.nbuckets) return;
    const int64_t lo = b * a.d;
    const int len = static_cast<int>((a.n - lo < a.d ? a.n - lo : static_cast<int64_t>(a.d)));
    const uint32_t w_lo = a.offsets[b], w_hi = a.offsets[b + 1];
    const uint32_t* src = a.words + w_lo;
    const int64_t avail = w_hi > w_lo ? static_cast<int64_t>(w_hi - w_lo) : 0;
    bool bad = avail == 0;
    a.norms[b] = __uint_as_float(avail ? __ldg(src) : 0u);
    int64_t next = 1;
    uint64_t win = 0;   // left-aligned
    int have = 0;
    auto refill = [&]() {
        const uint32_t w = next < avail ? __ldg(src + next) : 0u;
        win |= static_cast<uint64_t>(w) << (32 - have);
        have += 32;
        ++next;
    };
    refill();
    refill();
    int64_t used = 32;                 // stream bits consumed, norm included
    const uint32_t smax = static_cast<uint32_t>(a.s);
    uint8_t* out = a.codes + (FOUR ? lo / 2 : lo);
    uint32_t acc = 0;
    for (int e = 0; e < len; ++e) {
        if (have <= 32) refill();
        uint32_t level, sign;
        int clen;
        const uint32_t t = lut[win >> 56];
        if (t) {
            clen = static_cast<int>(t & 15u);
            sign = (t >> 4) & 1u;
            level = t >> 5;
        } else {
            // codeword longer than 8 bits (levels of 15 and above)
            uint32_t N = 1;
            int p = 0;
            for (;;) {
                const uint32_t bit = static_cast<uint32_t>((win << p) >> 63);
                ++p;
                if (!bit) break;
                if (N > 7) {                 // a level above 127: not a stream of codes
                    bad = true;
                    N = 1;
                    break;
                }
                const uint32_t v = static_cast<uint32_t>((win << (p - 1)) >> (64 - (N + 1)));
                p += static_cast<int>(N);
                N = v;
            }
            level = N - 1u;
            sign = 0u;
            if (level) {
                sign = static_cast<uint32_t>((win << p) >> 63);
                ++p;
            }
            clen = p;
        }
        win <<= clen;
        have -= clen;
        used += clen;
        if (level > smax) {
            bad = true;
            level = smax;
        }
        if (!level) sign = 0u;
        if (FOUR) {
            const uint32_t code = (sign << 3) | level;
            acc |= code << (8 * ((e >> 1) & 3) + ((e & 1) ? 0 : 4));
            if ((e & 7) == 7) {
                reinterpret_cast<uint32_t*>(out)[e >> 3] = acc;
                acc = 0u;
            }
        } else {
            acc |= ((sign << 7) | level) << (8 * (e & 3));
            if ((e & 3) == 3) {
                reinterpret_cast<uint32_t*>(out)[e >> 2] = acc;
                acc = 0u;
            }
        }
    }
    // the partial last word of a ragged bucket, byte by byte
    const int per_word = FOUR ? 8 : 4;
    const int rem = len % per_word;
    if (rem) {
        const int nbytes = FOUR ? (rem + 1) / 2 : rem;
        uint8_t* tail = out + (len / per_word) * 4;
        for (int j = 0; j < nbytes; ++j) tail[j] = static_cast<uint8_t>(acc >> (8 * j));
    }
    if (used > avail * 32) bad = true;
    if (bad && a.status) *a.status = GC_ERR_CORRUPT;
}

}  // namespace
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
    const int64_t nb = div_up(n, bucket), nchunks = div_up(nb, kChunk);
    return kTicketBytes + chunk_bytes(nchunks) + static_cast<size_t>(div_up(nb * 4, 16) * 16);
}

int qsgd_elias_encode(const uint8_t* codes, const float* norms, int64_t n, int bucket, int s_levels,
                      uint32_t* words, uint64_t capacity_words, uint32_t* offsets, void* workspace,
                      size_t ws_bytes, gc_stream_t stream) {
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
    if (n == 0) return cudaMemsetAsync(offsets, 0, sizeof(uint32_t), s) == cudaSuccess ? GC_OK : GC_ERR_CUDA;
    const bool four = s_levels <= 7;
    const int64_t nb = div_up(n, bucket), nchunks = div_up(nb, kChunk);
    const Ws ws = ws_layout(workspace, nchunks);
    if (cudaMemsetAsync(ws.ticket, 0, kTicketBytes, s) != cudaSuccess) return GC_ERR_CUDA;
    CountArgs ca{codes, n, bucket, nb, ws};
    const unsigned grid = static_cast<unsigned>(nchunks);
    if (four)
        k_elias_count<true><<<grid, kThreads, 0, s>>>(ca);
    else
        k_elias_count<false><<<grid, kThreads, 0, s>>>(ca);
    if (cudaGetLastError() != cudaSuccess) return GC_ERR_CUDA;
    EncodeArgs ea{codes, norms, n, bucket, nb, ws, words, offsets,
                  static_cast<int>(bucket_max_words(bucket, four)) + 2};
    const size_t smem = sizeof(uint32_t) * (256 + kChunk + static_cast<size_t>(kWarpsPerBlock) * ea.stage_stride);
    if (four)
        k_elias_encode<true><<<grid, kThreads, smem, s>>>(ea);
    else
        k_elias_encode<false><<<grid, kThreads, smem, s>>>(ea);
    return launch_status();
}

int qsgd_elias_decode(const uint32_t* words, const uint32_t* offsets, int64_t n, int bucket, int s_levels,
                      uint8_t* codes, float* norms, int* d_status, gc_stream_t stream) {
    if (n < 0 || !valid_bucket(bucket) || s_levels < 1 || s_levels > 127) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!words || !offsets || !codes || !norms) return GC_ERR_INVALID;
    if (!aligned16(words) || !aligned16(offsets) || !aligned16(codes) || !aligned16(norms) ||
        (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)))
        return GC_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nb = div_up(n, bucket);
    DecodeArgs a{words, offsets, n, bucket, nb, s_levels, codes, norms, d_status};
    const unsigned grid = static_cast<unsigned>(div_up(nb, kThreads));
    if (s_levels <= 7)
        k_elias_decode<true><<<grid, kThreads, 0, s>>>(a);
    else
        k_elias_decode<false><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

}  // extern "C"
