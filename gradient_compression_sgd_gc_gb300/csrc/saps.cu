// saps.cu -- SAPS seeded random-mask sparsification (stream compaction with a
// single-pass decoupled look-back scan), peer averaging over a perfect
// matching, and the EASGD elastic step.
//
// Sources: "Communication-Efficient Decentralized Learning with
// Sparsification and Adaptive Peer Selection", section II (coordinator sends
// the round seed; all workers draw the same Bernoulli mask; single-peer
// gossip with a doubly stochastic matrix; Algorithm 2 lines 9-10 average the
// received sparsified model); EASGD local and global updates from the IMerge
// design notes.  The look-back scan follows Merrill and Garland,
// "Single-pass Parallel Prefix Scan with Decoupled Look-back" (NVIDIA
// technical report NVR-2016-002).
#include "gc_common.cuh"
#include "../../include/gc_gb300_testing.h"

namespace gc {
namespace {

// ------------------------------------------------------------------ K6

constexpr int kItems = 16;                         // rounds of 32 elements per warp
constexpr int kWarpSpan = 32 * kItems;             // 512 elements per warp
constexpr int kTileElems = kWarpsPerBlock * kWarpSpan;   // 4096 elements per CTA tile
constexpr size_t kWsHeader = 64;                   // tile counter + padding

struct MaskArgs {
    int64_t n;
    uint64_t seed_t;
    uint32_t thr;                 // ceil(p * 2^24)
    int W;
    PtrTable<const float*> models;
    PtrTable<float*> vals;
    uint32_t* idx;
    int64_t capacity;
    uint64_t* d_count;
    unsigned long long* counter; // dynamic tile counter (workspace)
    uint64_t* state;             // per-tile look-back state (workspace)
    int64_t ntiles;
    int* d_status;
    uint32_t* group_mask = nullptr;  // per 32 elements: the mask bits (workspace), or null
    uint32_t* group_excl = nullptr;  // per 32 elements: masked entries before them, or null
    uint64_t wait_ns = 1000000000ull;  // bound on each look-back wait
    int64_t withhold_tile = -1;        // test hook: this tile never publishes (-1: none)
};

// Exclusive prefix of tile `tile` whose own count `agg` it has already
// published (publish_aggregate); run by one warp.  Walks back over its
// predecessors 32 at a time (one coalesced 256-byte read of their state
// words) until it meets one that has published its inclusive prefix, then
// publishes its own.  Pending predecessors are polled without sleeping
// (they publish their aggregate as soon as their mask is counted); every
// wait is bounded: after a.wait_ns the missing predecessors count as zero
// and GC_ERR_TIMEOUT is recorded.
__device__ uint64_t walk_back(const MaskArgs& a, int64_t tile, uint64_t agg, int lane) {
    const bool publish = tile != a.withhold_tile;
    if (tile == 0) return 0;
    bool timed_out = false;
    const uint64_t excl = lookback_exclusive(a.state, tile, lane, a.wait_ns, 0u, timed_out);
    if (lane == 0) {
        if (publish) st_state(a.state + tile, kFlagPrefix | (excl + agg));
        if (timed_out) atomicExch(a.d_status, GC_ERR_TIMEOUT);
    }
    return excl;
}

// Publishes tile `tile`'s aggregate (its inclusive prefix for tile 0).
__device__ __forceinline__ void publish_aggregate(const MaskArgs& a, int64_t tile, uint64_t agg, int lane) {
    if (lane == 0 && tile != a.withhold_tile)
        st_state(a.state + tile, (tile == 0 ? kFlagPrefix : kFlagAgg) | agg);
}

constexpr int kListCap = 1024;                // masked indices kept for a tile's deferred write
constexpr int kGroups = kTileElems / 32;      // 32-element groups per tile

struct TileStage {
    uint32_t gmask[kGroups];    // mask bits of each group
    uint32_t gex[kGroups];      // masked entries of the tile before each group
    int64_t tile;
    uint32_t agg;               // masked entries of the tile
};

template <bool CHECK>
__device__ __forceinline__ uint32_t hash_rounds(const MaskArgs& a, int64_t wbase, int lane) {
    uint32_t my_mask = 0;
#pragma unroll 4
    for (int r = 0; r < kItems; ++r) {
        const int64_t e = wbase + 32 * r + lane;
        bool hit = splitmix64_top24(a.seed_t ^ static_cast<uint64_t>(e)) < a.thr;
        if (CHECK) hit = hit && e < a.n;
        const uint32_t m = __ballot_sync(0xffffffffu, hit);
        if (lane == r) my_mask = m;
    }
    return my_mask;
}

// The total count, written by the CTA that writes the last tile.
__device__ __forceinline__ void finish_count(const MaskArgs& a, int64_t tile, uint64_t excl, uint32_t agg) {
    if (threadIdx.x == 0 && tile == a.ntiles - 1) {
        const uint64_t total = excl + agg;
        *a.d_count = total;
        if (total > static_cast<uint64_t>(a.capacity)) atomicExch(a.d_status, GC_ERR_CAPACITY);
    }
}

// The group tables of a tile whose exclusive prefix is `excl`.
__device__ __forceinline__ void write_groups(const MaskArgs& a, const TileStage& st, uint64_t excl) {
    if (a.group_mask == nullptr) return;
    const int64_t g0 = st.tile * kGroups;
    for (int g = threadIdx.x; g < kGroups; g += kThreads) {
        if ((g0 + g) * 32 < a.n) {
            a.group_mask[g0 + g] = st.gmask[g];
            a.group_excl[g0 + g] = static_cast<uint32_t>(excl + st.gex[g]);
        }
    }
}

// Output positions start .. start+count-1 from a list of indices: idx, then
// every worker's vals with one (entry, worker) pair per thread, so that all
// the random reads are in flight at once; stores stay coalesced per worker.
// Positions at or above the capacity are dropped.
__device__ void write_list(const MaskArgs& a, const uint32_t* list, uint64_t start, uint32_t count) {
    const uint64_t cap = static_cast<uint64_t>(a.capacity);
    const uint32_t kept = cap > start ? static_cast<uint32_t>(min(static_cast<uint64_t>(count), cap - start)) : 0u;
    for (uint32_t k = threadIdx.x; k < kept; k += kThreads) a.idx[start + k] = list[k];
    const uint32_t pairs = kept * static_cast<uint32_t>(a.W);
    for (uint32_t q = threadIdx.x; q < pairs; q += kThreads) {
        const uint32_t w = q / kept;
        const uint32_t k = q - w * kept;
        a.vals.p[w][start + k] = __ldg(a.models.p[w] + list[k]);
    }
}

// K6: a persistent grid; each CTA takes 4096-element tiles in order from a
// dynamic counter, so every predecessor of a claimed tile is held by a
// running CTA.  Warp w hashes elements tile*4096 + 512w + 32r + lane (r < 16)
// and keeps the ballot of round r in lane r; one block scan gives the tile's
// count, which is published at once.  The tile's masked indices are listed in
// shared memory and its prefix is only looked up after the CTA has hashed and
// published its NEXT tile: by then the predecessors have long published, so
// the look-back is short and its round trips overlap other work.  Then idx[],
// every worker's vals[] and the per-group tables (mask bits and the masked
// count before each 32-element group, used by the fused pair-average +
// elastic step) are written.  A tile with more masked entries than one list
// holds takes its prefix at once and is written in chunks through both lists.
__global__ void __launch_bounds__(kThreads)
k_saps_mask_compact(const MaskArgs a) {
    __shared__ uint32_t s_list[2 * kListCap];   // one list per stage; both for a dense tile
    __shared__ TileStage s_stage[2];
    __shared__ uint32_t s_warp_excl[kWarpsPerBlock];
    __shared__ uint32_t s_warp_tot[kWarpsPerBlock];
    __shared__ unsigned long long s_tile;
    __shared__ uint64_t s_excl;

    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    int cur = 0;              // stage (and list) of the tile being hashed
    bool have_prev = false;   // stage cur ^ 1 holds a tile waiting for its prefix
    // Every condition below that guards a barrier is uniform over the CTA.
    while (true) {
        if (threadIdx.x == 0) s_tile = atomicAdd(a.counter, 1ull);
        __syncthreads();
        const int64_t tile = static_cast<int64_t>(s_tile);
        const bool have = tile < a.ntiles;
        TileStage& st = s_stage[cur];
        uint32_t* list = s_list + cur * kListCap;
        const int64_t wbase = tile * kTileElems + static_cast<int64_t>(wib) * kWarpSpan;
        uint32_t my_mask = 0, round_excl = 0;
        if (have) {
            my_mask = wbase + kWarpSpan <= a.n ? hash_rounds<false>(a, wbase, lane)
                                               : hash_rounds<true>(a, wbase, lane);
            const uint32_t cnt = __popc(my_mask);
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < kItems; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            round_excl = incl - cnt;
            if (lane == kItems - 1) s_warp_tot[wib] = incl;
        }
        __syncthreads();
        if (have && wib == 0) {
            const uint32_t v = lane < kWarpsPerBlock ? s_warp_tot[lane] : 0u;
            uint32_t vi = v;
#pragma unroll
            for (int o = 1; o < kWarpsPerBlock; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, vi, o);
                if (lane >= o) vi += t;
            }
            if (lane < kWarpsPerBlock) s_warp_excl[lane] = vi - v;
            const uint32_t agg = __shfl_sync(0xffffffffu, vi, kWarpsPerBlock - 1);
            publish_aggregate(a, tile, agg, lane);
            if (lane == 0) {
                st.agg = agg;
                st.tile = tile;
            }
        }
        __syncthreads();
        // tile entries before round `lane` of this warp (lanes < kItems)
        const uint32_t before = have ? s_warp_excl[wib] + round_excl : 0u;
        const uint32_t agg = have ? st.agg : 0u;
        const uint32_t eb = static_cast<uint32_t>(wbase) + 32u * static_cast<uint32_t>(lane);
        if (have) {
            if (lane < kItems) {
                st.gmask[wib * kItems + lane] = my_mask;
                st.gex[wib * kItems + lane] = before;
            }
            if (agg <= static_cast<uint32_t>(kListCap)) {
                uint32_t pos = before;
                for (uint32_t mm = my_mask; mm != 0; mm &= mm - 1) list[pos++] = eb + (__ffs(mm) - 1);
            }
        }
        if (have_prev) {
            const TileStage& pv = s_stage[cur ^ 1];
            if (wib == 0) {
                const uint64_t ex = walk_back(a, pv.tile, pv.agg, lane);
                if (lane == 0) s_excl = ex;
            }
            __syncthreads();
            const uint64_t ex = s_excl;
            write_groups(a, pv, ex);
            write_list(a, s_list + (cur ^ 1) * kListCap, ex, pv.agg);
            finish_count(a, pv.tile, ex, pv.agg);
        }
        if (!have) break;
        if (agg > static_cast<uint32_t>(kListCap)) {
            __syncthreads();                  // s_excl and the previous tile's list are free
            if (wib == 0) {
                const uint64_t ex = walk_back(a, tile, agg, lane);
                if (lane == 0) s_excl = ex;
            }
            __syncthreads();
            const uint64_t ex = s_excl;
            write_groups(a, st, ex);
            for (uint32_t c0 = 0; c0 < agg; c0 += 2 * kListCap) {
                uint32_t pos = before;
                for (uint32_t mm = my_mask; mm != 0; mm &= mm - 1, ++pos)
                    if (pos - c0 < static_cast<uint32_t>(2 * kListCap)) s_list[pos - c0] = eb + (__ffs(mm) - 1);
                __syncthreads();
                write_list(a, s_list, ex + c0, min(agg - c0, static_cast<uint32_t>(2 * kListCap)));
                __syncthreads();
            }
            finish_count(a, tile, ex, agg);
            have_prev = false;
        } else {
            have_prev = true;
            cur ^= 1;
        }
    }
}

// Grid of the compaction: as many CTAs as are resident at once, at most one
// per tile.
int launch_mask(const MaskArgs& a, cudaStream_t s) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_saps_mask_compact, kThreads, 0) != cudaSuccess)
        return GC_ERR_CUDA;
    const int64_t resident = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    k_saps_mask_compact<<<static_cast<unsigned>(a.ntiles < resident ? a.ntiles : resident), kThreads, 0, s>>>(a);
    return launch_status();
}

// ------------------------------------------------------------------ K7

struct AvgArgs {
    PtrTable<float*> models;
    PtrTable<const float*> vals;
    int pairs[GC_MAX_WORKERS];
    int W;
    const uint32_t* idx;
    const uint64_t* d_count;
    int64_t capacity;
};

// Every received value of entry k is loaded before any model is written
// (for up to MAXP pairs), so that all of an entry's reads and its 2 * (W/2)
// scattered writes are in flight together.
template <int MAXP>
__global__ void __launch_bounds__(kThreads)
k_saps_peer_average(const AvgArgs a) {
    const uint64_t cnt = *a.d_count;
    const int64_t count = cnt < static_cast<uint64_t>(a.capacity) ? static_cast<int64_t>(cnt) : a.capacity;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int P = a.W / 2;
    for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < count; k += stride) {
        const uint32_t e = a.idx[k];
        if (MAXP > 0) {
            float va[MAXP > 0 ? MAXP : 1], vb[MAXP > 0 ? MAXP : 1];
#pragma unroll
            for (int q = 0; q < MAXP; ++q) {
                if (q < P) {
                    va[q] = __ldg(a.vals.p[a.pairs[2 * q]] + k);
                    vb[q] = __ldg(a.vals.p[a.pairs[2 * q + 1]] + k);
                }
            }
#pragma unroll
            for (int q = 0; q < MAXP; ++q) {
                if (q < P) {
                    const float v = __fmul_rn(__fadd_rn(va[q], vb[q]), 0.5f);
                    a.models.p[a.pairs[2 * q]][e] = v;
                    a.models.p[a.pairs[2 * q + 1]][e] = v;
                }
            }
        } else {
            for (int q = 0; q < P; ++q) {
                const int pa = a.pairs[2 * q], pb = a.pairs[2 * q + 1];
                const float v = __fmul_rn(__fadd_rn(__ldg(a.vals.p[pa] + k), __ldg(a.vals.p[pb] + k)), 0.5f);
                a.models.p[pa][e] = v;
                a.models.p[pb][e] = v;
            }
        }
    }
}

// ------------------------------------------------------------------ K8

struct EasgdArgs {
    PtrTable<float*> models;
    int W;
    int64_t n;
    float alpha, beta, inv_w;
    float* center;
};

__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

__device__ __forceinline__ float elastic(float w, float c, float alpha) {
    return fmaf(-alpha, __fsub_rn(w, c), w);
}

// K8, W <= 16: every worker's float4 at element 4i and the center's are
// loaded once, the pre-step mean is formed in worker order, and all W + 1
// vectors are written back.
template <int MAXW>
__global__ void __launch_bounds__(kThreads, 2)
k_easgd(const EasgdArgs a) {
    const int64_t nv = a.n >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i = gtid; i < nv; i += stride) {
        float4 m[MAXW];
#pragma unroll
        for (int k = 0; k < MAXW; ++k)
            if (k < a.W) m[k] = ld_f4(a.models.p[k] + 4 * i);
        const float4 c = ld_f4(a.center + 4 * i);
        float4 sum = m[0];
#pragma unroll
        for (int k = 1; k < MAXW; ++k)
            if (k < a.W) sum = f4_add(sum, m[k]);
#pragma unroll
        for (int k = 0; k < MAXW; ++k) {
            if (k < a.W) {
                st_stream_f4(a.models.p[k] + 4 * i,
                             make_float4(elastic(m[k].x, c.x, a.alpha), elastic(m[k].y, c.y, a.alpha),
                                         elastic(m[k].z, c.z, a.alpha), elastic(m[k].w, c.w, a.alpha)));
            }
        }
        const float4 mean = make_float4(__fmul_rn(sum.x, a.inv_w), __fmul_rn(sum.y, a.inv_w),
                                        __fmul_rn(sum.z, a.inv_w), __fmul_rn(sum.w, a.inv_w));
        st_stream_f4(a.center + 4 * i,
                     make_float4(fmaf(a.beta, __fsub_rn(mean.x, c.x), c.x), fmaf(a.beta, __fsub_rn(mean.y, c.y), c.y),
                                 fmaf(a.beta, __fsub_rn(mean.z, c.z), c.z), fmaf(a.beta, __fsub_rn(mean.w, c.w), c.w)));
    }
    // tail: the last n % 4 elements
    const int64_t t = (nv << 2) + gtid;
    if (gtid < (a.n & 3)) {
        const float c = a.center[t];
        float sum = 0.0f;
        for (int k = 0; k < a.W; ++k) sum = __fadd_rn(sum, a.models.p[k][t]);
        for (int k = 0; k < a.W; ++k) a.models.p[k][t] = elastic(a.models.p[k][t], c, a.alpha);
        a.center[t] = fmaf(a.beta, __fsub_rn(__fmul_rn(sum, a.inv_w), c), c);
    }
}

// K8, any W <= 64: two passes per element (sum, then update), the second
// re-reading the models.
__global__ void __launch_bounds__(kThreads)
k_easgd_wide(const EasgdArgs a) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < a.n; i += stride) {
        const float c = a.center[i];
        float sum = 0.0f;
        for (int k = 0; k < a.W; ++k) sum = __fadd_rn(sum, a.models.p[k][i]);
        for (int k = 0; k < a.W; ++k) a.models.p[k][i] = elastic(a.models.p[k][i], c, a.alpha);
        a.center[i] = fmaf(a.beta, __fsub_rn(__fmul_rn(sum, a.inv_w), c), c);
    }
}

// ------------------------------------------------------------------ one-pass round

// A whole SAPS round in one pass over the models: the round's mask and its
// compaction (idx, vals) with the decoupled look-back above, the pair
// average of the masked coordinates and the EASGD elastic step.  Each CTA
// takes a 4096-element tile from the dynamic counter, issues its first
// round of loads (one float4 of every worker and of the center per thread;
// the tile is streamed in rounds of 4 x NT elements), hashes all 4096
// elements, ranks the masked ones with one block scan per pair of rounds and
// publishes the tile's aggregate at once.  Then it streams the rounds
// without further barriers: a masked coordinate's pre-average values go to a
// shared-memory stash (the compacted output) and to a per-thread scratch row
// from which each worker reads its partner's value for the pair average; the
// elastic step and the center update are written back.  Last the CTA walks
// back for its exclusive prefix -- its predecessors have streamed their
// tiles by then -- and writes idx and vals from the stash.  A tile with more
// masked coordinates than the stash holds walks back first and writes them
// directly.  Results equal saps_mask_compact + saps_peer_average +
// easgd_step bit for bit while the count fits the capacity.
constexpr int kStash = 384;                      // masked entries kept per tile
// Threads per CTA of the one-pass round: 256 (two CTAs per SM) measured
// ahead of 128 (four per SM; 553 against 541 us at p = 0.01).
constexpr int kRoundThreads = 256;

struct RoundArgs {
    MaskArgs m;                                  // mask, compaction, look-back
    PtrTable<float*> models;
    int partner[GC_MAX_WORKERS];
    float alpha, beta, inv_w;
    float* center;
};

// Round r's float4 of every worker and of the center for element i0.
template <int MAXW>
__device__ __forceinline__ void round_load(const RoundArgs& a, int64_t i0, float4 (&v)[MAXW], float4& c) {
#pragma unroll
    for (int k = 0; k < MAXW; ++k)
        if (k < a.m.W) v[k] = ld_f4(a.models.p[k] + i0);
    c = ld_f4(a.center + i0);
}

template <int MAXW, int NT>
__global__ void __launch_bounds__(NT, 512 / NT)
k_saps_round(const RoundArgs a) {
    constexpr int kRoundN = 4 * NT;                   // elements per round
    constexpr int kRounds = kTileElems / kRoundN;     // 4 (256 threads) or 8 (128)
    constexpr int kPairs = kRounds / 2;               // round counts packed two per word
    constexpr int kNW = NT / 32;
    static_assert(kRounds * 4 <= 32 && kRounds % 2 == 0, "4 mask bits per round in one word");
    __shared__ float s_stash[kStash * MAXW];
    __shared__ uint32_t s_sidx[kStash];
    __shared__ float s_scratch[NT * MAXW];
    __shared__ uint32_t s_wsum[kPairs][kNW];
    __shared__ unsigned long long s_tile;
    __shared__ uint64_t s_excl;
    const MaskArgs& m = a.m;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_tile = atomicAdd(m.counter, 1ull);
    __syncthreads();
    const int64_t tile = static_cast<int64_t>(s_tile);
    const int64_t base = tile * kTileElems;
    const int W = m.W;
    const uint64_t cap = static_cast<uint64_t>(m.capacity);
    float* scratch = s_scratch + threadIdx.x * MAXW;

    // round 0's loads go out before the hashing
    float4 v[MAXW];
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t first = base + 4 * threadIdx.x;
    if (first + 4 <= m.n) round_load<MAXW>(a, first, v, c);
    // the mask of every round: 4 bits per round in `bits`
    uint32_t bits = 0;
#pragma unroll
    for (int r = 0; r < kRounds; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int64_t i = base + static_cast<int64_t>(r) * kRoundN + 4 * threadIdx.x + e;
            bits |= (i < m.n && splitmix64_top24(m.seed_t ^ static_cast<uint64_t>(i)) < m.thr ? 1u : 0u)
                    << (4 * r + e);
        }
    // per-round block scans, two rounds per 32-bit word (16-bit fields)
    uint32_t cw[kPairs], iw[kPairs];
#pragma unroll
    for (int q = 0; q < kPairs; ++q) {
        cw[q] = __popc((bits >> (8 * q)) & 0xFu) | (__popc((bits >> (8 * q + 4)) & 0xFu) << 16);
        iw[q] = cw[q];
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int q = 0; q < kPairs; ++q) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, iw[q], o);
            if (lane >= o) iw[q] += t;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int q = 0; q < kPairs; ++q) s_wsum[q][wib] = iw[q];
    }
    __syncthreads();
    // exclusive rank of this thread's first masked element in each round
    uint32_t rank_base[kRounds];
    uint32_t agg = 0;
#pragma unroll
    for (int q = 0; q < kPairs; ++q) {
        uint32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
            const uint32_t x = s_wsum[q][w];
            before += w < wib ? x : 0u;
            total += x;
        }
        const uint32_t ex = before + iw[q] - cw[q];
        rank_base[2 * q] = agg + (ex & 0xFFFFu);
        agg += total & 0xFFFFu;
        rank_base[2 * q + 1] = agg + (ex >> 16);
        agg += total >> 16;
    }
    const bool big = agg > static_cast<uint32_t>(kStash);
    if (wib == 0) {
        publish_aggregate(m, tile, agg, lane);
        if (big) {
            const uint64_t ex = walk_back(m, tile, agg, lane);
            if (lane == 0) s_excl = ex;
        }
    }
    if (big) __syncthreads();                    // block-uniform
    const uint64_t excl_big = big ? s_excl : 0;

#pragma unroll 1
    for (int r = 0; r < kRounds; ++r) {
        const int64_t i0 = base + static_cast<int64_t>(r) * kRoundN + 4 * threadIdx.x;
        if (i0 >= m.n) break;
        const uint32_t rb = (bits >> (4 * r)) & 15u;
        const uint32_t rank0 = rank_base[r];
        if (i0 + 4 <= m.n) {
            if (r > 0) round_load<MAXW>(a, i0, v, c);
            if (rb) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (!((rb >> e) & 1u)) continue;
                    const uint32_t rank = rank0 + __popc(rb & ((1u << e) - 1u));
#pragma unroll
                    for (int k = 0; k < MAXW; ++k)
                        if (k < W) scratch[k] = e == 0 ? v[k].x : e == 1 ? v[k].y : e == 2 ? v[k].z : v[k].w;
                    if (!big) {
                        s_sidx[rank] = static_cast<uint32_t>(i0 + e);
#pragma unroll
                        for (int k = 0; k < MAXW; ++k)
                            if (k < W) s_stash[rank * MAXW + k] = scratch[k];
                    } else if (excl_big + rank < cap) {
                        m.idx[excl_big + rank] = static_cast<uint32_t>(i0 + e);
#pragma unroll
                        for (int k = 0; k < MAXW; ++k)
                            if (k < W) m.vals.p[k][excl_big + rank] = scratch[k];
                    }
#pragma unroll
                    for (int k = 0; k < MAXW; ++k) {
                        if (k < W) {
                            float* dst = e == 0 ? &v[k].x : e == 1 ? &v[k].y : e == 2 ? &v[k].z : &v[k].w;
                            *dst = __fmul_rn(__fadd_rn(scratch[k], scratch[a.partner[k]]), 0.5f);
                        }
                    }
                }
            }
            float4 sum = v[0];
#pragma unroll
            for (int k = 1; k < MAXW; ++k)
                if (k < W) sum = f4_add(sum, v[k]);
#pragma unroll
            for (int k = 0; k < MAXW; ++k) {
                if (k < W) {
                    st_stream_f4(a.models.p[k] + i0,
                                 make_float4(elastic(v[k].x, c.x, a.alpha), elastic(v[k].y, c.y, a.alpha),
                                             elastic(v[k].z, c.z, a.alpha), elastic(v[k].w, c.w, a.alpha)));
                }
            }
            const float4 mean = make_float4(__fmul_rn(sum.x, a.inv_w), __fmul_rn(sum.y, a.inv_w),
                                            __fmul_rn(sum.z, a.inv_w), __fmul_rn(sum.w, a.inv_w));
            st_stream_f4(a.center + i0,
                         make_float4(fmaf(a.beta, __fsub_rn(mean.x, c.x), c.x), fmaf(a.beta, __fsub_rn(mean.y, c.y), c.y),
                                     fmaf(a.beta, __fsub_rn(mean.z, c.z), c.z), fmaf(a.beta, __fsub_rn(mean.w, c.w), c.w)));
        } else {
            // the last n % 4 elements, element by element
            for (int e = 0; i0 + e < m.n; ++e) {
                const int64_t i = i0 + e;
#pragma unroll
                for (int k = 0; k < MAXW; ++k)
                    if (k < W) scratch[k] = a.models.p[k][i];
                const float ce = a.center[i];
                const bool hit = (rb >> e) & 1u;
                if (hit) {
                    const uint32_t rank = rank0 + __popc(rb & ((1u << e) - 1u));
                    if (!big) {
                        s_sidx[rank] = static_cast<uint32_t>(i);
#pragma unroll
                        for (int k = 0; k < MAXW; ++k)
                            if (k < W) s_stash[rank * MAXW + k] = scratch[k];
                    } else if (excl_big + rank < cap) {
                        m.idx[excl_big + rank] = static_cast<uint32_t>(i);
#pragma unroll
                        for (int k = 0; k < MAXW; ++k)
                            if (k < W) m.vals.p[k][excl_big + rank] = scratch[k];
                    }
                }
                float y[MAXW];
#pragma unroll
                for (int k = 0; k < MAXW; ++k)
                    if (k < W) y[k] = hit ? __fmul_rn(__fadd_rn(scratch[k], scratch[a.partner[k]]), 0.5f) : scratch[k];
                float sum = y[0];
#pragma unroll
                for (int k = 1; k < MAXW; ++k)
                    if (k < W) sum = __fadd_rn(sum, y[k]);
#pragma unroll
                for (int k = 0; k < MAXW; ++k)
                    if (k < W) a.models.p[k][i] = elastic(y[k], ce, a.alpha);
                a.center[i] = fmaf(a.beta, __fsub_rn(__fmul_rn(sum, a.inv_w), ce), ce);
            }
        }
    }

    // C. the exclusive prefix (predecessors have long published), then idx
    // and vals from the stash
    if (!big && wib == 0) {
        const uint64_t ex = walk_back(m, tile, agg, lane);
        if (lane == 0) s_excl = ex;
    }
    __syncthreads();
    const uint64_t excl = s_excl;
    if (!big) {
        const uint32_t kept = cap > excl ? static_cast<uint32_t>(min(static_cast<uint64_t>(agg), cap - excl)) : 0u;
        for (uint32_t k = threadIdx.x; k < kept; k += NT) m.idx[excl + k] = s_sidx[k];
        const uint32_t pairs = kept * static_cast<uint32_t>(W);
        for (uint32_t q = threadIdx.x; q < pairs; q += NT) {
            const uint32_t w = q / kept;
            const uint32_t k = q - w * kept;
            m.vals.p[w][excl + k] = s_stash[k * MAXW + w];
        }
    }
    if (threadIdx.x == 0 && tile == m.ntiles - 1) {
        const uint64_t total = excl + agg;
        *m.d_count = total;
        if (total > cap) atomicExch(m.d_status, GC_ERR_CAPACITY);
    }
}

int64_t mask_tiles(int64_t n) { return (n + kTileElems - 1) / kTileElems; }

// 32-element groups of n, rounded up to a multiple of 4 (16-byte alignment).
int64_t ws_groups(int64_t n) { return ((n + 31) / 32 + 3) / 4 * 4; }

uint32_t* ws_group_mask(void* ws, int64_t n) {
    return reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + kWsHeader + sizeof(uint64_t) * mask_tiles(n));
}

uint32_t* ws_group_excl(void* ws, int64_t n) { return ws_group_mask(ws, n) + ws_groups(n); }

// ------------------------------------------------------------------ K7 + K8 fused

// SAPS pair averaging applied inside the EASGD pass.  The peers' values come
// from the compacted payload vals[w][rank]; the rank of a masked element is
// found from the per-32-element tables saps_mask_compact leaves in the
// workspace (mask bits + masked entries before the group), so the models are
// streamed once and never written at scattered addresses.  Worker w's
// masked coordinate becomes (x_w + received x_partner) * 0.5 -- the same
// value saps_peer_average writes -- and the elastic step then runs on it.
struct FusedArgs {
    PtrTable<float*> models;
    PtrTable<const float*> vals;
    int partner[GC_MAX_WORKERS];
    int W;
    int64_t n;
    float alpha, beta, inv_w;
    float* center;
    const uint32_t* group_mask;
    const uint32_t* group_excl;
    const uint64_t* d_count;
    int64_t capacity;
};

// Masked coordinates among the 4 elements of chunk i: the received peer
// values are averaged into the registers m[].
template <int MAXW>
__device__ __forceinline__ void average_masked(const FusedArgs& a, float4 (&m)[MAXW], uint32_t bits,
                                               uint32_t base, uint64_t usable) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (!((bits >> e) & 1u)) continue;
        const uint32_t rank = base + __popc(bits & ((1u << e) - 1u));
        if (rank >= usable) continue;
        float recv[MAXW];
#pragma unroll
        for (int k = 0; k < MAXW; ++k)
            if (k < a.W) recv[k] = __ldg(a.vals.p[a.partner[k]] + rank);
#pragma unroll
        for (int k = 0; k < MAXW; ++k) {
            if (k < a.W) {
                float* x = e == 0 ? &m[k].x : e == 1 ? &m[k].y : e == 2 ? &m[k].z : &m[k].w;
                *x = __fmul_rn(__fadd_rn(*x, recv[k]), 0.5f);
            }
        }
    }
}

// Grid-stride over float4 chunks with the next chunk's group tables loaded
// one iteration ahead, so that the payload reads of a chunk are issued
// together with its model loads instead of after a dependent round trip
// (the grid is several waves of CTAs, each thread a few chunks).
template <int MAXW>
__global__ void __launch_bounds__(kThreads, 2)
k_saps_average_easgd(const FusedArgs a) {
    const uint64_t cnt = *a.d_count;
    const uint64_t usable = cnt < static_cast<uint64_t>(a.capacity) ? cnt : static_cast<uint64_t>(a.capacity);
    const int64_t nv = a.n >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    uint32_t gm = 0, ge = 0;
    if (first < nv) {
        gm = __ldg(a.group_mask + ((4 * first) >> 5));
        ge = __ldg(a.group_excl + ((4 * first) >> 5));
    }
    for (int64_t i = first; i < nv; i += stride) {
        float4 m[MAXW];
#pragma unroll
        for (int k = 0; k < MAXW; ++k)
            if (k < a.W) m[k] = ld_f4(a.models.p[k] + 4 * i);
        const float4 c = ld_f4(a.center + 4 * i);
        const int64_t nxt = i + stride;
        uint32_t gm_n = 0, ge_n = 0;
        if (nxt < nv) {
            gm_n = __ldg(a.group_mask + ((4 * nxt) >> 5));
            ge_n = __ldg(a.group_excl + ((4 * nxt) >> 5));
        }
        const uint32_t sh = static_cast<uint32_t>((4 * i) & 31);
        const uint32_t bits = (gm >> sh) & 15u;
        if (bits) average_masked<MAXW>(a, m, bits, ge + __popc(gm & ((1u << sh) - 1u)), usable);
        float4 sum = m[0];
#pragma unroll
        for (int k = 1; k < MAXW; ++k)
            if (k < a.W) sum = f4_add(sum, m[k]);
#pragma unroll
        for (int k = 0; k < MAXW; ++k) {
            if (k < a.W) {
                st_stream_f4(a.models.p[k] + 4 * i,
                             make_float4(elastic(m[k].x, c.x, a.alpha), elastic(m[k].y, c.y, a.alpha),
                                         elastic(m[k].z, c.z, a.alpha), elastic(m[k].w, c.w, a.alpha)));
            }
        }
        const float4 mean = make_float4(__fmul_rn(sum.x, a.inv_w), __fmul_rn(sum.y, a.inv_w),
                                        __fmul_rn(sum.z, a.inv_w), __fmul_rn(sum.w, a.inv_w));
        st_stream_f4(a.center + 4 * i,
                     make_float4(fmaf(a.beta, __fsub_rn(mean.x, c.x), c.x), fmaf(a.beta, __fsub_rn(mean.y, c.y), c.y),
                                 fmaf(a.beta, __fsub_rn(mean.z, c.z), c.z), fmaf(a.beta, __fsub_rn(mean.w, c.w), c.w)));
        gm = gm_n;
        ge = ge_n;
    }
    if (first == 0 && (a.n & 3)) {
        // the last n % 4 elements, one thread
        for (int64_t t = nv << 2; t < a.n; ++t) {
            const uint32_t gmt = __ldg(a.group_mask + (t >> 5));
            const uint32_t sh = static_cast<uint32_t>(t & 31);
            const bool hit = (gmt >> sh) & 1u;
            const uint32_t rank = __ldg(a.group_excl + (t >> 5)) + __popc(gmt & ((1u << sh) - 1u));
            float v[GC_MAX_WORKERS];
            for (int k = 0; k < a.W; ++k) v[k] = a.models.p[k][t];
            if (hit && rank < usable)
                for (int k = 0; k < a.W; ++k) v[k] = __fmul_rn(__fadd_rn(v[k], a.vals.p[a.partner[k]][rank]), 0.5f);
            const float c = a.center[t];
            float sum = 0.0f;
            for (int k = 0; k < a.W; ++k) sum = __fadd_rn(sum, v[k]);
            for (int k = 0; k < a.W; ++k) a.models.p[k][t] = elastic(v[k], c, a.alpha);
            a.center[t] = fmaf(a.beta, __fsub_rn(__fmul_rn(sum, a.inv_w), c), c);
        }
    }
}

// Any W <= 64: one element per thread, models read twice.
__global__ void __launch_bounds__(kThreads)
k_saps_average_easgd_wide(const FusedArgs a) {
    const uint64_t cnt = *a.d_count;
    const uint64_t usable = cnt < static_cast<uint64_t>(a.capacity) ? cnt : static_cast<uint64_t>(a.capacity);
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= a.n) return;
    const uint32_t gm = __ldg(a.group_mask + (t >> 5));
    const uint32_t sh = static_cast<uint32_t>(t & 31);
    const bool hit = (gm >> sh) & 1u;
    const uint32_t rank = __ldg(a.group_excl + (t >> 5)) + __popc(gm & ((1u << sh) - 1u));
    const bool avg = hit && rank < usable;
    const float c = a.center[t];
    float sum = 0.0f;
    for (int k = 0; k < a.W; ++k) {
        float v = a.models.p[k][t];
        if (avg) v = __fmul_rn(__fadd_rn(v, a.vals.p[a.partner[k]][rank]), 0.5f);
        sum = __fadd_rn(sum, v);
    }
    for (int k = 0; k < a.W; ++k) {
        float v = a.models.p[k][t];
        if (avg) v = __fmul_rn(__fadd_rn(v, a.vals.p[a.partner[k]][rank]), 0.5f);
        a.models.p[k][t] = elastic(v, c, a.alpha);
    }
    a.center[t] = fmaf(a.beta, __fsub_rn(__fmul_rn(sum, a.inv_w), c), c);
}



// ---------------------------------------------------------------- one rank per worker

// The pair average of a worker whose peer runs in another process: the peer's
// gathered values arrive in `peer` (same order as idx), and the masked
// coordinates become fl(fl(mine + peer) * 0.5) -- the same value the peer
// computes (fp addition commutes), and the value k_saps_peer_average writes.
struct RemoteAvgArgs {
    float* model;
    const uint32_t* idx;
    const uint64_t* d_count;
    const float* mine;
    const float* peer;
    int64_t capacity;
};

__global__ void __launch_bounds__(kThreads)
k_saps_pair_average_remote(const RemoteAvgArgs a) {
    const uint64_t cnt = *a.d_count;
    const int64_t count = cnt < static_cast<uint64_t>(a.capacity) ? static_cast<int64_t>(cnt) : a.capacity;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < count; k += stride)
        a.model[a.idx[k]] = __fmul_rn(__fadd_rn(__ldg(a.mine + k), __ldg(a.peer + k)), 0.5f);
}

// The elastic step of one worker given the sum of all W workers' models
// (formed by an all-reduce across processes): w <- w - alpha (w - c), and
// c <- c + beta (sum / W - c), as k_easgd does with the sum formed locally.
struct EasgdSumArgs {
    float* model;
    const float* sum;
    float* center;
    int64_t n;
    float alpha, beta, inv_w;
};

__global__ void __launch_bounds__(kThreads)
k_easgd_from_sum(const EasgdSumArgs a) {
    const int64_t nv = a.n >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i = gtid; i < nv; i += stride) {
        const float4 m = ld_f4(a.model + 4 * i);
        const float4 c = ld_f4(a.center + 4 * i);
        const float4 sm = ld_stream_f4(a.sum + 4 * i);
        st_stream_f4(a.model + 4 * i, make_float4(elastic(m.x, c.x, a.alpha), elastic(m.y, c.y, a.alpha),
                                                  elastic(m.z, c.z, a.alpha), elastic(m.w, c.w, a.alpha)));
        st_stream_f4(a.center + 4 * i,
                     make_float4(fmaf(a.beta, __fsub_rn(__fmul_rn(sm.x, a.inv_w), c.x), c.x),
                                 fmaf(a.beta, __fsub_rn(__fmul_rn(sm.y, a.inv_w), c.y), c.y),
                                 fmaf(a.beta, __fsub_rn(__fmul_rn(sm.z, a.inv_w), c.z), c.z),
                                 fmaf(a.beta, __fsub_rn(__fmul_rn(sm.w, a.inv_w), c.w), c.w)));
    }
    const int64_t t = (nv << 2) + gtid;
    if (gtid < (a.n & 3)) {
        const float c = a.center[t];
        a.model[t] = elastic(a.model[t], c, a.alpha);
        a.center[t] = fmaf(a.beta, __fsub_rn(__fmul_rn(a.sum[t], a.inv_w), c), c);
    }
}

}  // namespace
}  // namespace gc

using namespace gc;

extern "C" {

uint64_t saps_round_seed(uint64_t base_seed, uint64_t t) { return splitmix64(base_seed + t); }

int saps_matching(uint64_t seed_t, int W, int* pairs_out) {
    if (W < 2 || W > GC_MAX_WORKERS || (W & 1) || !pairs_out) return GC_ERR_INVALID;
    for (int i = 0; i < W; ++i) pairs_out[i] = i;
    const uint64_t base = splitmix64(seed_t);
    for (int i = W - 1; i >= 1; --i) {
        const int j = static_cast<int>(splitmix64(base ^ static_cast<uint64_t>(i)) % static_cast<uint64_t>(i + 1));
        const int tmp = pairs_out[i];
        pairs_out[i] = pairs_out[j];
        pairs_out[j] = tmp;
    }
    return GC_OK;
}

size_t saps_workspace_bytes(int64_t n) {
    if (n <= 0) return kWsHeader;
    // header | tile states (8 B per tile) | group mask (4 B per 32 elements) |
    // group exclusive counts (4 B per 32 elements), each part 16-byte aligned
    return kWsHeader + sizeof(uint64_t) * static_cast<size_t>(mask_tiles(n)) +
           2 * sizeof(uint32_t) * static_cast<size_t>(ws_groups(n));
}

static int mask_compact_impl(int64_t n, double p, uint64_t seed_t, const float* const* models, int W,
                             uint32_t* idx, float* const* vals, int64_t capacity, uint64_t* d_count,
                             void* workspace, size_t workspace_bytes, int* d_status, gc_stream_t stream,
                             int64_t withhold_tile, uint64_t wait_ns) {
    if (n < 0 || n > 0xFFFFFFFFll || W < 1 || W > GC_MAX_WORKERS || capacity < 0) return GC_ERR_INVALID;
    if (!(p > 0.0 && p <= 1.0)) return GC_ERR_INVALID;
    if (!d_count || !workspace || !d_status || !models || (capacity > 0 && (!idx || !vals)))
        return GC_ERR_INVALID;
    if (workspace_bytes < saps_workspace_bytes(n)) return GC_ERR_INVALID;
    if (!aligned16(workspace) || !aligned16(d_count)) return GC_ERR_ALIGN;
    if (capacity > 0 && !aligned16(idx)) return GC_ERR_ALIGN;
    MaskArgs a;
    for (int w = 0; w < W; ++w) {
        if (!models[w] || (capacity > 0 && !vals[w])) return GC_ERR_INVALID;
        if (!aligned16(models[w]) || (capacity > 0 && !aligned16(vals[w]))) return GC_ERR_ALIGN;
        a.models.p[w] = models[w];
        a.vals.p[w] = capacity > 0 ? vals[w] : nullptr;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (cudaMemsetAsync(d_count, 0, sizeof(uint64_t), s) != cudaSuccess) return GC_ERR_CUDA;
        return GC_OK;
    }
    a.n = n;
    a.seed_t = seed_t;
    a.thr = static_cast<uint32_t>(ceil(p * 16777216.0));
    a.W = W;
    a.idx = idx;
    a.capacity = capacity;
    a.d_count = d_count;
    a.counter = static_cast<unsigned long long*>(workspace);
    a.state = reinterpret_cast<uint64_t*>(static_cast<char*>(workspace) + kWsHeader);
    a.ntiles = mask_tiles(n);
    a.d_status = d_status;
    a.group_mask = ws_group_mask(workspace, n);
    a.group_excl = ws_group_excl(workspace, n);
    a.withhold_tile = withhold_tile;
    a.wait_ns = wait_ns;
    // the counter and look-back states must start at zero; the group tables
    // are written in full by the kernel
    if (cudaMemsetAsync(workspace, 0, kWsHeader + sizeof(uint64_t) * static_cast<size_t>(a.ntiles), s) !=
        cudaSuccess)
        return GC_ERR_CUDA;
    return launch_mask(a, s);
}

int saps_mask_compact(int64_t n, double p, uint64_t seed_t, const float* const* models, int W,
                      uint32_t* idx, float* const* vals, int64_t capacity, uint64_t* d_count,
                      void* workspace, size_t workspace_bytes, int* d_status, gc_stream_t stream) {
    return mask_compact_impl(n, p, seed_t, models, W, idx, vals, capacity, d_count, workspace,
                             workspace_bytes, d_status, stream, -1, 1000000000ull);
}

int gc_testing_saps_mask_compact_withhold(int64_t n, double p, uint64_t seed_t,
                                          const float* const* models, int W, uint32_t* idx,
                                          float* const* vals, int64_t capacity, uint64_t* d_count,
                                          void* workspace, size_t workspace_bytes, int* d_status,
                                          int64_t withhold_tile, uint64_t wait_ns, gc_stream_t stream) {
    if (wait_ns == 0 || wait_ns > 1000000000ull) return GC_ERR_INVALID;
    return mask_compact_impl(n, p, seed_t, models, W, idx, vals, capacity, d_count, workspace,
                             workspace_bytes, d_status, stream, withhold_tile, wait_ns);
}

int saps_peer_average(float* const* models, const float* const* vals, const uint32_t* idx,
                      const uint64_t* d_count, const int* pairs, int W, int64_t capacity,
                      gc_stream_t stream) {
    if (W < 2 || W > GC_MAX_WORKERS || (W & 1) || capacity < 0) return GC_ERR_INVALID;
    if (!models || !pairs || !d_count) return GC_ERR_INVALID;
    if (capacity == 0) return GC_OK;
    if (!vals || !idx) return GC_ERR_INVALID;
    AvgArgs a;
    bool seen[GC_MAX_WORKERS] = {false};
    for (int w = 0; w < W; ++w) {
        const int q = pairs[w];
        if (q < 0 || q >= W || seen[q]) return GC_ERR_INVALID;
        seen[q] = true;
        a.pairs[w] = q;
        if (!models[w] || !vals[w]) return GC_ERR_INVALID;
        if (!aligned16(models[w]) || !aligned16(vals[w])) return GC_ERR_ALIGN;
        a.models.p[w] = models[w];
        a.vals.p[w] = vals[w];
    }
    if (!aligned16(idx)) return GC_ERR_ALIGN;
    a.W = W;
    a.idx = idx;
    a.d_count = d_count;
    a.capacity = capacity;
    int grid = grid_for(4);
    if (grid <= 0) return GC_ERR_CUDA;
    const int64_t need = (capacity + kThreads - 1) / kThreads;
    if (need < grid) grid = static_cast<int>(need);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (W <= 16)
        k_saps_peer_average<8><<<grid, kThreads, 0, s>>>(a);
    else
        k_saps_peer_average<0><<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

int saps_average_easgd_step(float* const* models, const float* const* vals, const uint64_t* d_count,
                            const int* pairs, int W, int64_t n, int64_t capacity, float alpha, float beta,
                            float* center, const void* workspace, size_t workspace_bytes,
                            gc_stream_t stream) {
    if (n < 0 || n > 0xFFFFFFFFll || W < 2 || W > GC_MAX_WORKERS || (W & 1) || capacity < 0 ||
        !isfinite(alpha) || !isfinite(beta))
        return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!models || !pairs || !d_count || !center || !workspace || (capacity > 0 && !vals))
        return GC_ERR_INVALID;
    if (workspace_bytes < saps_workspace_bytes(n)) return GC_ERR_INVALID;
    if (!aligned16(center) || !aligned16(workspace)) return GC_ERR_ALIGN;
    FusedArgs a;
    bool seen[GC_MAX_WORKERS] = {false};
    for (int w = 0; w < W; ++w) {
        const int q = pairs[w];
        if (q < 0 || q >= W || seen[q]) return GC_ERR_INVALID;
        seen[q] = true;
    }
    for (int q = 0; q < W / 2; ++q) {
        a.partner[pairs[2 * q]] = pairs[2 * q + 1];
        a.partner[pairs[2 * q + 1]] = pairs[2 * q];
    }
    for (int w = 0; w < W; ++w) {
        if (!models[w] || (capacity > 0 && !vals[w])) return GC_ERR_INVALID;
        if (!aligned16(models[w]) || (capacity > 0 && !aligned16(vals[w]))) return GC_ERR_ALIGN;
        a.models.p[w] = models[w];
        a.vals.p[w] = capacity > 0 ? vals[w] : nullptr;
    }
    a.W = W;
    a.n = n;
    a.alpha = alpha;
    a.beta = beta;
    a.inv_w = static_cast<float>(1.0 / W);
    a.center = center;
    void* ws = const_cast<void*>(workspace);
    a.group_mask = ws_group_mask(ws, n);
    a.group_excl = ws_group_excl(ws, n);
    a.d_count = d_count;
    a.capacity = capacity;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (W <= 16) {
        // 24 times the resident CTAs (2 per SM), each thread a few chunks
        // apart: 0.97-0.99 of the copy peak, against 0.90-0.92 for one
        // resident wave striding over everything and 0.88 for one chunk per
        // thread (whose payload reads then wait on the group tables)
        const int64_t want = ((n >> 2) + kThreads - 1) / kThreads;
        const int64_t cap = static_cast<int64_t>(grid_for(2)) * 24;
        if (cap <= 0) return GC_ERR_CUDA;
        const unsigned grid = static_cast<unsigned>(want < cap ? (want > 0 ? want : 1) : cap);
        if (W <= 4)
            k_saps_average_easgd<4><<<grid, kThreads, 0, s>>>(a);
        else
            k_saps_average_easgd<16><<<grid, kThreads, 0, s>>>(a);
    } else {
        const unsigned grid = static_cast<unsigned>((n + kThreads - 1) / kThreads);
        k_saps_average_easgd_wide<<<grid, kThreads, 0, s>>>(a);
    }
    return launch_status();
}

static int saps_round_impl(int64_t n, double p, uint64_t seed_t, float* const* models, int W, const int* pairs,
                           float alpha, float beta, float* center, uint32_t* idx, float* const* vals,
                           int64_t capacity, uint64_t* d_count, void* workspace, size_t workspace_bytes,
                           int* d_status, gc_stream_t stream, bool force_one_pass) {
    if (n < 0 || n > 0xFFFFFFFFll || W < 2 || W > GC_MAX_WORKERS || (W & 1) || capacity < 0 ||
        !(p > 0.0 && p <= 1.0) || !isfinite(alpha) || !isfinite(beta))
        return GC_ERR_INVALID;
    if (!models || !pairs || !center || !d_count || !d_status || !workspace || (capacity > 0 && (!idx || !vals)))
        return GC_ERR_INVALID;
    if (workspace_bytes < saps_workspace_bytes(n)) return GC_ERR_INVALID;
    if (!aligned16(workspace) || !aligned16(d_count) || !aligned16(center) || (capacity > 0 && !aligned16(idx)))
        return GC_ERR_ALIGN;
    RoundArgs a;
    bool seen[GC_MAX_WORKERS] = {false};
    for (int w = 0; w < W; ++w) {
        const int q = pairs[w];
        if (q < 0 || q >= W || seen[q]) return GC_ERR_INVALID;
        seen[q] = true;
    }
    for (int q = 0; q < W / 2; ++q) {
        a.partner[pairs[2 * q]] = pairs[2 * q + 1];
        a.partner[pairs[2 * q + 1]] = pairs[2 * q];
    }
    for (int w = 0; w < W; ++w) {
        if (!models[w] || (capacity > 0 && !vals[w])) return GC_ERR_INVALID;
        if (!aligned16(models[w]) || (capacity > 0 && !aligned16(vals[w]))) return GC_ERR_ALIGN;
    }
    // The one-pass kernel while a tile's expected masked count (4096 p) stays
    // well inside its stash; otherwise, and for W > 16, the compaction and
    // then the fused pair average + elastic step.
    if (W > 16 || (!force_one_pass && p * kTileElems > 0.75 * kStash)) {
        if (force_one_pass) return GC_ERR_INVALID;
        const int rc = saps_mask_compact(n, p, seed_t, models, W, idx, vals, capacity, d_count, workspace,
                                         workspace_bytes, d_status, stream);
        if (rc != GC_OK) return rc;
        return saps_average_easgd_step(models, vals, d_count, pairs, W, n, capacity, alpha, beta, center,
                                       workspace, workspace_bytes, stream);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) return cudaMemsetAsync(d_count, 0, sizeof(uint64_t), s) == cudaSuccess ? GC_OK : GC_ERR_CUDA;
    MaskArgs& m = a.m;
    for (int w = 0; w < W; ++w) {
        a.models.p[w] = models[w];
        m.models.p[w] = models[w];
        m.vals.p[w] = capacity > 0 ? vals[w] : nullptr;
    }
    m.n = n;
    m.seed_t = seed_t;
    m.thr = static_cast<uint32_t>(ceil(p * 16777216.0));
    m.W = W;
    m.idx = idx;
    m.capacity = capacity;
    m.d_count = d_count;
    m.counter = static_cast<unsigned long long*>(workspace);
    m.state = reinterpret_cast<uint64_t*>(static_cast<char*>(workspace) + kWsHeader);
    m.ntiles = mask_tiles(n);
    m.d_status = d_status;
    a.alpha = alpha;
    a.beta = beta;
    a.inv_w = static_cast<float>(1.0 / W);
    a.center = center;
    if (cudaMemsetAsync(workspace, 0, kWsHeader + sizeof(uint64_t) * static_cast<size_t>(m.ntiles), s) !=
        cudaSuccess)
        return GC_ERR_CUDA;
    const unsigned grid = static_cast<unsigned>(m.ntiles);
    if (W <= 4)
        k_saps_round<4, kRoundThreads><<<grid, kRoundThreads, 0, s>>>(a);
    else
        k_saps_round<16, kRoundThreads><<<grid, kRoundThreads, 0, s>>>(a);
    return launch_status();
}

int saps_round(int64_t n, double p, uint64_t seed_t, float* const* models, int W, const int* pairs,
               float alpha, float beta, float* center, uint32_t* idx, float* const* vals, int64_t capacity,
               uint64_t* d_count, void* workspace, size_t workspace_bytes, int* d_status,
               gc_stream_t stream) {
    return saps_round_impl(n, p, seed_t, models, W, pairs, alpha, beta, center, idx, vals, capacity, d_count,
                           workspace, workspace_bytes, d_status, stream, false);
}

int gc_testing_saps_round_one_pass(int64_t n, double p, uint64_t seed_t, float* const* models, int W,
                                   const int* pairs, float alpha, float beta, float* center, uint32_t* idx,
                                   float* const* vals, int64_t capacity, uint64_t* d_count, void* workspace,
                                   size_t workspace_bytes, int* d_status, gc_stream_t stream) {
    return saps_round_impl(n, p, seed_t, models, W, pairs, alpha, beta, center, idx, vals, capacity, d_count,
                           workspace, workspace_bytes, d_status, stream, true);
}

int easgd_step(float* const* models, int W, int64_t n, float alpha, float beta, float* center,
               gc_stream_t stream) {
    if (n < 0 || W < 1 || W > GC_MAX_WORKERS || !isfinite(alpha) || !isfinite(beta)) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!models || !center) return GC_ERR_INVALID;
    EasgdArgs a;
    for (int w = 0; w < W; ++w) {
        if (!models[w]) return GC_ERR_INVALID;
        if (!aligned16(models[w])) return GC_ERR_ALIGN;
        a.models.p[w] = models[w];
    }
    if (!aligned16(center)) return GC_ERR_ALIGN;
    a.W = W;
    a.n = n;
    a.alpha = alpha;
    a.beta = beta;
    a.inv_w = static_cast<float>(1.0 / W);
    a.center = center;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // one float4 (one element for the wide kernel) per thread, grid covering n
    const int64_t items = W <= 16 ? (n >> 2) + 1 : n;
    const unsigned grid = static_cast<unsigned>((items + kThreads - 1) / kThreads);
    if (W <= 4)
        k_easgd<4><<<grid, kThreads, 0, s>>>(a);
    else if (W <= 16)
        k_easgd<16><<<grid, kThreads, 0, s>>>(a);
    else
        k_easgd_wide<<<grid, kThreads, 0, s>>>(a);
    return launch_status();
}

int saps_pair_average_remote(float* model, const uint32_t* idx, const uint64_t* d_count, const float* mine,
                             const float* peer, int64_t capacity, gc_stream_t stream) {
    if (capacity < 0) return GC_ERR_INVALID;
    if (capacity == 0) return GC_OK;
    if (!model || !idx || !d_count || !mine || !peer) return GC_ERR_INVALID;
    if (!aligned16(model) || !aligned16(idx) || !aligned16(d_count) || !aligned16(mine) || !aligned16(peer))
        return GC_ERR_ALIGN;
    RemoteAvgArgs a{model, idx, d_count, mine, peer, capacity};
    const int64_t want = (capacity + kThreads - 1) / kThreads;
    const int64_t cap_grid = static_cast<int64_t>(grid_for(8));
    const unsigned grid = static_cast<unsigned>(want < cap_grid ? want : (cap_grid > 0 ? cap_grid : 1));
    k_saps_pair_average_remote<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return launch_status();
}

int easgd_step_from_sum(float* model, const float* model_sum, int W, int64_t n, float alpha, float beta,
                        float* center, gc_stream_t stream) {
    if (n < 0 || W < 1 || !isfinite(alpha) || !isfinite(beta)) return GC_ERR_INVALID;
    if (n == 0) return GC_OK;
    if (!model || !model_sum || !center) return GC_ERR_INVALID;
    if (!aligned16(model) || !aligned16(model_sum) || !aligned16(center)) return GC_ERR_ALIGN;
    EasgdSumArgs a{model, model_sum, center, n, alpha, beta, static_cast<float>(1.0 / W)};
    const int64_t items = (n >> 2) + 1;
    const unsigned grid = static_cast<unsigned>((items + kThreads - 1) / kThreads);
    k_easgd_from_sum<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return launch_status();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// saps_mask_compact_noalloc: the same compaction without a caller workspace.
//
// Some callers cannot hand this library a workspace: a plug-in running inside
// a host framework whose device allocator it may not call, a training loop
// whose device memory is planned once up front and may not grow, or code that
// must not risk the implicit device-wide synchronisation that cudaMalloc and
// cudaFree can cause.  For them the look-back scratch (the tile counter and
// one state word per tile) lives in a fixed array in device memory that every
// GPU which loads this library holds until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents; each call clears the part it uses on its own stream before the
// kernel runs.  Two calls whose work overlaps on the GPU (different streams
// without ordering between them) race on the array and give wrong results:
// order them on one stream or with events.
//
// Host code cannot use the array's name as a device address (on the host it
// names a host-side stand-in), so every call looks the address up with
// cudaGetSymbolAddress, with the device current, and passes it to the kernel.
// Looking it up per call keeps no pointer across a context teardown and
// re-creation; the first call on a device may also load the module, so make
// that first call before any stream capture.  The stream must belong to the
// current device: the array and the SM count both come from that device.
// ---------------------------------------------------------------------------

namespace gc {
namespace {

constexpr int64_t kNoAllocMaxN = int64_t(1) << 26;                  // 67,108,864 elements
constexpr int64_t kNoAllocMaxTiles = kNoAllocMaxN / kTileElems;    // 16,384 tiles
constexpr size_t kNoAllocWords = kWsHeader / sizeof(uint64_t) + kNoAllocMaxTiles;

}  // namespace

// 16,392 words = 131,136 bytes of device memory per GPU.
static __device__ __align__(256) unsigned long long g_noalloc_scratch[kNoAllocWords];

namespace {

// The current device's copy of the scratch array, after checking that
// `stream` runs on that device.
int noalloc_scratch_address(cudaStream_t stream, void** out) {
    int dev = -1, sdev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GC_ERR_CUDA;
    }
    if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) {
        cudaGetLastError();
        return GC_ERR_CUDA;
    }
    if (sdev != dev) return GC_ERR_INVALID;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return GC_ERR_CUDA;
    }
    *out = p;
    return GC_OK;
}

}  // namespace
}  // namespace gc

extern "C" int saps_mask_compact_noalloc(int64_t n, double p, uint64_t seed_t,
                                         const float* const* models, int W, uint32_t* idx,
                                         float* const* vals, int64_t capacity, uint64_t* d_count,
                                         int* d_status, gc_stream_t stream) {
    using namespace gc;
    if (n < 0 || n > kNoAllocMaxN || W < 1 || W > GC_MAX_WORKERS || capacity < 0) return GC_ERR_INVALID;
    if (!(p > 0.0 && p <= 1.0)) return GC_ERR_INVALID;
    if (!d_count || !d_status || !models || (capacity > 0 && (!idx || !vals))) return GC_ERR_INVALID;
    if (!aligned16(d_count)) return GC_ERR_ALIGN;
    if (capacity > 0 && !aligned16(idx)) return GC_ERR_ALIGN;
    MaskArgs a;
    for (int w = 0; w < W; ++w) {
        if (!models[w] || (capacity > 0 && !vals[w])) return GC_ERR_INVALID;
        if (!aligned16(models[w]) || (capacity > 0 && !aligned16(vals[w]))) return GC_ERR_ALIGN;
        a.models.p[w] = models[w];
        a.vals.p[w] = capacity > 0 ? vals[w] : nullptr;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) {
        if (cudaMemsetAsync(d_count, 0, sizeof(uint64_t), s) != cudaSuccess) return GC_ERR_CUDA;
        return GC_OK;
    }
    void* scratch = nullptr;
    const int st = noalloc_scratch_address(s, &scratch);
    if (st != GC_OK) return st;
    a.n = n;
    a.seed_t = seed_t;
    a.thr = static_cast<uint32_t>(ceil(p * 16777216.0));
    a.W = W;
    a.idx = idx;
    a.capacity = capacity;
    a.d_count = d_count;
    a.counter = static_cast<unsigned long long*>(scratch);
    a.state = reinterpret_cast<uint64_t*>(static_cast<char*>(scratch) + kWsHeader);
    a.ntiles = mask_tiles(n);
    a.d_status = d_status;
    const size_t used = kWsHeader + sizeof(uint64_t) * static_cast<size_t>(a.ntiles);
    if (cudaMemsetAsync(scratch, 0, used, s) != cudaSuccess) return GC_ERR_CUDA;
    return launch_mask(a, s);
}
