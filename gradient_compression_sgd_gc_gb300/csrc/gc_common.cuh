// gc_common.cuh -- device helpers shared by the sm_103a kernels of
// libgc_gb300.so: cache-hinted 128-bit loads/stores, the counter-based hash,
// launch geometry and host-side argument checks.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <math.h>

#include "../../include/gc_gb300.h"

namespace gc {

// ---------------------------------------------------------------- launch

constexpr int kThreads = 256;          // threads per CTA for the streaming kernels
constexpr int kWarpsPerBlock = kThreads / 32;

// Persistent-grid size: `per_sm` CTAs on every SM of the current device.
inline int grid_for(int per_sm) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms * per_sm;
}

// Blocks of kThreads threads for one warp per tile.
inline unsigned blocks_for_tiles(int64_t tiles) {
    return static_cast<unsigned>((tiles + kWarpsPerBlock - 1) / kWarpsPerBlock);
}

// Buckets per CTA for a decode that gives each thread one bucket (or part of
// one), so that an SM's time is its bucket count: W streams of nb buckets, at
// most maxb buckets a CTA, `slots` CTAs resident at once (SMs x CTAs per SM).
// A grid of maxb-bucket CTAs leaves a few SMs one CTA more than the rest, or
// SMs idle; instead, the fewest waves of `slots` CTAs that hold the buckets,
// and the buckets spread evenly over those CTAs.  The grid is then
// ceil(nb / result) CTAs per stream.  nb, W, slots, maxb >= 1.
inline int64_t even_buckets_per_cta(int64_t nb, int64_t W, int64_t slots, int64_t maxb) {
    int64_t waves = (W * nb + slots * maxb - 1) / (slots * maxb);
    if (waves < 1) waves = 1;
    for (;; ++waves) {
        const int64_t per_stream = slots * waves / W;
        if (per_stream < 1) continue;
        const int64_t b = (nb + per_stream - 1) / per_stream;
        if (b <= maxb) return b;
    }
}

inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? GC_OK : GC_ERR_CUDA;
}

// Launches `kernel` (kThreads threads per CTA, no dynamic shared memory) on
// as many CTAs as are resident on the current device at once, at most
// `want`: the kernel strides over its work.
template <typename Args>
int launch_persistent(void (*kernel)(Args), int64_t want, cudaStream_t s, const Args& a) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess)
        return GC_ERR_CUDA;
    const int64_t resident = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    const int64_t grid = want < resident ? (want > 0 ? want : 1) : resident;
    kernel<<<static_cast<unsigned>(grid), kThreads, 0, s>>>(a);
    return launch_status();
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool finite_pos(float x) { return isfinite(x) && x > 0.0f; }

// Kernel-parameter pointer tables (copied by value into the launch).
template <typename T>
struct PtrTable {
    T p[GC_MAX_WORKERS];
};

// ---------------------------------------------------------------- memory
// Plain C++ intrinsics (not volatile asm) so that the compiler can hoist
// independent loads above earlier stores; buffers are __restrict__ where the
// kernels rely on that.

// Streaming 128-bit read of data used once (evict-first, "cache streaming").
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}

// 128-bit read of data the same thread later overwrites (coherent path).
__device__ __forceinline__ float4 ld_f4(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}

// Streaming 128-bit store (evict-first).
__device__ __forceinline__ void st_stream_f4(float* p, float4 v) {
    __stcs(reinterpret_cast<float4*>(p), v);
}

// ---------------------------------------------------------------- hash

// Top 24 bits of the SplitMix64 output of x (Steele, Lea, Flood 2014).  The
// generator's last step z ^ (z >> 31) leaves bits 40..63 unchanged, so it is
// skipped.
__device__ __forceinline__ uint32_t splitmix64_top24(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return static_cast<uint32_t>(z >> 40);
}

__host__ __device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// ---------------------------------------------------------------- look-back

// Decoupled look-back (Merrill and Garland, "Single-pass Parallel Prefix
// Scan with Decoupled Look-back", 2016) over 64-bit state words, one per
// tile: the flag in the top two bits (1: the tile's aggregate, 2: its
// inclusive prefix), the value below.  A state word carries its own value and
// no other data is published through it, so relaxed single-copy-atomic
// 64-bit accesses at GPU scope are enough (no acquire/release fences).
constexpr uint64_t kFlagAgg = 1ull << 62;
constexpr uint64_t kFlagPrefix = 2ull << 62;
constexpr uint64_t kValueMask = (1ull << 62) - 1;

__device__ __forceinline__ uint64_t ld_state(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_state(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Exclusive prefix of tile `tile` (> 0), by one warp: walks back over the
// predecessors' states 32 at a time (one coalesced 256-byte read) until it
// meets an inclusive prefix, summing the aggregates on the way.  A pending
// predecessor is polled again (after `backoff_ns` of sleep, 0: at once);
// every wait is bounded: after wait_ns the predecessors still pending count
// as zero and timed_out is set.  Every lane returns the prefix.
__device__ __forceinline__ uint64_t lookback_exclusive(const uint64_t* state, int64_t tile, int lane,
                                                       uint64_t wait_ns, unsigned backoff_ns, bool& timed_out) {
    uint64_t excl = 0;
    int64_t end = tile - 1;
    const uint64_t t0 = global_ns();
    while (true) {
        const int64_t j = end - lane;
        uint64_t st = j >= 0 ? ld_state(state + j) : kFlagPrefix;
        while (true) {
            const bool pending = (st >> 62) == 0;
            if (!__any_sync(0xffffffffu, pending)) break;
            // lane 0's clock decides, so the whole warp leaves together
            const bool expired = __shfl_sync(0xffffffffu, global_ns() - t0 > wait_ns, 0);
            if (expired) {
                timed_out = true;
                if (pending) st = kFlagAgg;   // unknown predecessor counts as 0
                break;
            }
            if (backoff_ns) __nanosleep(backoff_ns);
            if (pending) st = ld_state(state + j);
        }
        const unsigned prefix_lanes = __ballot_sync(0xffffffffu, (st >> 62) == 2);
        const int last = prefix_lanes ? __ffs(prefix_lanes) - 1 : 31;
        uint64_t v = lane <= last ? (st & kValueMask) : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        excl += v;
        if (prefix_lanes) break;
        end -= 32;
    }
    return excl;
}

// bf16 bit pattern -> fp32 (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace gc
