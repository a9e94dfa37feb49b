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

// bf16 bit pattern -> fp32 (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace gc
