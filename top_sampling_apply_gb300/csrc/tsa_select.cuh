// Block- and cluster-level reductions and the cluster radix-select digit step
// shared by the sample and top-k kernels.  Blocks have kSelThreads = 256
// threads, one per 8-bit digit bin.
#pragma once

#include "tsa_device.cuh"

namespace tsa {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

struct Hist {  // one 8-bit digit histogram: token counts and fixed-point masses
    uint32_t cnt[256];
    unsigned long long mass[256];
};

// Barrier policies for the block helpers below: the whole CTA, or a named
// barrier over the first N threads (the consumer warps of a kernel whose
// remaining warps do other work).
struct BlockSync {
    __device__ static __forceinline__ void sync() { __syncthreads(); }
};
template <int ID, int N>
struct NamedSync {
    __device__ static __forceinline__ void sync() { asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory"); }
};

struct Scratch {  // per-CTA reduction scratch
    uint64_t r64[kSelWarps];
    float rf[kSelWarps];
    uint32_t u0;
    uint32_t u1;
    uint64_t above;
};

template <class Sync = BlockSync>
__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, Scratch &sc) {
    v = warp_max_u64(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    Sync::sync();
    if (l == 0) sc.r64[w] = v;
    Sync::sync();
    uint64_t r = sc.r64[0];
#pragma unroll
    for (int i = 1; i < kSelWarps; ++i) r = sc.r64[i] > r ? sc.r64[i] : r;
    return r;
}
// Sum in a fixed order (warp tree, then warps in index order): deterministic.
template <class Sync = BlockSync>
__device__ __forceinline__ float block_sum_f32(float v, Scratch &sc) {
    v = warp_sum_f32(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    Sync::sync();
    if (l == 0) sc.rf[w] = v;
    Sync::sync();
    float r = 0.f;
#pragma unroll
    for (int i = 0; i < kSelWarps; ++i) r += sc.rf[i];
    return r;
}
template <class Sync = BlockSync>
__device__ __forceinline__ float block_min_f32(float v, Scratch &sc) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    Sync::sync();
    if (l == 0) sc.rf[w] = v;
    Sync::sync();
    float r = sc.rf[0];
#pragma unroll
    for (int i = 1; i < kSelWarps; ++i) r = fminf(r, sc.rf[i]);
    return r;
}
// Exclusive prefix (in thread order) of a per-thread count; `total` gets the sum.
template <class Sync = BlockSync>
__device__ __forceinline__ uint32_t block_excl_scan_u32(uint32_t v, Scratch &sc, uint32_t &total) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (l >= o) incl += t;
    }
    Sync::sync();
    if (l == 31) sc.r64[w] = incl;
    Sync::sync();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int i = 0; i < kSelWarps; ++i) {
        if (i < w) before += (uint32_t)sc.r64[i];
        all += (uint32_t)sc.r64[i];
    }
    total = all;
    return before + incl - v;
}

// One 8-bit digit of a cluster-wide radix select.  Every CTA has filled its
// own histogram `mine` and passed a cluster barrier; each CTA then reads all
// C histograms through distributed shared memory and reaches the same
// decision.
//   count select (MASS = false): the digit D holding the `base`-th largest key
//     (base counts from 1 within the current prefix); `above` = keys in
//     digits above D.
//   mass select (MASS = true): the lowest non-empty digit D whose mass
//     strictly above (base + digits above D) is still below `pz`; `above` =
//     mass in digits above D.  D = 0xFFFFFFFF if there is none.
// `total` receives the count (or mass) over all digits.
template <bool MASS>
__device__ __forceinline__ uint32_t cluster_digit(Hist &mine, uint32_t C, uint64_t base, double pz,
                                                  Scratch &sc, uint64_t &above, uint64_t &total) {
    const int d = threadIdx.x;
    uint32_t cnt = 0;
    unsigned long long mass = 0;
    // every CTA's entry requested before any is summed (a rolled loop would
    // wait out one remote round trip per CTA)
    constexpr uint32_t kMaxC = 16;  // the largest cluster the callers launch
    uint32_t cv[kMaxC];
    unsigned long long mv[kMaxC];
#pragma unroll
    for (uint32_t r = 0; r < kMaxC; ++r) {
        cv[r] = r < C ? dsmem_ld_u32(dsmem_addr(&mine.cnt[d], r)) : 0u;
        if (MASS) mv[r] = r < C ? dsmem_ld_u64(dsmem_addr(&mine.mass[d], r)) : 0ull;
    }
#pragma unroll
    for (uint32_t r = 0; r < kMaxC; ++r) {
        cnt += cv[r];
        if (MASS) mass += mv[r];
    }
    const uint64_t val = MASS ? (uint64_t)mass : (uint64_t)cnt;
    const int w = d >> 5, l = d & 31;
    uint64_t incl = val;  // suffix within the warp: lanes l .. 31
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (l + o < 32) incl += t;
    }
    __syncthreads();
    if (l == 0) sc.r64[w] = incl;
    __syncthreads();
    uint64_t later = 0, all = 0;
#pragma unroll
    for (int i = 0; i < kSelWarps; ++i) {
        all += sc.r64[i];
        if (i > w) later += sc.r64[i];
    }
    total = all;
    const uint64_t excl = incl - val + later;  // strictly above digit d
    __syncthreads();
    if (d == 0) sc.u0 = 0xFFFFFFFFu;
    __syncthreads();
    if (!MASS) {
        if (cnt > 0 && excl < base && base <= excl + cnt) sc.u0 = (uint32_t)d;
    } else {
        if (cnt > 0 && (double)(base + excl) < pz) atomicMin(&sc.u0, (uint32_t)d);
    }
    __syncthreads();
    const uint32_t D = sc.u0;
    if (D < 256u && d == (int)D) sc.above = excl;
    __syncthreads();
    above = (D < 256u) ? sc.above : 0ull;
    __syncthreads();
    return D;
}

}  // namespace tsa
