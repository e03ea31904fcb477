// Device-side building blocks shared by the selection kernels (sm_103a):
// order-preserving float keys, the Philox4x32-10 stream and Gumbel transform,
// element unpacking, and inline-PTX wrappers for mbarriers, 1-D bulk copies
// (global -> shared), cluster barriers and distributed shared memory.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tsa {

// ---------------------------------------------------------------- constants
constexpr uint32_t kStatusTimeout = 1u;          // device status bit: a bounded wait ran out
constexpr unsigned long long kWaitLimitNs = 500ull * 1000ull * 1000ull;  // 0.5 s

// ---------------------------------------------------------------- float keys
// Monotone map float -> uint32 (larger float -> larger key).  -0.0 maps to the
// key of +0.0 so that the two tie and the index decides.
__device__ __forceinline__ uint32_t okey(float x) {
    uint32_t u = __float_as_uint(x);
    u = (u == 0x80000000u) ? 0u : u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float okey_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// Composite ranking key: value descending, then index ascending, as one u64
// where the larger key ranks first.
__device__ __forceinline__ uint64_t rank_key(float x, uint32_t idx) {
    return ((uint64_t)okey(x) << 32) | (uint64_t)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t rank_key_index(uint64_t k) {
    return 0xFFFFFFFFu - (uint32_t)k;
}
__device__ __forceinline__ float rank_key_value(uint64_t k) {
    return okey_value((uint32_t)(k >> 32));
}

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies with the key advanced by the Weyl constants.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t pa = (uint64_t)0xD2511F53u * c.x;  // one wide multiply each
        const uint64_t pd = (uint64_t)0xCD9E8D57u * c.z;
        c = make_uint4((uint32_t)(pd >> 32) ^ c.y ^ k0, (uint32_t)pd, (uint32_t)(pa >> 32) ^ c.w ^ k1,
                       (uint32_t)pa);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// The block of four words for tokens 4q .. 4q+3 of row `row`.
__device__ __forceinline__ uint4 token_block(uint64_t seed, uint64_t offset, uint32_t row,
                                             uint32_t q) {
    return philox4x32_10(make_uint4(q, row, (uint32_t)offset, (uint32_t)(offset >> 32)),
                         (uint32_t)seed, (uint32_t)(seed >> 32));
}
__device__ __forceinline__ uint32_t block_word(uint4 blk, uint32_t j) {
    return j == 0 ? blk.x : j == 1 ? blk.y : j == 2 ? blk.z : blk.w;
}

// Standard Gumbel variate from a 32-bit word: u = (2 (x >> 9) + 1) 2^-24 on
// the odd lattice (never 0 or 1, exact in fp32), E = -ln u computed from the
// exact 1 - u when u >= 1/2, G = -ln E.  Uses CUDA's logf / log1pf.
__device__ __forceinline__ float gumbel_of(uint32_t x) {
    const float u = (float)(2u * (x >> 9) + 1u) * 0x1p-24f;
    const float e = (u < 0.5f) ? -logf(u) : -log1pf(-(1.0f - u));
    return -logf(e);
}
// Upper bound of gumbel_of over all words (G at u = 1 - 2^-24 is 16.6355),
// with margin, used only to skip tokens that cannot win.
constexpr float kGumbelMax = 16.64f;

// ---------------------------------------------------------------- elements
template <int DT> struct Elem;
template <> struct Elem<0> {  // f32
    static constexpr int AE = 4;  // elements per 16-byte vector
    static constexpr int SIZE = 4;
    static constexpr int NPASS = 4;  // 8-bit radix passes that resolve a key
    __device__ static __forceinline__ void unpack(const uint4 &v, float *x) {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
    __device__ static __forceinline__ float load1(const void *p, int64_t i) {
        return __ldg(reinterpret_cast<const float *>(p) + i);
    }
    __device__ static __forceinline__ void store_ninf(uint4 &v, uint32_t drop) {
        if (drop & 1u) v.x = 0xFF800000u;
        if (drop & 2u) v.y = 0xFF800000u;
        if (drop & 4u) v.z = 0xFF800000u;
        if (drop & 8u) v.w = 0xFF800000u;
    }
};
template <> struct Elem<2> {  // bf16
    static constexpr int AE = 8;
    static constexpr int SIZE = 2;
    static constexpr int NPASS = 2;
    __device__ static __forceinline__ void unpack(const uint4 &v, float *x) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[2 * j] = __uint_as_float(w[j] << 16);
            x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
    __device__ static __forceinline__ float load1(const void *p, int64_t i) {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
        return __uint_as_float((uint32_t)h << 16);
    }
    __device__ static __forceinline__ void store_ninf(uint4 &v, uint32_t drop) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (drop & (1u << (2 * j))) w[j] = (w[j] & 0xFFFF0000u) | 0xFF80u;
            if (drop & (2u << (2 * j))) w[j] = (w[j] & 0x0000FFFFu) | 0xFF800000u;
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Elem<1> {  // f16
    static constexpr int AE = 8;
    static constexpr int SIZE = 2;
    static constexpr int NPASS = 3;  // widened f16 keys have 13 trailing zero bits
    __device__ static __forceinline__ float h2f(uint32_t h) {
        return __half2float(__ushort_as_half((unsigned short)h));
    }
    __device__ static __forceinline__ void unpack(const uint4 &v, float *x) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[2 * j] = h2f(w[j] & 0xFFFFu);
            x[2 * j + 1] = h2f(w[j] >> 16);
        }
    }
    __device__ static __forceinline__ float load1(const void *p, int64_t i) {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
        return h2f(h);
    }
    __device__ static __forceinline__ void store_ninf(uint4 &v, uint32_t drop) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (drop & (1u << (2 * j))) w[j] = (w[j] & 0xFFFF0000u) | 0xFC00u;
            if (drop & (2u << (2 * j))) w[j] = (w[j] & 0x0000FFFFu) | 0xFC000000u;
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Every thread of every CTA in the cluster must execute these (aligned forms).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
    cluster_arrive();
    cluster_wait();
}
// The shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t dsmem_ld_u64(uint32_t a) {
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t a) {
    return __uint_as_float(dsmem_ld_u32(a));
}
__device__ __forceinline__ void dsmem_st_u64(uint32_t a, uint64_t v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t dsmem_atomic_add_u32(uint32_t a, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`; on
// give-up the status flag is raised and false returned.  Never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned int *status,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 4-byte asynchronous copy global -> shared (cp.async), grouped per thread.
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// 2^x with the SFU approximation (ex2.approx.ftz.f32: about 2 ulp).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: let the next kernel on the stream start its
// prologue early / wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- warp helpers
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
    // two 32-bit warp reductions: the largest high word, then the largest
    // low word among the lanes that hold it
    const uint32_t hi = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(v >> 32));
    const uint32_t lo = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(v >> 32) == hi ? (uint32_t)v : 0u);
    return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// ---------------------------------------------------------------- row slicing
// A row of V elements is split into a misaligned head (< AE elements up to the
// first 16-byte boundary), nvec 16-byte vectors, and a tail (< AE elements).
// CTA c of a C-CTA cluster owns vectors [floor(c nvec / C), floor((c+1) nvec / C))
// plus the head (c == 0) and the tail (c == C-1).  In shared memory the
// CTA's vectors sit at vector slots 1 .. nv, the head in slot 0 and the tail
// in slot nv + 1, so that element e lives at smem element e - base.
struct RowSlice {
    int64_t head, nvec, tail;
    int64_t vc0, nv;       // first aligned vector and count owned by this CTA
    int64_t base;          // global element index of smem element 0
    int64_t lo, hi;        // global element range owned by this CTA
    int vbeg, vend;        // smem vector slots holding data: [vbeg, vend)
};

template <int AE, int SIZE>
__device__ __forceinline__ RowSlice make_slice(const void *row_ptr, int64_t V, uint32_t c, uint32_t C) {
    RowSlice s;
    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(row_ptr) & 15u) / SIZE;
    s.head = (AE - (int64_t)mis) % AE;
    if (s.head >= V) {
        s.head = V;
        s.nvec = 0;
        s.tail = 0;
    } else {
        s.nvec = (V - s.head) / AE;
        s.tail = V - s.head - s.nvec * AE;
    }
    s.vc0 = (int64_t)c * s.nvec / C;
    const int64_t vc1 = (int64_t)(c + 1) * s.nvec / C;
    s.nv = vc1 - s.vc0;
    s.base = s.head + s.vc0 * AE - AE;
    s.lo = (c == 0) ? 0 : s.head + s.vc0 * AE;
    s.hi = (c == C - 1) ? V : s.head + vc1 * AE;
    s.vbeg = (c == 0 && s.head > 0) ? 0 : 1;
    s.vend = (int)((c == C - 1 && s.tail > 0) ? s.nv + 2 : s.nv + 1);
    return s;
}

// The same split in 32-bit arithmetic (rows < 2^31 elements, < 2^26 vectors).
struct Slice32 {
    int32_t head, nvec, tail, vc0, nv, base, lo, hi, vbeg, vend;
};
template <int AE, int SIZE>
__device__ __forceinline__ Slice32 make_slice32(const void *row_ptr, int32_t V, uint32_t c, uint32_t C) {
    Slice32 s;
    const int32_t mis = (int32_t)(reinterpret_cast<uintptr_t>(row_ptr) & 15u) / SIZE;
    s.head = (AE - mis) % AE;
    if (s.head >= V) {
        s.head = V;
        s.nvec = 0;
        s.tail = 0;
    } else {
        s.nvec = (V - s.head) / AE;
        s.tail = V - s.head - s.nvec * AE;
    }
    s.vc0 = (int32_t)((c * (uint32_t)s.nvec) / C);
    const int32_t vc1 = (int32_t)(((c + 1) * (uint32_t)s.nvec) / C);
    s.nv = vc1 - s.vc0;
    s.base = s.head + s.vc0 * AE - AE;
    s.lo = (c == 0) ? 0 : s.head + s.vc0 * AE;
    s.hi = (c == C - 1) ? V : s.head + vc1 * AE;
    s.vbeg = (c == 0 && s.head > 0) ? 0 : 1;
    s.vend = (c == C - 1 && s.tail > 0) ? s.nv + 2 : s.nv + 1;
    return s;
}

}  // namespace tsa
