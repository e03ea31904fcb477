// topk: the exact k largest logits of each row, sorted by value descending,
// ties to the lower index (lm-head-topk, "API", "Method" and "Correctness").
//
// The pages' design cuts the row into 2,048-entry chunks, takes k candidates
// per chunk by repeated block argmax and merges them.  Here one thread-block
// cluster owns a row held on chip (each CTA's slice pulled from HBM once with
// cp.async.bulk).  For k <= kThreshK, first the threshold path:
//   0. each thread's largest key; each CTA's r-th largest of those (r =
//      ceil(k / C)) is t_c, and t = min over the CTAs' t_c bounds the k-th
//      largest key from below (each CTA holds r distinct elements >= t_c, so
//      the row holds C r >= k elements >= t).  Every element >= t goes to its
//      CTA's list (no histogram, so no shared atomic queues on the few hot
//      bins of a row's top digit), and when the lists hold at most kTopkCap
//      keys in all, step 4 ranks them.
// Otherwise (larger k, or a row with too many keys >= t, such as one of many
// equal values) a cluster-wide radix select on order-preserving keys finds
// the k-th largest value v_k exactly, so no chunk has to offer k candidates:
//   1. 8-bit digit histograms per CTA, merged through distributed shared
//      memory, resolve v_k and how many of its ties are still needed;
//   2. the ties are taken in index order: CTAs hold consecutive index ranges,
//      so lower-ranked CTAs' tie counts give each CTA its share, and an
//      ordered block scan picks the lowest-index ties inside the CTA;
//   3. each CTA keeps its selected (value, index) rank keys (exactly k over
//      the cluster).
//   4. Every CTA copies all the lists' keys through distributed shared memory
//      and ranks its share of them by counting larger keys (keys are distinct:
//      the index is part of them), so the CTAs write the values (exact copies
//      re-read from the row) and indices of ranks < k in parallel, with no
//      sort.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_host.h"
#include "tsa_select.cuh"

namespace tsa {

namespace {
constexpr int kThreads = kSelThreads;
constexpr int kChunks = 4;
constexpr int kMaxCluster = 16;
constexpr int kTopkCap = 2048;  // the largest k, and the keys a CTA's list holds
// the threshold path runs for k up to this (its bound lists a few times k
// keys; larger k take the radix select directly)
constexpr int kThreshK = 256;
static_assert(kThreshK <= kSelThreads, "each CTA's bound is a rank among its threads' maxima");

// The slice's bytes, and at least room for kTopkCap keys.
__host__ __device__ constexpr size_t topk_slice_region(int64_t max_vec) {
    return (size_t)(max_vec + 2) * 16 > (size_t)kTopkCap * 8 ? (size_t)(max_vec + 2) * 16 : (size_t)kTopkCap * 8;
}

struct __align__(16) TopkCtl {
    uint64_t mbar[kChunks];
    uint32_t cand_count;
    uint32_t tc;  // this CTA's bound t_c (threshold path)
    Scratch sc;
    uint32_t q_cnt[kMaxCluster];
    uint32_t q_off[kMaxCluster];
    uint32_t cand_total;
    uint32_t fits;  // threshold path: every list fits its buffer
};
}  // namespace

__device__ unsigned int g_topk_status;

template <int DT>
__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    constexpr int npass = E::NPASS;
    // keys of widened bf16 / f16 values have constant low bits (0 for
    // non-negative values, all ones for negative ones); NaN takes the largest
    // key of that form, so it ranks above +inf
    constexpr uint32_t low_ones = npass >= 4 ? 0u : (0xFFFFFFFFu >> (8 * npass));
    constexpr uint32_t nan_key = 0xFFFFFFFFu & ~low_ones;

    extern __shared__ __align__(128) uint8_t smem[];
    uint4 *slice = reinterpret_cast<uint4 *>(smem);
    // the other CTAs' sorted lists are copied over the slice once it is read
    uint64_t *others = reinterpret_cast<uint64_t *>(smem);
    Hist *hist = reinterpret_cast<Hist *>(smem + topk_slice_region(a.max_vec));
    uint64_t *merge = reinterpret_cast<uint64_t *>(hist + 2);  // this CTA's selected keys
    TopkCtl &ctl = *reinterpret_cast<TopkCtl *>(merge + kTopkCap);

    const uint32_t C = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const uint32_t row = cluster_id_x();
    const int tid = threadIdx.x;
    const int64_t V = a.V;
    const uint32_t K = (uint32_t)a.k;
    const uint8_t *row_ptr = reinterpret_cast<const uint8_t *>(a.logits) + (size_t)row * a.stride * E::SIZE;
    const RowSlice s = make_slice<AE, E::SIZE>(row_ptr, V, rank, C);

    if (tid == 0) {
        for (int j = 0; j < kChunks; ++j) mbar_init(&ctl.mbar[j], 1);
        ctl.cand_count = 0;
        mbar_init_fence();
    }
    __syncthreads();
    const int64_t cv = (s.nv + kChunks - 1) / kChunks;
    if (tid == 0) {
        const uint8_t *src = row_ptr + (size_t)(s.head + s.vc0 * AE) * E::SIZE;
        for (int j = 0; j < kChunks; ++j) {
            const int64_t v0 = min((int64_t)j * cv, s.nv), v1 = min((int64_t)(j + 1) * cv, s.nv);
            const uint32_t bytes = v1 > v0 ? (uint32_t)((v1 - v0) * 16) : 0u;
            mbar_arrive_expect_tx(&ctl.mbar[j], bytes);
            if (bytes) bulk_g2s(slice + 1 + v0, src + v0 * 16, bytes, &ctl.mbar[j]);
        }
    }
    if (rank == 0 && tid < s.head) {
        const int64_t j = tid - s.base;
        if (E::SIZE == 4) reinterpret_cast<uint32_t *>(slice)[j] = reinterpret_cast<const uint32_t *>(row_ptr)[tid];
        else reinterpret_cast<unsigned short *>(slice)[j] = reinterpret_cast<const unsigned short *>(row_ptr)[tid];
    }
    if (rank == C - 1 && tid < s.tail) {
        const int64_t e = s.head + s.nvec * AE + tid;
        const int64_t j = e - s.base;
        if (E::SIZE == 4) reinterpret_cast<uint32_t *>(slice)[j] = reinterpret_cast<const uint32_t *>(row_ptr)[e];
        else reinterpret_cast<unsigned short *>(slice)[j] = reinterpret_cast<const unsigned short *>(row_ptr)[e];
    }
    __syncthreads();
    cluster_sync();
    for (int j = 0; j < kChunks; ++j) mbar_wait_bounded(&ctl.mbar[j], 0, &g_topk_status);
    const int lane = tid & 31;

    // push the set bits of a lane's vector (elements e0 ..) as rank keys onto
    // this CTA's list, one shared atomic per warp; keys past kTopkCap are
    // counted but not stored
    auto push_keys = [&](uint32_t sel, const float (&x)[AE], int64_t e0) {
        const uint32_t n = __popc(sel);
        uint32_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t;
        }
        const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
        uint32_t basep = 0;
        if (lane == 31) basep = atomicAdd(&ctl.cand_count, total);
        basep = __shfl_sync(0xFFFFFFFFu, basep, 31);
        uint32_t pos = basep + incl - n;
#pragma unroll
        for (int t = 0; t < AE; ++t)
            if (sel & (1u << t)) {
                if (pos < (uint32_t)kTopkCap) {
                    const uint32_t k = (x[t] != x[t]) ? nan_key : okey(x[t]);
                    merge[pos] = ((uint64_t)k << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)(e0 + t));
                }
                ++pos;
            }
    };

    // the in-row elements of vector slot v as bits: slots 1 .. nv hold
    // whole vectors of this CTA's range; only the head slot (0, first CTA)
    // and the tail slot (nv + 1, last CTA) can hold elements outside it
    const int nv = (int)s.nv, base32 = (int)s.base, lo32 = (int)s.lo, hi32 = (int)s.hi;
    constexpr uint32_t kAll = (1u << AE) - 1u;
    auto vbits_of = [&](int v) -> uint32_t {
        if (v >= 1 && v <= nv) return kAll;
        const int e0 = base32 + v * AE;
        uint32_t b = 0;
#pragma unroll
        for (int t = 0; t < AE; ++t) b |= (e0 + t >= lo32 && e0 + t < hi32) ? 1u << t : 0u;
        return b;
    };

    // ---- 0. the threshold path (k <= kThreshK)
    bool listed = false;
    if (K <= (uint32_t)kThreshK) {
        uint32_t kmax = 0;  // below every element's key
#pragma unroll 4
        for (int v = s.vbeg + tid; v < s.vend; v += kThreads) {
            float x[AE];
            E::unpack(slice[v], x);
            const uint32_t vb = vbits_of(v);
#pragma unroll
            for (int t = 0; t < AE; ++t) {
                const uint32_t k = (x[t] != x[t]) ? nan_key : okey(x[t]);
                kmax = ((vb >> t) & 1u) && k > kmax ? k : kmax;
            }
        }
        uint32_t *tk = hist[0].cnt;  // the threads' maxima
        tk[tid] = kmax;
        __syncthreads();
        const uint32_t r = (K + C - 1) / C;  // <= kThreshK <= kThreads
        {
            // this thread's rank among the CTA's maxima (equal keys by thread)
            const uint4 *tk4 = reinterpret_cast<const uint4 *>(tk);
            uint32_t rk = 0;
#pragma unroll 8
            for (int j = 0; j < kThreads / 4; ++j) {
                const uint4 o = tk4[j];
                const int jb = 4 * j;
                rk += (o.x > kmax || (o.x == kmax && jb < tid)) ? 1u : 0u;
                rk += (o.y > kmax || (o.y == kmax && jb + 1 < tid)) ? 1u : 0u;
                rk += (o.z > kmax || (o.z == kmax && jb + 2 < tid)) ? 1u : 0u;
                rk += (o.w > kmax || (o.w == kmax && jb + 3 < tid)) ? 1u : 0u;
            }
            if (rk == r - 1u) ctl.tc = kmax;
        }
        cluster_sync();
        uint32_t tmin = 0xFFFFFFFFu;
#pragma unroll
        for (uint32_t c = 0; c < (uint32_t)kMaxCluster; ++c) {
            const uint32_t tcv = c < C ? dsmem_ld_u32(dsmem_addr(&ctl.tc, c)) : 0xFFFFFFFFu;
            tmin = tcv < tmin ? tcv : tmin;
        }
        // every element >= t to this CTA's list
        for (int v0 = s.vbeg; v0 < s.vend; v0 += kThreads) {
            const int v = v0 + tid;
            float x[AE];
            uint32_t sel = 0;
            if (v < s.vend) {
                E::unpack(slice[v], x);
                const uint32_t vb = vbits_of(v);
#pragma unroll
                for (int t = 0; t < AE; ++t) {
                    const uint32_t k = (x[t] != x[t]) ? nan_key : okey(x[t]);
                    sel |= k >= tmin ? 1u << t : 0u;
                }
                sel &= vb;
            }
            if (!__any_sync(0xFFFFFFFFu, sel != 0)) continue;
            push_keys(sel, x, (int64_t)base32 + (int64_t)v * AE);
        }
        cluster_sync();  // every CTA's list and count are final
        if (tid < (int)C) ctl.q_cnt[tid] = dsmem_ld_u32(dsmem_addr(&ctl.cand_count, tid));
        __syncthreads();
        if (tid == 0) {
            uint32_t o = 0;
            bool f = true;
            for (uint32_t c2 = 0; c2 < C; ++c2) {
                o += ctl.q_cnt[c2];
                f = f && ctl.q_cnt[c2] <= (uint32_t)kTopkCap;
            }
            // the ranking step below copies at most kTopkCap keys
            ctl.fits = (f && o <= (uint32_t)kTopkCap && o >= K) ? 1u : 0u;
        }
        __syncthreads();
        listed = ctl.fits != 0u;
        if (!listed) {
            cluster_sync();  // every CTA has read the counts before any list is reset
            if (tid == 0) ctl.cand_count = 0;
            __syncthreads();
        }
    }

    if (!listed) {
    // ---- 1. the k-th largest key
    uint32_t prefix = 0, D = 0;
    uint64_t need = K;
    for (int pass = 0; pass < npass; ++pass) {
        const int shift = 24 - 8 * pass;
        Hist &h = hist[pass & 1];
        h.cnt[tid] = 0;
        __syncthreads();
        const uint32_t hmask = pass ? (0xFFFFFFFFu << (shift + 8)) : 0u;
        uint32_t run_bin = 0xFFFFFFFFu, run_n = 0;
        for (int v = s.vbeg + tid; v < s.vend; v += kThreads) {
            float x[AE];
            E::unpack(slice[v], x);
            const uint32_t vb = vbits_of(v);
#pragma unroll
            for (int t = 0; t < AE; ++t) {
                if (!((vb >> t) & 1u)) continue;
                const uint32_t k = (x[t] != x[t]) ? nan_key : okey(x[t]);
                if ((k & hmask) != (prefix & hmask)) continue;
                const uint32_t bin = (k >> shift) & 255u;
                if (bin != run_bin) {
                    if (run_n) atomicAdd(&h.cnt[run_bin], run_n);
                    run_bin = bin;
                    run_n = 0;
                }
                ++run_n;
            }
        }
        if (run_n) atomicAdd(&h.cnt[run_bin], run_n);
        __syncthreads();
        cluster_sync();
        uint64_t above = 0, total = 0;
        D = cluster_digit<false>(h, C, need, 0.0, ctl.sc, above, total);
        prefix |= D << shift;
        need -= above;
    }
    const uint32_t key_k = prefix | ((prefix & 0x80000000u) ? 0u : low_ones);

    // ---- 2. this CTA's share of the `need` lowest-index ties at key_k
    {
        Hist &h = hist[(npass - 1) & 1];
        if (tid < (int)C) ctl.q_cnt[tid] = dsmem_ld_u32(dsmem_addr(&h.cnt[D], tid));
        __syncthreads();
    }
    uint64_t before = 0;
    for (uint32_t r = 0; r < rank; ++r) before += ctl.q_cnt[r];
    const uint64_t mine = ctl.q_cnt[rank];
    const uint32_t take = need > before ? (uint32_t)min(need - before, mine) : 0u;

    // ---- 3. this CTA's selected rank keys, into its own buffer (any order):
    // every key above key_k, and its share of the ties -- all of them, none,
    // or (in the one CTA where the share ends) the lowest-index `take`, found
    // with an ordered block scan per tile
    if (tid == 0) ctl.cand_count = 0;
    __syncthreads();
    const bool partial = take > 0 && take < mine;  // the same on every thread
    uint32_t tie_seen = 0;  // ties of this CTA in earlier vector tiles
    for (int64_t v0 = s.vbeg; v0 < s.vend; v0 += kThreads) {
        const int64_t v = v0 + tid;
        float x[AE];
        uint32_t gt = 0, eq = 0;
        const int64_t e0 = s.base + v * AE;
        if (v < s.vend) {
            E::unpack(slice[v], x);
            const uint32_t vb = vbits_of((int)v);
#pragma unroll
            for (int t = 0; t < AE; ++t) {
                if (!((vb >> t) & 1u)) continue;
                const uint32_t k = (x[t] != x[t]) ? nan_key : okey(x[t]);
                if (k > key_k) gt |= 1u << t;
                else if (k == key_k) eq |= 1u << t;
            }
        }
        uint32_t sel = gt | (take == mine ? eq : 0u);
        if (partial) {
            uint32_t tile_ties = 0;
            const uint32_t my_tie0 = tie_seen + block_excl_scan_u32(__popc(eq), ctl.sc, tile_ties);
            tie_seen += tile_ties;
            uint32_t jt = my_tie0;
#pragma unroll
            for (int t = 0; t < AE; ++t)
                if (eq & (1u << t)) {
                    if (jt < take) sel |= 1u << t;
                    ++jt;
                }
        }
        if (!__any_sync(0xFFFFFFFFu, sel != 0)) continue;
        push_keys(sel, x, e0);
    }
    __syncthreads();
    }  // !listed

    // ---- 4. place every key at its rank: every CTA copies all the cluster's
    // keys (exactly k, distinct since the index is part of the key) into its
    // own shared memory, then ranks its share of them -- positions
    // [rank k / C, (rank + 1) k / C) of the concatenation -- by counting the
    // larger keys, and writes those tokens at their ranks.
    const uint32_t n_mine = min(ctl.cand_count, (uint32_t)kTopkCap);
    if (!listed) cluster_sync();  // every CTA's keys and count are final (the threshold path synced)
    if (tid < (int)C) ctl.q_cnt[tid] = min(dsmem_ld_u32(dsmem_addr(&ctl.cand_count, tid)), (uint32_t)kTopkCap);
    __syncthreads();
    if (tid == 0) {
        uint32_t o = 0;
        for (uint32_t c2 = 0; c2 < C; ++c2) {
            ctl.q_off[c2] = o;
            o += ctl.q_cnt[c2];
        }
        ctl.cand_total = min(o, (uint32_t)kTopkCap);
    }
    __syncthreads();
    (void)n_mine;
    {
        // position q of the concatenation is key q - q_off[c2] of CTA c2;
        // a thread's copies are independent, so they are all in flight at once
        const uint32_t n_cat = ctl.cand_total;
        constexpr int kPer = kTopkCap / kThreads;
        uint64_t kv[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const uint32_t q = (uint32_t)tid + (uint32_t)(u * kThreads);
            kv[u] = 0ull;
            if (q < n_cat) {
                uint32_t c2 = 0;
                for (uint32_t c3 = 1; c3 < C; ++c3) c2 = q >= ctl.q_off[c3] ? c3 : c2;
                kv[u] = dsmem_ld_u64(dsmem_addr(merge, c2) + (q - ctl.q_off[c2]) * 8u);
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const uint32_t q = (uint32_t)tid + (uint32_t)(u * kThreads);
            if (q < n_cat) others[q] = kv[u];
        }
    }
    __syncthreads();
    cluster_sync();  // no CTA leaves while another still reads its keys
    const uint32_t n_all = ctl.cand_total;
    const uint32_t p0 = (uint32_t)((uint64_t)n_all * rank / C), p1 = (uint32_t)((uint64_t)n_all * (rank + 1) / C);
    // two threads per key, each counting over half of the keys
    const uint32_t half = (n_all + 1) / 2;
    for (uint32_t q = p0 + (uint32_t)(tid >> 1); q < p1; q += kThreads / 2) {
        const uint64_t key = others[q];
        const uint32_t b0 = (tid & 1) ? half : 0u, b1 = (tid & 1) ? n_all : half;
        uint32_t larger = 0;
        for (uint32_t t2 = b0; t2 < b1; ++t2) larger += others[t2] > key ? 1u : 0u;
        larger += __shfl_xor_sync(__activemask(), larger, 1);
        if ((tid & 1) == 0 && larger < K) {
            const uint32_t idx = rank_key_index(key);
            a.indices[(size_t)row * K + larger] = (int64_t)idx;
            a.values[(size_t)row * K + larger] = E::load1(row_ptr, idx);
        }
    }
}

template __global__ void topk_kernel<0>(TopkArgs);
template __global__ void topk_kernel<1>(TopkArgs);
template __global__ void topk_kernel<2>(TopkArgs);

size_t topk_smem_bytes(int64_t max_vec) {
    return topk_slice_region(max_vec) + 2 * sizeof(Hist) + kTopkCap * sizeof(uint64_t) + sizeof(TopkCtl);
}

int topk_launch(const TopkArgs &args, int dtype, int cluster, int64_t max_vec, cudaStream_t st) {
    const void *fn = dtype == 0 ? (const void *)topk_kernel<0>
                   : dtype == 1 ? (const void *)topk_kernel<1>
                                : (const void *)topk_kernel<2>;
    const size_t smem = topk_smem_bytes(max_vec);
    if (prepare_kernel(fn, smem, cluster) != 0) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(args.B * cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    TopkArgs a = args;
    a.max_vec = max_vec;
    void *params[] = {&a};
    return cudaLaunchKernelExC(&cfg, fn, params) == cudaSuccess ? 0 : -1;
}

unsigned int *topk_status_ptr() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_status) != cudaSuccess) return nullptr;
    return reinterpret_cast<unsigned int *>(p);
}

}  // namespace tsa
