// sample: fused bitmask + temperature + top-k / top-p / min-p keep-threshold +
// Gumbel-max draw (logits-processor, "API" and "Method"; logits-mask-xpu,
// "Method" for top_k == 1).
//
// One thread-block cluster of C CTAs owns one row.  Each CTA pulls its slice
// of the row from HBM into shared memory exactly once with 1-D bulk copies
// (cp.async.bulk, completing on mbarriers) and every later pass reads shared
// memory only.  Cluster-wide exchanges go through distributed shared memory.
//
//  phase A  (every row)  mask + NaN -> -inf (written back in shared memory),
//           per-thread max / lowest argmax, online sum of exp((l - m) / T),
//           and a lower bound tau on the k-th largest logit from the thread
//           maxima (r = ceil(k / warps) per warp: the warps' r-th largest
//           maxima are >= k distinct logits).
//  X1       cluster exchange of (argmax key, m, Z, tau) -> global m, a, Z, tau.
//  greedy   T <= 0 or top_k == 1: token = a.
//  fast     theta = max(tau, min-p cut): every logit >= theta goes into the
//           leader's candidate buffer.  The buffer holds the whole keep set
//           (v* >= theta), so the leader sorts it, resolves v*, and draws.
//  general  when no bound exists or the buffer overflows: cluster radix
//           select (8-bit digits of the order-preserving key) for the k-th
//           largest (counts) and for the top-p boundary (fixed-point masses),
//           then every CTA draws over its own kept tokens and the best score
//           is reduced across the cluster.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_select.cuh"
#include "tsa_host.h"

namespace tsa {

constexpr int kThreads = kSelThreads;
constexpr int kWarps = kSelWarps;
constexpr int kChunks = 4;      // bulk copies (and mbarriers) per CTA slice
constexpr int kMergeCap = 512;  // leader candidate buffer (u64 rank keys)
constexpr int kMaxCluster = 16;
constexpr int kTauMaxK = 32 * kWarps;  // largest k for which tau is formed

// Fixed-point scale of per-token masses in the general path's histograms.
// Masses are <= 1 and rows have < 2^23 tokens, so sums stay below 2^63.
constexpr float kMassScale = 1099511627776.0f;  // 2^40

struct __align__(16) Ctl {
    uint64_t mbar[kChunks];
    // this CTA's contributions, read remotely by the whole cluster
    uint64_t x_argmax;  // rank_key of the CTA max
    float x_z;          // sum exp((l - m_cta) / T) over the CTA's allowed tokens
    float x_tau;        // lower bound on the row's k-th largest logit
    uint64_t x_best;    // rank key of the best perturbed score
    uint32_t cand_count;  // leader only: candidates appended
    uint32_t pad0;
    Scratch sc;  // block reduction scratch
    // gathered from the cluster (slot r = CTA r)
    uint64_t q_key[kMaxCluster];
    float q_z[kMaxCluster];
    float q_tau[kMaxCluster];
    // candidate prefix-mass scan scratch
    double wsum[kWarps];
    uint32_t wlast[kWarps];
    // broadcast slots
    uint64_t g_argmax;
    float g_m, g_z, g_tau, g_vstar;
    uint32_t g_u1;
};

constexpr size_t kUnionBytes =
    (2 * sizeof(Hist) > kMergeCap * sizeof(uint64_t)) ? 2 * sizeof(Hist) : kMergeCap * sizeof(uint64_t);

__device__ unsigned int g_sample_status;

// Mask bits of elements e0 .. e0 + AE - 1 (bit t <-> element e0 + t); bits of
// elements outside [0, 32 W) are 0.  e0 > -AE.
template <int AE>
__device__ __forceinline__ uint32_t mask_bits(const int32_t *mrow, int64_t e0, int64_t W) {
    if (e0 >= 0) {
        const int64_t wi = e0 >> 5;
        const uint32_t s = (uint32_t)(e0 & 31);
        const uint32_t lo = (wi < W) ? (uint32_t)__ldg(mrow + wi) : 0u;
        const uint32_t hi = (s + AE > 32 && wi + 1 < W) ? (uint32_t)__ldg(mrow + wi + 1) : 0u;
        return __funnelshift_r(lo, hi, s);
    }
    return (uint32_t)__ldg(mrow) << (uint32_t)(-e0);
}

template <int DT>
__global__ void __launch_bounds__(kThreads) sample_kernel(SampleArgs a) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint4 *slice = reinterpret_cast<uint4 *>(smem);
    uint8_t *uni = smem + (size_t)(a.max_vec + 2) * 16;
    uint64_t *merge = reinterpret_cast<uint64_t *>(uni);
    Hist *hist = reinterpret_cast<Hist *>(uni);
    Ctl &ctl = *reinterpret_cast<Ctl *>(uni + kUnionBytes);

    const uint32_t C = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const uint32_t row = cluster_id_x();
    const int tid = threadIdx.x;
    const int64_t V = a.V;
    const uint8_t *row_ptr = reinterpret_cast<const uint8_t *>(a.logits) + (size_t)row * a.stride * E::SIZE;
    const int32_t *mrow = a.mask ? a.mask + (size_t)row * a.mstride : nullptr;
    const int64_t W = (V + 31) >> 5;

    const float T = a.temperature ? __ldg(a.temperature + row) : a.temperature_s;
    const int32_t K = a.top_k ? __ldg(a.top_k + row) : a.top_k_s;
    const float P = a.top_p ? __ldg(a.top_p + row) : a.top_p_s;
    const float MP = a.min_p ? __ldg(a.min_p + row) : a.min_p_s;
    const bool greedy = !(T > 0.f) || K == 1;
    const bool k_on = !greedy && K > 1;
    const bool p_on = !greedy && P < 1.f;
    const bool m_on = !greedy && MP > 0.f;
    const bool need_z = p_on;
    const bool need_tau = k_on && K <= kTauMaxK;
    const float invT = greedy ? 1.f : 1.f / T;
    const float c2 = invT * 1.4426950408889634f;  // log2(e) / T

    const RowSlice s = make_slice<AE, E::SIZE>(row_ptr, V, rank, C);

    // ---- set-up: barriers, counters, bulk copies in flight
    if (tid == 0) {
        for (int j = 0; j < kChunks; ++j) mbar_init(&ctl.mbar[j], 1);
        ctl.cand_count = 0;
        mbar_init_fence();
    }
    __syncthreads();
    const int64_t cv = (s.nv + kChunks - 1) / kChunks;  // vectors per chunk
    if (tid == 0) {
        const uint8_t *src = row_ptr + (size_t)(s.head + s.vc0 * AE) * E::SIZE;
        for (int j = 0; j < kChunks; ++j) {
            const int64_t v0 = min((int64_t)j * cv, s.nv), v1 = min((int64_t)(j + 1) * cv, s.nv);
            const uint32_t bytes = v1 > v0 ? (uint32_t)((v1 - v0) * 16) : 0u;
            mbar_arrive_expect_tx(&ctl.mbar[j], bytes);
            if (bytes) bulk_g2s(slice + 1 + v0, src + v0 * 16, bytes, &ctl.mbar[j]);
        }
    }
    // head / tail elements with plain loads
    if (rank == 0 && tid < s.head) {
        const int64_t e = tid;
        const float x = E::load1(row_ptr, e);
        const int64_t j = e - s.base;
        if (E::SIZE == 4) reinterpret_cast<float *>(slice)[j] = x;
        else reinterpret_cast<unsigned short *>(slice)[j] =
            reinterpret_cast<const unsigned short *>(row_ptr)[e];
    }
    if (rank == C - 1 && tid < s.tail) {
        const int64_t e = s.head + s.nvec * AE + tid;
        const int64_t j = e - s.base;
        if (E::SIZE == 4) reinterpret_cast<float *>(slice)[j] = E::load1(row_ptr, e);
        else reinterpret_cast<unsigned short *>(slice)[j] =
            reinterpret_cast<const unsigned short *>(row_ptr)[e];
    }
    __syncthreads();
    cluster_sync();  // every CTA of the cluster is running and initialised

    // ---- phase A
    float mx = -INFINITY, z = 0.f;
    uint32_t mi = 0xFFFFFFFFu;
    for (int j = 0; j < kChunks; ++j) {
        int64_t v0 = 1 + min((int64_t)j * cv, s.nv), v1 = 1 + min((int64_t)(j + 1) * cv, s.nv);
        if (j == 0) v0 = s.vbeg;
        if (j == kChunks - 1) v1 = s.vend;
        mbar_wait_bounded(&ctl.mbar[j], 0, &g_sample_status);  // zero-byte chunks complete at once
        for (int64_t v = v0 + tid; v < v1; v += kThreads) {
            uint4 raw = slice[v];
            float x[AE];
            E::unpack(raw, x);
            const int64_t e0 = s.base + v * AE;
            uint32_t keep = (1u << AE) - 1u;
            if (mrow) keep &= mask_bits<AE>(mrow, e0, W);
            if (e0 < s.lo || e0 + AE > s.hi) {
#pragma unroll
                for (int t = 0; t < AE; ++t)
                    if (e0 + t < s.lo || e0 + t >= s.hi) keep &= ~(1u << t);
            }
#pragma unroll
            for (int t = 0; t < AE; ++t)
                if (x[t] != x[t]) keep &= ~(1u << t);
            if (keep != (1u << AE) - 1u) {
                const uint32_t drop = ~keep & ((1u << AE) - 1u);
#pragma unroll
                for (int t = 0; t < AE; ++t)
                    if (drop & (1u << t)) x[t] = -INFINITY;
                E::store_ninf(raw, drop);
                slice[v] = raw;
            }
            float vmax = x[0];
#pragma unroll
            for (int t = 1; t < AE; ++t) vmax = fmaxf(vmax, x[t]);
            if (need_z && vmax > -INFINITY) {
                if (vmax > mx) z *= exp2f((mx - vmax) * c2);
                const float mref = fmaxf(mx, vmax);
#pragma unroll
                for (int t = 0; t < AE; ++t) z += exp2f((x[t] - mref) * c2);
            }
#pragma unroll
            for (int t = 0; t < AE; ++t)
                if (x[t] > mx) {
                    mx = x[t];
                    mi = (uint32_t)(e0 + t);
                }
        }
    }

    // CTA summaries: argmax key, Z relative to the CTA max, tau
    const uint64_t my_key = (mx > -INFINITY) ? rank_key(mx, mi) : 0ull;
    const uint64_t cta_key = block_max_u64(my_key, ctl.sc);
    const float cta_m = cta_key ? rank_key_value(cta_key) : -INFINITY;
    float cta_z = 0.f;
    if (need_z) {
        const float zt = (mx > -INFINITY) ? z * exp2f((mx - cta_m) * c2) : 0.f;
        cta_z = block_sum_f32(zt, ctl.sc);
    }
    float cta_tau = -INFINITY;
    if (need_tau) {
        // r-th largest thread maximum of each warp (remove the top r-1 first)
        const int r = (K + kWarps - 1) / kWarps;
        uint32_t key = okey(mx);
        uint32_t kth = 0;
        for (int it = 0; it < r; ++it) {
            kth = __reduce_max_sync(0xFFFFFFFFu, key);
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, key == kth);
            if ((tid & 31) == __ffs(hit) - 1) key = 0;
        }
        cta_tau = block_min_f32(okey_value(kth), ctl.sc);
    }
    if (tid == 0) {
        ctl.x_argmax = cta_key;
        ctl.x_z = cta_z;
        ctl.x_tau = cta_tau;
    }
    cluster_sync();  // X1: summaries visible

    // global m, a, Z, tau (same fixed order in every CTA)
    if (tid < (int)C) {
        ctl.q_key[tid] = dsmem_ld_u64(dsmem_addr(&ctl.x_argmax, tid));
        ctl.q_z[tid] = dsmem_ld_f32(dsmem_addr(&ctl.x_z, tid));
        ctl.q_tau[tid] = dsmem_ld_f32(dsmem_addr(&ctl.x_tau, tid));
    }
    __syncthreads();
    if (tid == 0) {
        uint64_t gk = 0;
        float gtau = -INFINITY;
        for (uint32_t r = 0; r < C; ++r) {
            gk = ctl.q_key[r] > gk ? ctl.q_key[r] : gk;
            gtau = fmaxf(gtau, ctl.q_tau[r]);
        }
        const float gm = gk ? rank_key_value(gk) : -INFINITY;
        float gz = 0.f;
        if (need_z)
            for (uint32_t r = 0; r < C; ++r)
                if (ctl.q_key[r]) gz += ctl.q_z[r] * exp2f((rank_key_value(ctl.q_key[r]) - gm) * c2);
        ctl.g_argmax = gk;
        ctl.g_m = gm;
        ctl.g_z = gz;
        ctl.g_tau = gtau;
    }
    __syncthreads();
    const uint64_t gkey = ctl.g_argmax;
    const float m = ctl.g_m;
    const uint32_t amax = gkey ? rank_key_index(gkey) : 0xFFFFFFFFu;
    const bool empty = (gkey == 0) || !(m > -INFINITY);

    if (empty || greedy) {
        if (rank == 0 && tid == 0) {
            a.tokens[row] = empty ? -1 : (int64_t)amax;
            if (a.vstar_out) a.vstar_out[row] = empty ? __int_as_float(0x7FC00000) : m;
        }
        cluster_sync();  // nobody leaves while summaries may still be read
        return;
    }

    // min-p cut: l >= m + T ln(min_p), rounded up to the next float; the
    // argmax class is always kept.
    float v_m = -INFINITY;
    if (m_on) {
        const double cut = (double)m + (double)T * log((double)MP);
        v_m = fminf(__double2float_ru(cut), m);
    }
    float theta = fmaxf(v_m, ctl.g_tau);
    const bool filtered = k_on || p_on || m_on;
    float vstar = -INFINITY;
    bool done = false;

    if (filtered && (theta > -INFINITY || V <= kMergeCap)) {
        // ---- fast path: append every logit >= theta to the leader's buffer
        const uint32_t cnt_addr = dsmem_addr(&ctl.cand_count, 0);
        const uint32_t merge_addr = dsmem_addr(merge, 0);
        const int lane = tid & 31;
        for (int64_t v0 = s.vbeg; v0 < s.vend; v0 += kThreads) {
            const int64_t v = v0 + tid;
            uint32_t hit = 0;
            float x[AE];
            if (v < s.vend) {
                E::unpack(slice[v], x);
#pragma unroll
                for (int t = 0; t < AE; ++t)
                    if (x[t] >= theta && x[t] > -INFINITY) hit |= 1u << t;
            }
            if (!__any_sync(0xFFFFFFFFu, hit != 0)) continue;
            const uint32_t n = __popc(hit);
            uint32_t incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += t;
            }
            const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
            uint32_t basep = 0;
            if (lane == 31) basep = dsmem_atomic_add_u32(cnt_addr, total);
            basep = __shfl_sync(0xFFFFFFFFu, basep, 31);
            uint32_t pos = basep + incl - n;
            const int64_t e0 = s.base + v * AE;
#pragma unroll
            for (int t = 0; t < AE; ++t)
                if (hit & (1u << t)) {
                    if (pos < (uint32_t)kMergeCap)
                        dsmem_st_u64(merge_addr + pos * 8u, rank_key(x[t], (uint32_t)(e0 + t)));
                    ++pos;
                }
        }
        cluster_sync();  // X2: candidates in the leader's buffer
        if (tid == 0) ctl.g_u1 = dsmem_ld_u32(cnt_addr);
        __syncthreads();
        const uint32_t n = ctl.g_u1;
        cluster_arrive();  // X3 arrive: the leader's counter has been read
        if (n <= (uint32_t)kMergeCap) {
            done = true;
            if (rank == 0) {
                // sort the candidates (rank key descending) with a bitonic network
                uint32_t n2 = 1;
                while (n2 < n) n2 <<= 1;
                for (uint32_t i = n + tid; i < n2; i += kThreads) merge[i] = 0ull;
                __syncthreads();
                for (uint32_t kk = 2; kk <= n2; kk <<= 1)
                    for (uint32_t jj = kk >> 1; jj > 0; jj >>= 1) {
                        for (uint32_t i = tid; i < n2; i += kThreads) {
                            const uint32_t p = i ^ jj;
                            if (p > i) {
                                const uint64_t ki = merge[i], kp = merge[p];
                                const bool desc = (i & kk) == 0;
                                if (desc ? (ki < kp) : (ki > kp)) {
                                    merge[i] = kp;
                                    merge[p] = ki;
                                }
                            }
                        }
                        __syncthreads();
                    }
                // k-th largest (the buffer holds every logit >= tau, tau <= v_k)
                float v_k = -INFINITY;
                if (k_on && (uint32_t)K <= n) v_k = rank_key_value(merge[K - 1]);
                float lo = fmaxf(v_k, v_m);
                // top-p: the last position whose exclusive prefix mass < p Z
                float v_p = -INFINITY;
                if (p_on) {
                    const double pz = (double)P * (double)ctl.g_z;
                    // exclusive prefix sums of w in sorted order (double)
                    double acc = 0.0;  // running carry across 256-wide tiles
                    uint32_t last = 0;
                    for (uint32_t t0 = 0; t0 < n; t0 += kThreads) {
                        const uint32_t i = t0 + tid;
                        double w = 0.0;
                        if (i < n) w = (double)exp2f((rank_key_value(merge[i]) - m) * c2);
                        // block exclusive scan of w
                        double incl = w;
                        const int lane = tid & 31, wp = tid >> 5;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const double t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                            if (lane >= o) incl += t;
                        }
                        double *wsum = ctl.wsum;
                        __syncthreads();
                        if (lane == 31) wsum[wp] = incl;
                        __syncthreads();
                        double before = acc;
                        for (int q = 0; q < wp; ++q) before += wsum[q];
                        const double excl = before + incl - w;
                        const bool ok = (i < n) && (i == 0 || excl < pz);
                        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, ok);
                        uint32_t *wlast = ctl.wlast;
                        if (lane == 0) wlast[wp] = bal ? (uint32_t)(t0 + wp * 32 + 31 - __clz(bal)) + 1u : 0u;
                        __syncthreads();
                        for (int q = 0; q < kWarps; ++q) last = max(last, wlast[q]);
                        double tile = 0.0;
                        for (int q = 0; q < kWarps; ++q) tile += wsum[q];
                        acc += tile;
                        __syncthreads();
                    }
                    v_p = rank_key_value(merge[last - 1]);
                    if (!(P > 0.f)) v_p = m;
                }
                vstar = fmaxf(lo, v_p);
                // Gumbel-max over the kept prefix of the sorted candidates
                uint64_t best = 0ull;
                for (uint32_t i = tid; i < n; i += kThreads) {
                    const uint64_t kk2 = merge[i];
                    const float x = rank_key_value(kk2);
                    if (!(x >= vstar)) continue;
                    const uint32_t idx = rank_key_index(kk2);
                    const uint4 blk = token_block(a.seed, a.offset, row, idx >> 2);
                    const float sc = (x - m) * invT + gumbel_of(block_word(blk, idx & 3));
                    const uint64_t key = rank_key(sc, idx);
                    best = key > best ? key : best;
                }
                best = block_max_u64(best, ctl.sc);
                if (tid == 0) {
                    a.tokens[row] = (int64_t)rank_key_index(best);
                    if (a.vstar_out) a.vstar_out[row] = vstar;
                }
            }
        }
        cluster_wait();  // X3 wait
        if (done) return;
        __syncthreads();
    }

    // ---- general path: cluster radix select, then a distributed draw.
    // Each pass fills this CTA's histogram for one 8-bit digit, one cluster
    // barrier publishes it, and every CTA reads all C histograms.  Passes
    // alternate between two histogram buffers, so a CTA clearing buffer X in
    // pass n cannot race a peer still reading X from pass n - 2.
    if (filtered) {
        const int npass = E::NPASS;
        // keys of widened bf16 / f16 logits have constant low bits: 0 for
        // non-negative values, all ones for negative ones
        const uint32_t low_ones = npass >= 4 ? 0u : (0xFFFFFFFFu >> (8 * npass));
        int gpass = 0;
        float lo_v = v_m;
        float v_k = -INFINITY;
        if (k_on) {
            // the k-th largest logit among those >= v_m
            uint32_t prefix = 0;
            uint64_t need = (uint64_t)K;
            bool all_kept = false;
            for (int pass = 0; pass < npass; ++pass, ++gpass) {
                const int shift = 24 - 8 * pass;
                Hist &h = hist[gpass & 1];
                h.cnt[tid] = 0;
                __syncthreads();
                const uint32_t hmask = pass ? (0xFFFFFFFFu << (shift + 8)) : 0u;
                uint32_t run_bin = 0xFFFFFFFFu, run_n = 0;
                for (int64_t v = s.vbeg + tid; v < s.vend; v += kThreads) {
                    float x[AE];
                    E::unpack(slice[v], x);
#pragma unroll
                    for (int t = 0; t < AE; ++t) {
                        if (!(x[t] > -INFINITY) || !(x[t] >= lo_v)) continue;
                        const uint32_t k = okey(x[t]);
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
                const uint32_t D = cluster_digit<false>(h, C, need, 0.0, ctl.sc, above, total);
                if (pass == 0 && total <= (uint64_t)K) {  // top-k keeps every candidate
                    all_kept = true;
                    ++gpass;
                    break;
                }
                prefix |= D << shift;
                need -= above;
            }
            if (!all_kept) v_k = okey_value(prefix | ((prefix & 0x80000000u) ? 0u : low_ones));
        }
        lo_v = fmaxf(lo_v, v_k);
        float v_p = -INFINITY;
        if (p_on) {
            if (!(P > 0.f)) {
                v_p = m;
            } else {
                // top-p boundary among logits >= lo_v: the lowest key whose mass
                // strictly above is below p * Z (fixed-point masses: exact sums)
                const double pz = (double)P * (double)ctl.g_z * (double)kMassScale;
                uint32_t prefix = 0;
                uint64_t mass_above = 0;
                for (int pass = 0; pass < npass; ++pass, ++gpass) {
                    const int shift = 24 - 8 * pass;
                    Hist &h = hist[gpass & 1];
                    h.cnt[tid] = 0;
                    h.mass[tid] = 0ull;
                    __syncthreads();
                    const uint32_t hmask = pass ? (0xFFFFFFFFu << (shift + 8)) : 0u;
                    uint32_t run_bin = 0xFFFFFFFFu, run_n = 0;
                    unsigned long long run_m = 0;
                    for (int64_t v = s.vbeg + tid; v < s.vend; v += kThreads) {
                        float x[AE];
                        E::unpack(slice[v], x);
#pragma unroll
                        for (int t = 0; t < AE; ++t) {
                            if (!(x[t] > -INFINITY) || !(x[t] >= lo_v)) continue;
                            const uint32_t k = okey(x[t]);
                            if ((k & hmask) != (prefix & hmask)) continue;
                            const uint32_t bin = (k >> shift) & 255u;
                            const float w = exp2f((x[t] - m) * c2);
                            const unsigned long long wf = (unsigned long long)(w * kMassScale);
                            if (bin != run_bin) {
                                if (run_n) {
                                    atomicAdd(&h.cnt[run_bin], run_n);
                                    atomicAdd(&h.mass[run_bin], run_m);
                                }
                                run_bin = bin;
                                run_n = 0;
                                run_m = 0;
                            }
                            ++run_n;
                            run_m += wf;
                        }
                    }
                    if (run_n) {
                        atomicAdd(&h.cnt[run_bin], run_n);
                        atomicAdd(&h.mass[run_bin], run_m);
                    }
                    __syncthreads();
                    cluster_sync();
                    uint64_t above = 0, total = 0;
                    const uint32_t D = cluster_digit<true>(h, C, mass_above, pz, ctl.sc, above, total);
                    if (D > 255u) {  // unreachable for p > 0: the top bin has no mass above
                        prefix = okey(m);
                        ++gpass;
                        break;
                    }
                    prefix |= D << shift;
                    mass_above += above;
                }
                v_p = fminf(okey_value(prefix | ((prefix & 0x80000000u) ? 0u : low_ones)), m);
            }
        }
        vstar = fmaxf(lo_v, v_p);
    }

    // ---- distributed Gumbel-max over this CTA's kept tokens
    {
        const uint4 blk_a = token_block(a.seed, a.offset, row, amax >> 2);
        float best_sc = gumbel_of(block_word(blk_a, amax & 3));  // the argmax is always kept
        uint32_t best_i = amax;
        float cut = (best_sc - kGumbelMax) * T + m;  // below this no token can win
        for (int64_t v = s.vbeg + tid; v < s.vend; v += kThreads) {
            float x[AE];
            E::unpack(slice[v], x);
            float vmax = x[0];
#pragma unroll
            for (int t = 1; t < AE; ++t) vmax = fmaxf(vmax, x[t]);
            if (!(vmax >= vstar) || !(vmax >= cut)) continue;
            const int64_t e0 = s.base + v * AE;
            uint32_t q_cached = 0xFFFFFFFFu;
            uint4 blk = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int t = 0; t < AE; ++t) {
                const float xt = x[t];
                if (!(xt > -INFINITY) || !(xt >= vstar)) continue;
                const float ub = (xt - m) * invT + kGumbelMax;
                if (ub < best_sc) continue;
                const uint32_t e = (uint32_t)(e0 + t);
                if ((e >> 2) != q_cached) {
                    q_cached = e >> 2;
                    blk = token_block(a.seed, a.offset, row, q_cached);
                }
                const float sc = (xt - m) * invT + gumbel_of(block_word(blk, e & 3));
                if (sc > best_sc || (sc == best_sc && e < best_i)) {
                    best_sc = sc;
                    best_i = e;
                    cut = (best_sc - kGumbelMax) * T + m;
                }
            }
        }
        const uint64_t bk = block_max_u64(rank_key(best_sc, best_i), ctl.sc);
        if (tid == 0) ctl.x_best = bk;
        cluster_sync();
        if (rank == 0 && tid < (int)C) ctl.q_key[tid] = dsmem_ld_u64(dsmem_addr(&ctl.x_best, tid));
        __syncthreads();
        if (rank == 0 && tid == 0) {
            uint64_t g = 0;
            for (uint32_t r = 0; r < C; ++r) g = ctl.q_key[r] > g ? ctl.q_key[r] : g;
            a.tokens[row] = (int64_t)rank_key_index(g);
            if (a.vstar_out) a.vstar_out[row] = vstar;
        }
        cluster_sync();
    }
}

template __global__ void sample_kernel<0>(SampleArgs);
template __global__ void sample_kernel<1>(SampleArgs);
template __global__ void sample_kernel<2>(SampleArgs);

// ---------------------------------------------------------------- host side
size_t sample_smem_bytes(int64_t max_vec) {
    return (size_t)(max_vec + 2) * 16 + kUnionBytes + sizeof(Ctl);
}

int sample_launch(const SampleArgs &args, int dtype, int cluster, int64_t max_vec, cudaStream_t st) {
    const void *fn = dtype == 0 ? (const void *)sample_kernel<0>
                   : dtype == 1 ? (const void *)sample_kernel<1>
                                : (const void *)sample_kernel<2>;
    const size_t smem = sample_smem_bytes(max_vec);
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
    SampleArgs a = args;
    a.max_vec = max_vec;
    void *params[] = {&a};
    return cudaLaunchKernelExC(&cfg, fn, params) == cudaSuccess ? 0 : -1;
}

unsigned int *sample_status_ptr() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sample_status) != cudaSuccess) return nullptr;
    return reinterpret_cast<unsigned int *>(p);
}

}  // namespace tsa
