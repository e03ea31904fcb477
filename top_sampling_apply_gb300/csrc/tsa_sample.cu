// sample: fused bitmask + temperature + top-k / top-p / min-p keep-threshold +
// Gumbel-max draw (logits-processor, "API" and "Method"; logits-mask-xpu,
// "Method" for top_k == 1).
//
// Two kernels on the caller's stream; the second is launched with
// programmatic dependent launch so it is scheduled while the first drains.
//
// slice kernel -- a row is cut into S slices of at most ~32 KB.  A persistent
//   grid of CTAs streams (row, slice) work items, double-buffered in shared
//   memory: a slice comes from HBM exactly once by a 1-D bulk copy
//   (cp.async.bulk onto an mbarrier) and its mask words by cp.async, so the
//   next item's copy is in flight while the current one is processed.  CTAs
//   never wait for each other.  Per item (the mask bits are applied to each
//   16-byte vector as it is read; NaN is never a maximum or a candidate):
//     slice max and lowest argmax,
//     sum of exp((l - m_s) / T) relative to the slice max, and a lower bound
//     on the row's k-th largest logit from the thread maxima (each warp's
//     r-th largest maximum, r = ceil(k / warps): the warps' top-r maxima are
//     k distinct logits >= the bound).  With a bound theta_s (that bound, or
//     the min-p cut at the slice max, which is below the row's cut) every
//     logit >= theta_s is published as a candidate.  Unfiltered rows draw
//     the slice's Gumbel-max winner instead.  A 32-byte summary per item
//     goes to the workspace.
// merge kernel -- one CTA per row: global max, argmax and
//   Z = sum_s z_s exp((m_s - m) / T) (slice order), theta = max of the slice
//   bounds.  Greedy: the argmax.  Unfiltered: the best slice winner.
//   Filtered: the candidates >= theta hold every token of the keep set and
//   every logit above them, so the k-th value, the top-p prefix mass and the
//   min-p cut are exact on them once sorted; a Gumbel-max draw over the kept
//   candidates gives the token.  Rows with no bound, or whose candidates
//   overflow, take the general path: the CTA re-reads the row (from L2) and
//   runs an exact radix select (8-bit digits of the order-preserving key:
//   counts for top-k, fixed-point masses for top-p) and the draw.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_host.h"
#include "tsa_select.cuh"
#include "tsa_sample_common.cuh"

namespace tsa {

using namespace sample_detail;

namespace {
constexpr int kTauMaxK = 32 * kWarps;  // largest k for which a thread-maximum bound is formed
constexpr int kMergeCap = 4096;        // candidates the merge can hold (a power of two)
static_assert(kMergeCap * 8 >= (int)sizeof(GHist), "the general path's histograms reuse the candidate buffer");
constexpr int kSliceCap = 512;         // candidates a slice may publish
constexpr int kMaxSlices = 64;
constexpr uint32_t kNoCandidates = 0xFFFFFFFFu;  // slice published no candidate list

struct __align__(16) SliceSumm {  // 32 bytes per (row, slice) in the workspace
    uint64_t argmax_key;  // rank key of the slice max; 0 when the slice has no allowed token
    float z;              // sum exp((l - m_s) / T) over the slice's allowed tokens
    float tau;            // lower bound on the row's k-th largest logit, or -inf
    uint32_t ncand;       // candidates published (may exceed the cap) or kNoCandidates
    uint32_t best_idx;    // unfiltered rows: the slice's Gumbel-max winner
    float best_x;
    uint32_t pad;
};

struct __align__(16) SliceCtl {
    uint64_t mbar[2];
    Scratch sc;
    int32_t vb[kMaxSlices + 1];  // first vector of each slice (rows aligned like row 0)
    int32_t g_head, g_nvec, g_tail;
    // per-warp summaries, double-buffered by item parity
    uint64_t w_key[2][kWarps];
    uint64_t w_best[2][kWarps];
    float w_z[2][kWarps];
    float w_tau[2][kWarps];
    uint32_t n, nq;
};

struct __align__(16) MergeCtl {
    SelCtl sel;
    uint32_t n, pad;
    uint64_t wk2[2], wb2[2];
    uint32_t wt2[2], wf2[2];
    float wz2[2];
    uint64_t q_key[kMaxSlices];
    uint32_t q_n[kMaxSlices];
    uint64_t g_key, g_best;
    float g_z, g_tau;
    uint32_t g_flags;
};

__host__ __device__ constexpr size_t round16(size_t x) { return (x + 15) & ~(size_t)15; }
__host__ __device__ inline size_t slice_bytes(int64_t max_vec) { return (size_t)(max_vec + 2) * 16; }
__host__ __device__ inline size_t mask_bytes(int64_t max_words) { return round16((size_t)(max_words + 2) * 4); }
__host__ __device__ inline size_t queue_bytes(int64_t max_vec) { return round16((size_t)(max_vec + 2) * 2); }

// Per-thread running max, lowest argmax and sum of 2^((l - max) c2).
struct Acc {
    float mx;
    uint32_t mi;
    float z;
};

}  // namespace

__device__ unsigned int g_sample_status;

// Workspace: [B][S] slice summaries, then [B][S][kSliceCap] candidate rank keys.
size_t sample_workspace_layout(int64_t B, int S, size_t *summ_off, size_t *cand_off) {
    const size_t summ = (size_t)B * S * sizeof(SliceSumm);
    *summ_off = 0;
    *cand_off = (summ + 255) & ~(size_t)255;
    return *cand_off + (size_t)B * S * kSliceCap * 8;
}

// ============================================================== slice kernel
template <int DT, int NBUF>
__global__ void __launch_bounds__(kThreads, 3) sample_slice_kernel(SampleArgs a) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    constexpr uint32_t kFull = (1u << AE) - 1u;
    extern __shared__ __align__(128) uint8_t smem[];
    const size_t sb = slice_bytes(a.max_vec), mb = mask_bytes(a.max_words);
    uint8_t *mask_base = smem + NBUF * sb;
    uint16_t *queue = reinterpret_cast<uint16_t *>(mask_base + NBUF * mb);
    // per vector: the top 16 bits of the order key of its (masked) maximum,
    // rounded up, so `vkey[v] >= key16(t)` holds whenever the vector has a
    // logit >= t (a conservative filter for the later passes)
    uint16_t *vkey = reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(queue) + queue_bytes(a.max_vec));
    SliceCtl &ctl = *reinterpret_cast<SliceCtl *>(reinterpret_cast<uint8_t *>(vkey) + queue_bytes(a.max_vec));

    pdl_launch_dependents();  // the merge kernel may be scheduled as CTAs retire

    const uint32_t S = (uint32_t)a.slices;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t V = (int32_t)a.V;
    const uint32_t G = gridDim.x;
    const int64_t g_rows = G / S;  // the item index advances by G = g_rows * S + g_sl
    const uint32_t g_sl = G % S;
    uint8_t *ws = reinterpret_cast<uint8_t *>(a.workspace);
    SliceSumm *summ = reinterpret_cast<SliceSumm *>(ws + a.summ_off);
    uint64_t *cands = reinterpret_cast<uint64_t *>(ws + a.cand_off);
    const bool has_mask = a.mask != nullptr;

    auto row_ptr = [&](int64_t row) {
        return reinterpret_cast<const uint8_t *>(a.logits) + (size_t)row * a.stride * E::SIZE;
    };
    // Slice geometry: rows with the first row's 16-byte misalignment (all of
    // them when the row stride is a multiple of 16 bytes) use a table of the
    // vector split computed once; other rows compute it.
    const int32_t mis0 = (int32_t)(reinterpret_cast<uintptr_t>(a.logits) & 15u) / E::SIZE;
    if (tid <= (int)S) {
        const Slice32 s0 = make_slice32<AE, E::SIZE>(a.logits, V, min((uint32_t)tid, S - 1), S);
        ctl.vb[tid] = tid < (int)S ? s0.vc0 : s0.vc0 + s0.nv;
        if (tid == 0) {
            ctl.g_head = s0.head;
            ctl.g_nvec = s0.nvec;
            ctl.g_tail = s0.tail;
        }
    }
    auto geometry = [&](const uint8_t *rp, uint32_t c) -> Slice32 {
        const int32_t mis = (int32_t)(reinterpret_cast<uintptr_t>(rp) & 15u) / E::SIZE;
        if (mis != mis0) return make_slice32<AE, E::SIZE>(rp, V, c, S);
        Slice32 s;
        s.head = ctl.g_head;
        s.nvec = ctl.g_nvec;
        s.tail = ctl.g_tail;
        s.vc0 = ctl.vb[c];
        const int32_t vc1 = ctl.vb[c + 1];
        s.nv = vc1 - s.vc0;
        s.base = s.head + s.vc0 * AE - AE;
        s.lo = (c == 0) ? 0 : s.head + s.vc0 * AE;
        s.hi = (c == S - 1) ? V : s.head + vc1 * AE;
        s.vbeg = (c == 0 && s.head > 0) ? 0 : 1;
        s.vend = (c == S - 1 && s.tail > 0) ? s.nv + 2 : s.nv + 1;
        return s;
    };
    auto advance = [&](int64_t &row, uint32_t &sl) {
        row += g_rows;
        sl += g_sl;
        if (sl >= S) {
            sl -= S;
            ++row;
        }
    };
    // Start the copies of item (row, sl) into buffer b: the slice's aligned
    // vectors by one bulk copy, its mask words by 4-byte cp.async (one group
    // per thread per item, committed even when empty).
    auto issue = [&](int64_t row, uint32_t sl, int b) {
        if (row < a.B) {
            const uint8_t *rp = row_ptr(row);
            const Slice32 s = geometry(rp, sl);
            if (tid == 0) {
                const uint32_t bytes = (uint32_t)s.nv * 16u;
                mbar_arrive_expect_tx(&ctl.mbar[b], bytes);
                if (bytes)
                    bulk_g2s(smem + b * sb + 16, rp + (size_t)(s.head + s.vc0 * AE) * E::SIZE, bytes,
                             &ctl.mbar[b]);
            }
            if (has_mask && s.hi > s.lo) {
                const int32_t *mrow = a.mask + (size_t)row * a.mstride;
                const int32_t w0 = s.lo >> 5, nw = ((s.hi - 1) >> 5) - w0 + 1;
                uint32_t *mw = reinterpret_cast<uint32_t *>(mask_base + b * mb);
                for (int32_t j = tid; j < nw; j += kThreads) cp_async_4(mw + j, mrow + w0 + j);
            }
        }
        cp_async_commit();
    };

    if (tid == 0) {
        for (int j = 0; j < NBUF; ++j) mbar_init(&ctl.mbar[j], 1);
        mbar_init_fence();
    }
    __syncthreads();
    int64_t row = blockIdx.x / S;
    uint32_t sl = blockIdx.x % S;
    int64_t prow = row;
    uint32_t psl = sl;
    for (int j = 0; j < NBUF; ++j) {
        issue(prow, psl, j);
        advance(prow, psl);
    }

    for (int it = 0; row < a.B; ++it, advance(row, sl)) {
        const int b = NBUF == 1 ? 0 : (it & 1);
        const int par = it & 1;
        uint4 *slice = reinterpret_cast<uint4 *>(smem + b * sb);
        const uint32_t *mw = reinterpret_cast<const uint32_t *>(mask_base + b * mb);
        const uint8_t *rp = row_ptr(row);
        const Slice32 s = geometry(rp, sl);
        const int32_t base = s.base;
        const int nv = s.nv;
        const RowParams rpm = row_params(a, row);
        const bool need_z = rpm.p_on;
        const bool need_tau = rpm.k_on && rpm.K <= kTauMaxK;
        const float c2 = rpm.c2, invT = rpm.invT, T = rpm.T;
        const int32_t wlo = s.lo >> 5;
        const int32_t moff = base - 32 * wlo;  // bit of smem element 0 in the mask buffer
        const bool straddle = (moff & (AE - 1)) != 0;
        // mask bits of interior vector v (bit t <-> element base + v AE + t)
        auto vec_bits = [&](int v) -> uint32_t {
            if (!has_mask) return kFull;
            const int32_t rel = moff + v * AE;
            const uint32_t mword = mw[rel >> 5];
            const uint32_t k = straddle ? __funnelshift_r(mword, mw[(rel >> 5) + 1], rel & 31) : (mword >> (rel & 31));
            return k & kFull;
        };
        // allowed logits of vector v; disallowed (or out-of-row) become -inf.
        // The two boundary slots were cleaned in shared memory by phase A.
        auto load_vec = [&](int v, float *x) {
            E::unpack(slice[v], x);
            if (v >= 1 && v <= nv && has_mask) {
                const uint32_t k = vec_bits(v);
#pragma unroll
                for (int t = 0; t < AE; ++t) x[t] = (k >> t) & 1u ? x[t] : -INFINITY;
            }
        };

        // ---- wait for the slice (one warp polls) and its mask words
        if (warp == 0) mbar_wait_bounded(&ctl.mbar[b], (uint32_t)(it / NBUF) & 1u, &g_sample_status);
        if (NBUF == 2) cp_async_wait<1>();
        else cp_async_wait<0>();
        if (sl == 0 && tid < s.head) {  // misaligned row start: plain loads
            if (E::SIZE == 4) reinterpret_cast<uint32_t *>(slice)[tid - base] = reinterpret_cast<const uint32_t *>(rp)[tid];
            else reinterpret_cast<unsigned short *>(slice)[tid - base] = reinterpret_cast<const unsigned short *>(rp)[tid];
        }
        if (sl == S - 1 && tid < s.tail) {
            const int32_t e = s.head + s.nvec * AE + tid;
            if (E::SIZE == 4) reinterpret_cast<uint32_t *>(slice)[e - base] = reinterpret_cast<const uint32_t *>(rp)[e];
            else reinterpret_cast<unsigned short *>(slice)[e - base] = reinterpret_cast<const unsigned short *>(rp)[e];
        }
        if (tid == 0) {
            ctl.n = 0;
            ctl.nq = 0;
        }
        __syncthreads();

        // ---- phase A: two independent accumulators per thread.  NaN never
        // wins a max (fmaxf skips it) and adds ~2^-126 to the exponent sum.
        const bool need_vkey = !rpm.greedy;
        auto store_vkey = [&](int v, float vmax) {
            if (need_vkey) vkey[v] = (uint16_t)((okey(vmax) + 0xFFFFu) >> 16);
        };
        auto accumulate = [&](const float *x, int32_t e0, Acc &A) -> float {
            float vmax = x[0];
#pragma unroll
            for (int t = 1; t < AE; ++t) vmax = fmaxf(vmax, x[t]);
            if (vmax > A.mx) {  // rare after the first few vectors
                if (need_z) A.z *= ex2_approx((A.mx - vmax) * c2);
                int tt = AE - 1;
#pragma unroll
                for (int t = AE - 1; t >= 0; --t)
                    if (x[t] == vmax) tt = t;
                A.mx = vmax;
                A.mi = (uint32_t)(e0 + tt);
            }
            if (need_z && A.mx > -INFINITY) {
                // (x - mx) c2, not x c2 - mx c2: the product mx c2 would be
                // rounded once and scale every term alike, by up to |mx c2| 2^-24
#pragma unroll
                for (int t = 0; t < AE; ++t) A.z += ex2_approx(fmaxf((x[t] - A.mx) * c2, -126.f));
            }
            return vmax;
        };
        auto boundary_slot = [&](int v, Acc &A) {  // head / tail slot: per-element checks, cleaned in place
            uint4 raw = slice[v];
            float x[AE];
            E::unpack(raw, x);
            uint32_t drop = 0;
#pragma unroll
            for (int t = 0; t < AE; ++t) {
                const int32_t e = base + v * AE + t;
                bool ok = e >= s.lo && e < s.hi && x[t] == x[t];
                if (ok && has_mask) ok = (mw[(e >> 5) - wlo] >> (e & 31)) & 1u;
                if (!ok) {
                    drop |= 1u << t;
                    x[t] = -INFINITY;
                }
            }
            if (drop) {
                E::store_ninf(raw, drop);
                slice[v] = raw;
            }
            store_vkey(v, accumulate(x, base + v * AE, A));
        };
        Acc A0 = {-INFINITY, 0xFFFFFFFFu, 0.f}, A1 = {-INFINITY, 0xFFFFFFFFu, 0.f};
        if (s.vbeg == 0 && tid == 0) boundary_slot(0, A0);
        int v = 1 + tid;
        for (; v + kThreads <= nv; v += 2 * kThreads) {
            float x0[AE], x1[AE];
            load_vec(v, x0);
            load_vec(v + kThreads, x1);
            const float m0 = accumulate(x0, base + v * AE, A0);
            const float m1 = accumulate(x1, base + (v + kThreads) * AE, A1);
            store_vkey(v, m0);
            store_vkey(v + kThreads, m1);
        }
        if (v <= nv) {
            float x0[AE];
            load_vec(v, x0);
            store_vkey(v, accumulate(x0, base + v * AE, A0));
        }
        if (s.vend == nv + 2 && tid == kThreads - 1) boundary_slot(nv + 1, A1);
        // merge the two accumulators (value desc, index asc)
        Acc A = A0;
        if (A1.mx > A0.mx || (A1.mx == A0.mx && A1.mi < A0.mi)) A = A1;
        if (need_z && A.mx > -INFINITY) {
            A.z = (A0.mx > -INFINITY ? A0.z * ex2_approx((A0.mx - A.mx) * c2) : 0.f) +
                  (A1.mx > -INFINITY ? A1.z * ex2_approx((A1.mx - A.mx) * c2) : 0.f);
        }

        // ---- slice summaries: warp level, one block barrier
        {
            const uint32_t kv = (A.mx > -INFINITY) ? okey(A.mx) : 0u;
            const uint32_t wkv = __reduce_max_sync(0xFFFFFFFFu, kv);
            const uint32_t wmi = __reduce_min_sync(0xFFFFFFFFu, (kv == wkv && wkv) ? A.mi : 0xFFFFFFFFu);
            const uint64_t wk = wkv ? (((uint64_t)wkv << 32) | (uint64_t)(0xFFFFFFFFu - wmi)) : 0ull;
            const float wm = wkv ? okey_value(wkv) : -INFINITY;
            float wz = 0.f;
            if (need_z) wz = warp_sum_f32(A.mx > -INFINITY ? A.z * ex2_approx((A.mx - wm) * c2) : 0.f);
            float wtau = -INFINITY;
            if (need_tau) {  // the warp's r-th largest thread maximum (remove the top r - 1)
                const int r = (rpm.K + kWarps - 1) / kWarps;
                uint32_t kk = kv, kth = 0;
                for (int i = 0; i < r; ++i) {
                    kth = __reduce_max_sync(0xFFFFFFFFu, kk);
                    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, kk == kth);
                    if (lane == __ffs(hit) - 1) kk = 0;
                }
                wtau = kth ? okey_value(kth) : -INFINITY;
            }
            uint64_t wb = 0;
            if (rpm.unfiltered) {  // seed: every thread maximum's perturbed score vs the warp max
                float sc = -INFINITY;
                if (A.mx > -INFINITY) {
                    const uint4 blk = token_block(a.seed, a.offset, (uint32_t)row, A.mi >> 2);
                    sc = (A.mx - wm) * invT + gumbel_of(block_word(blk, A.mi & 3));
                }
                wb = warp_max_u64(A.mx > -INFINITY ? rank_key(sc, A.mi) : 0ull);
            }
            if (lane == 0) {
                ctl.w_key[par][warp] = wk;
                ctl.w_z[par][warp] = wz;
                ctl.w_tau[par][warp] = wtau;
                ctl.w_best[par][warp] = wb;
            }
        }
        __syncthreads();
        uint64_t s_key = 0;
        float s_tau = INFINITY;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) {
            s_key = ctl.w_key[par][i] > s_key ? ctl.w_key[par][i] : s_key;
            s_tau = fminf(s_tau, ctl.w_tau[par][i]);
        }
        if (!need_tau) s_tau = -INFINITY;
        const float m_s = s_key ? rank_key_value(s_key) : -INFINITY;

        uint32_t ncand = 0;
        uint32_t best_i = 0xFFFFFFFFu;
        float best_x = -INFINITY;
        if (rpm.filtered && s_key) {
            const float v_m_s = rpm.m_on ? min_p_cut(m_s, rpm.tlnmp) : -INFINITY;  // below the row's cut
            const float theta = fmaxf(s_tau, v_m_s);
            if (theta > -INFINITY || s.hi - s.lo <= kSliceCap) {
                // ---- publish every allowed logit >= theta of this slice
                uint64_t *out = cands + (size_t)(row * S + sl) * kSliceCap;
                const uint32_t th16 = okey(theta) >> 16;
                for (int v0 = s.vbeg; v0 < s.vend; v0 += kThreads) {
                    const int vv = v0 + tid;
                    uint32_t hit = 0;
                    float x[AE];
                    if (vv < s.vend && vkey[vv] >= th16) {
                        load_vec(vv, x);
#pragma unroll
                        for (int t = 0; t < AE; ++t)
                            if (x[t] >= theta && x[t] > -INFINITY) hit |= 1u << t;
                    }
                    if (!__any_sync(0xFFFFFFFFu, hit != 0)) continue;
                    const uint32_t nh = __popc(hit);
                    uint32_t incl = nh;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                        if (lane >= o) incl += t;
                    }
                    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
                    uint32_t basep = 0;
                    if (lane == 31) basep = atomicAdd(&ctl.n, total);
                    basep = __shfl_sync(0xFFFFFFFFu, basep, 31);
                    uint32_t pos = basep + incl - nh;
                    const int32_t e0 = base + vv * AE;
#pragma unroll
                    for (int t = 0; t < AE; ++t)
                        if (hit & (1u << t)) {
                            if (pos < (uint32_t)kSliceCap) __stcg(out + pos, rank_key(x[t], (uint32_t)(e0 + t)));
                            ++pos;
                        }
                }
                __syncthreads();
                ncand = ctl.n;
            } else {
                ncand = kNoCandidates;
            }
        } else if (rpm.unfiltered && s_key) {
            // ---- this slice's Gumbel-max winner (scores relative to m_s),
            // seeded with the best thread maximum.  A logit below `cut`
            // cannot win even with the largest Gumbel value; the vectors
            // holding one at or above it are queued and their Philox blocks
            // computed densely, and a uniform must clear gumbel_u_floor
            // before the exact Gumbel transform is evaluated.
            uint64_t seed_key = 0;
#pragma unroll
            for (int i = 0; i < kWarps; ++i) {
                const uint64_t wb = ctl.w_best[par][i];
                if (!wb) continue;
                const float sc = rank_key_value(wb) + (rank_key_value(ctl.w_key[par][i]) - m_s) * invT;
                const uint64_t k2 = rank_key(sc, rank_key_index(wb));
                seed_key = k2 > seed_key ? k2 : seed_key;
            }
            float best = rank_key_value(seed_key);
            uint32_t bi = rank_key_index(seed_key);
            const float cut0 = fmaf(best - kGumbelMax, T, m_s);
            const uint32_t cut16 = okey(cut0) >> 16;
            for (int v0 = s.vbeg; v0 < s.vend; v0 += kThreads) {
                const int vv = v0 + tid;
                const bool q = vv < s.vend && vkey[vv] >= cut16;
                const uint32_t bal = __ballot_sync(0xFFFFFFFFu, q);
                if (!bal) continue;
                uint32_t qb = 0;
                if (lane == 0) qb = atomicAdd(&ctl.nq, (uint32_t)__popc(bal));
                qb = __shfl_sync(0xFFFFFFFFu, qb, 0);
                if (q) queue[qb + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)vv;
            }
            __syncthreads();
            const uint32_t nq = ctl.nq;
            float cut = cut0;
            for (uint32_t qi = tid; qi < nq; qi += kThreads) {
                const int vv = queue[qi];
                float x[AE];
                load_vec(vv, x);
                const int32_t e0 = base + vv * AE;
                uint32_t q_cached = 0xFFFFFFFFu;
                uint4 blk = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int t = 0; t < AE; ++t) {
                    const float xt = x[t];
                    if (!(xt >= cut) || !(xt > -INFINITY)) continue;
                    const uint32_t e = (uint32_t)(e0 + t);
                    if ((e >> 2) != q_cached) {
                        q_cached = e >> 2;
                        blk = token_block(a.seed, a.offset, (uint32_t)row, q_cached);
                    }
                    const uint32_t word = block_word(blk, e & 3);
                    const float srel = (xt - m_s) * invT;
                    const float need = best - srel;  // the Gumbel value this token must beat
                    if (need > kTopBitsMargin && (word >> 22) != 0x3FFu) continue;
                    if (word_uniform(word) < gumbel_u_floor(need)) continue;
                    const float sc = srel + gumbel_of(word);
                    if (sc > best || (sc == best && e < bi)) {
                        best = sc;
                        bi = e;
                        cut = fmaf(best - kGumbelMax, T, m_s);
                    }
                }
            }
            const uint64_t bk = block_max_u64(rank_key(best, bi), ctl.sc);
            best_i = rank_key_index(bk);
            float bx[AE];
            const int32_t j = (int32_t)best_i - base;
            E::unpack(slice[j / AE], bx);
            best_x = bx[j % AE];
        }
        if (tid == 0) {
            float s_z = 0.f;
            if (need_z && s_key) {
#pragma unroll
                for (int i = 0; i < kWarps; ++i)
                    if (ctl.w_key[par][i]) s_z += ctl.w_z[par][i] * ex2_approx((rank_key_value(ctl.w_key[par][i]) - m_s) * c2);
            }
            SliceSumm o;
            o.argmax_key = s_key;
            o.z = s_z;
            o.tau = s_tau;
            o.ncand = ncand;
            o.best_idx = best_i;
            o.best_x = best_x;
            o.pad = 0;
            SliceSumm *my = summ + row * S + sl;
            __stcg(reinterpret_cast<float4 *>(my), reinterpret_cast<const float4 *>(&o)[0]);
            __stcg(reinterpret_cast<float4 *>(my) + 1, reinterpret_cast<const float4 *>(&o)[1]);
        }
        // this item is done with buffer b: refill it
        __syncthreads();
        fence_proxy_async_smem();
        issue(prow, psl, b);
        advance(prow, psl);
    }
}

// ============================================================== merge kernel
template <int DT>
__global__ void __launch_bounds__(kThreads) sample_merge_kernel(SampleArgs a) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *cand = reinterpret_cast<uint64_t *>(smem);
    Hist &hist = *reinterpret_cast<Hist *>(smem + kMergeCap * 8);
    MergeCtl &ctl = *reinterpret_cast<MergeCtl *>(smem + kMergeCap * 8 + sizeof(Hist));

    const int64_t row = blockIdx.x;
    const uint32_t S = (uint32_t)a.slices;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint8_t *ws = reinterpret_cast<const uint8_t *>(a.workspace);
    const SliceSumm *summ = reinterpret_cast<const SliceSumm *>(ws + a.summ_off) + row * S;
    const uint64_t *cands = reinterpret_cast<const uint64_t *>(ws + a.cand_off) + (size_t)row * S * kSliceCap;
    const RowParams rpm = row_params(a, row);
    const float invT = rpm.invT, c2 = rpm.c2;

    pdl_wait_primary();  // the slice kernel's summaries and candidates are visible

    // slice r -> lane r of warps 0 and 1; warp-level reductions in a fixed
    // lane order, so every result is deterministic
    if (tid < 64) {
        SliceSumm o;
        if (tid < (int)S) {
            reinterpret_cast<float4 *>(&o)[0] = __ldcg(reinterpret_cast<const float4 *>(summ + tid));
            reinterpret_cast<float4 *>(&o)[1] = __ldcg(reinterpret_cast<const float4 *>(summ + tid) + 1);
        } else {
            o.argmax_key = 0;
            o.z = 0.f;
            o.tau = -INFINITY;
            o.ncand = 0;
            o.best_idx = 0xFFFFFFFFu;
            o.best_x = -INFINITY;
        }
        if (tid < (int)S) {
            ctl.q_key[tid] = o.argmax_key;
            ctl.q_n[tid] = o.ncand;
        }
        const uint64_t wk = warp_max_u64(o.argmax_key);
        const uint32_t wt = __reduce_max_sync(0xFFFFFFFFu, o.argmax_key ? okey(o.tau) : 0u);
        const bool ovf = o.argmax_key && o.ncand > (uint32_t)kSliceCap;  // no complete list
        const uint32_t wf = __ballot_sync(0xFFFFFFFFu, ovf);
        if (lane == 0) {
            ctl.wk2[warp] = wk;
            ctl.wt2[warp] = wt;
            ctl.wf2[warp] = wf;
        }
        __syncwarp();
        // both warps need the row max: a named barrier over the first 64 threads
        asm volatile("bar.sync 1, 64;" ::: "memory");
        const uint64_t gk = ctl.wk2[0] > ctl.wk2[1] ? ctl.wk2[0] : ctl.wk2[1];
        const float gm = gk ? rank_key_value(gk) : -INFINITY;
        float zr = 0.f;
        if (rpm.p_on && o.argmax_key) zr = o.z * ex2_approx((rank_key_value(o.argmax_key) - gm) * c2);
        zr = warp_sum_f32(zr);
        uint64_t br = 0;
        if (rpm.unfiltered && o.argmax_key && o.best_idx != 0xFFFFFFFFu) {
            // the slice winner rescored against the row max
            const uint32_t idx = o.best_idx;
            const uint4 blk = token_block(a.seed, a.offset, (uint32_t)row, idx >> 2);
            br = rank_key((o.best_x - gm) * invT + gumbel_of(block_word(blk, idx & 3)), idx);
        }
        br = warp_max_u64(br);
        if (lane == 0) {
            ctl.wz2[warp] = zr;
            ctl.wb2[warp] = br;
        }
        asm volatile("bar.sync 1, 64;" ::: "memory");
        if (tid == 0) {
            ctl.g_key = gk;
            const uint32_t t2 = max(ctl.wt2[0], ctl.wt2[1]);
            ctl.g_tau = t2 ? okey_value(t2) : -INFINITY;
            ctl.g_flags = (ctl.wf2[0] | ctl.wf2[1]) ? 1u : 0u;
            ctl.g_z = ctl.wz2[0] + ctl.wz2[1];
            ctl.g_best = ctl.wb2[0] > ctl.wb2[1] ? ctl.wb2[0] : ctl.wb2[1];
            ctl.n = 0;
        }
    }
    __syncthreads();
    const uint64_t gkey = ctl.g_key;
    const float m = gkey ? rank_key_value(gkey) : -INFINITY;
    const uint32_t amax = gkey ? rank_key_index(gkey) : 0u;
    float vstar = -INFINITY;
    int64_t token = -1;
    if (!gkey) {
        vstar = __int_as_float(0x7FC00000);
    } else if (rpm.greedy) {
        token = amax;
        vstar = m;
    } else if (rpm.unfiltered) {
        token = rank_key_index(ctl.g_best);
    } else {
        const float v_m = rpm.m_on ? min_p_cut(m, rpm.tlnmp) : -INFINITY;
        const float theta = fmaxf(ctl.g_tau, v_m);
        bool done = false;
        if (!ctl.g_flags) {
            // gather the candidates >= theta: warp w takes slices w, w + 8, ...
            // and issues up to 8 loads per lane before using any
            for (uint32_t r = warp; r < S; r += kWarps) {
                const uint32_t nr = ctl.q_key[r] ? ctl.q_n[r] : 0u;
                const uint64_t *src = cands + (size_t)r * kSliceCap;
                for (uint32_t j0 = 0; j0 < nr; j0 += 32 * 8) {
                    uint64_t kv[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t j = j0 + u * 32 + lane;
                        kv[u] = j < nr ? __ldcg(src + j) : 0ull;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const bool keep = kv[u] && rank_key_value(kv[u]) >= theta;
                        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
                        if (!bal) continue;
                        uint32_t bp = 0;
                        if (lane == 0) bp = atomicAdd(&ctl.n, (uint32_t)__popc(bal));
                        bp = __shfl_sync(0xFFFFFFFFu, bp, 0);
                        const uint32_t pos = bp + __popc(bal & ((1u << lane) - 1u));
                        if (keep && pos < (uint32_t)kMergeCap) cand[pos] = kv[u];
                    }
                }
            }
            __syncthreads();
            done = select_from_candidates<BlockSync>(a, row, rpm, cand, ctl.n, (uint32_t)kMergeCap, theta, v_m, m,
                                                     ctl.g_z, hist, ctl.sel, token, vstar);
        }
        if (!done)
            general_path<DT, BlockSync>(a, row, rpm, m, amax, (double)ctl.g_z, v_m, smem, ctl.sel, token, vstar);
    }
    (void)AE;
    if (tid == 0) {
        a.tokens[row] = token;
        if (a.vstar_out) a.vstar_out[row] = vstar;
    }
}

// ---------------------------------------------------------------- host side
size_t sample_smem_bytes(int64_t max_vec, int64_t max_words, int nbuf) {
    return (size_t)nbuf * (slice_bytes(max_vec) + mask_bytes(max_words)) + 2 * queue_bytes(max_vec) + sizeof(SliceCtl);
}
static size_t merge_smem_bytes() { return (size_t)kMergeCap * 8 + sizeof(Hist) + sizeof(MergeCtl); }

namespace {
struct Fit {
    const void *fn;
    int device;
    size_t smem;
    int blocks;
};
Fit g_fits[32];
int g_nfits = 0;

int resident_blocks(const void *fn, size_t smem) {  // co-resident CTAs on the device (cached)
    int dev = 0;
    cudaGetDevice(&dev);
    for (int i = 0; i < g_nfits; ++i)
        if (g_fits[i].fn == fn && g_fits[i].device == dev && g_fits[i].smem == smem) return g_fits[i].blocks;
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem) != cudaSuccess) per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int n = per_sm * sms;
    if (g_nfits < 32) g_fits[g_nfits++] = {fn, dev, smem, n};
    return n;
}
}  // namespace

int sample_launch(const SampleArgs &args, int dtype, int slices, int64_t max_vec, int nbuf, cudaStream_t st) {
    if (args.B >= kRowKernelMinB) return sample_row_launch(args, dtype, st);
    const void *slice_fns[3][2] = {{(const void *)sample_slice_kernel<0, 1>, (const void *)sample_slice_kernel<0, 2>},
                                   {(const void *)sample_slice_kernel<1, 1>, (const void *)sample_slice_kernel<1, 2>},
                                   {(const void *)sample_slice_kernel<2, 1>, (const void *)sample_slice_kernel<2, 2>}};
    const void *merge_fns[3] = {(const void *)sample_merge_kernel<0>, (const void *)sample_merge_kernel<1>,
                                (const void *)sample_merge_kernel<2>};
    const void *fn = slice_fns[dtype][nbuf - 1];
    const void *mfn = merge_fns[dtype];
    const int AE = dtype == 0 ? 4 : 8;
    const int64_t max_words = (max_vec + 2) * AE / 32 + 3;
    const size_t smem = sample_smem_bytes(max_vec, max_words, nbuf);
    const size_t msmem = merge_smem_bytes();
    if (prepare_kernel(fn, smem, 1) != 0 || prepare_kernel(mfn, msmem, 1) != 0) return -1;
    const int64_t items = args.B * slices;
    int64_t grid = resident_blocks(fn, smem);
    if (grid < 1) return -1;
    if (grid > items) grid = items;
    SampleArgs a = args;
    a.max_vec = max_vec;
    a.max_words = max_words;
    a.slices = slices;
    size_t so = 0, co = 0;
    sample_workspace_layout(args.B, slices, &so, &co);
    a.summ_off = so;
    a.cand_off = co;
    void *params[] = {&a};
    if (cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kThreads), params, smem, st) != cudaSuccess) return -1;
    // the merge: one CTA per row, scheduled while the slice kernel drains
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)args.B, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = msmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, mfn, params) == cudaSuccess ? 0 : -1;
}

unsigned int *sample_status_ptr() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sample_status) != cudaSuccess) return nullptr;
    return reinterpret_cast<unsigned int *>(p);
}

}  // namespace tsa
