// sample, one CTA per row (logits-processor, "API" and "Method";
// logits-mask-xpu, "Method" for top_k == 1), for batches with enough rows to
// occupy the GPU.
//
// A producer warp streams the row through a ring of shared-memory stages: each
// stage is one 1-D bulk copy (cp.async.bulk) of up to kStageVec 16-byte
// vectors plus the mask words that cover them (4-byte cp.async), both
// completing on the stage's "full" mbarrier; the eight consumer warps release
// a stage on its "empty" mbarrier.  Every logit is read from HBM once.
//
// Each consumer thread keeps, over the vectors it reads (vector j of a stage
// goes to thread j mod 256): the maximum, its lowest index, and the sum of
// exp((l - max) / T) relative to its own maximum.  A keep-threshold lower
// bound theta rises as the row streams by:
//   - top-k: each warp's r-th largest thread maximum, r = ceil(k / 8), is a
//     logit with at least r - 1 larger ones among distinct thread maxima in
//     that warp, so the minimum over the 8 warps has at least k logits of
//     the row at or above it;
//   - min-p: the cut m + T ln(min_p) at the largest maximum seen so far,
//     which is below the cut at the row maximum.
// Both only grow, so reading another warp's published value late is safe.
// Every allowed logit >= theta at the time it is read is pushed as a rank key
// into a shared candidate list; since the final threshold is at least every
// earlier one, the list holds every logit >= the final theta.  The first
// stage is read twice (once to seed theta, once to push).  Unfiltered rows
// draw Gumbel-max in the stream instead, each thread pruning tokens that
// cannot beat its own best score.  At the end the consumer warps reduce the
// row's maximum, argmax and normaliser, and resolve the exact keep-threshold
// and the draw from the candidates; a row with no usable threshold (top-p
// alone), an overflowing list or a NaN in the normaliser takes the general
// path, which re-reads the row.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_host.h"
#include "tsa_sample_common.cuh"
#include "tsa_select.cuh"

namespace tsa {

using namespace sample_detail;

namespace {
constexpr int kCW = kWarps;            // consumer warps
constexpr int kCT = kCW * 32;          // consumer threads (threadIdx.x < kCT)
constexpr int kRowThreads = kCT + 32;  // plus the producer warp
constexpr int kStages = 4;
constexpr int kStageVec = 1024;  // 16-byte vectors per stage (16 KB)
constexpr int kVecPerThread = kStageVec / kCT;
// mask words one stage may span (8 elements per vector, unaligned start), plus
// one spare word read by the straddling bit extraction
constexpr int kStageWords = (kStageVec * 8 / 32 + 2 + 7) & ~7;
constexpr int kCandCap = 2048;
constexpr int kRefresh = 4;  // stages between threshold refreshes
constexpr int kTauMaxR = 32;  // largest r = ceil(k / 8) for which the top-k bound is formed

using CSync = NamedSync<1, kCT>;

enum Mode { kGreedy = 0, kFilter = 1, kFilterZ = 2, kZOnly = 3, kUnfiltered = 4 };

struct __align__(16) RowCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    SelCtl sel;
    uint32_t ncand;
    float wtau[kCW];  // per-warp top-k bound (grows)
    float wmax[kCW];  // per-warp running maximum (grows)
    uint64_t wkey[kCW];
    float wz[kCW];
    uint64_t wbest[kCW];
};

struct Acc {
    float mx;      // running maximum
    uint32_t mi;   // its lowest index
    float z0, z1;  // sum of 2^((l - mx) c2), two partial sums
    float nm;      // -mx c2
    float sbest;   // unfiltered: best score (l - ref) / T + G
    uint32_t sbi;
    float gcut;    // unfiltered: logits below it cannot beat sbest
};

struct Ctx {
    int64_t row;
    float T, invT, c2, theta, ref;
    uint64_t seed, offset;
    uint64_t *cand;
    uint32_t *ncand;
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (the arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Accumulate one element group (x[0 .. n) at indices e0 ..) into the thread's
// running maximum / argmax / normaliser; returns the group maximum.
template <int N, bool Z>
__device__ __forceinline__ float accumulate(const float *x, uint32_t e0, float c2, Acc &A) {
    float vmax = x[0];
    if (N == 4) {
        vmax = fmaxf(fmax3(x[0], x[1], x[2]), x[3]);
    } else {
#pragma unroll
        for (int t = 1; t < N; ++t) vmax = fmaxf(vmax, x[t]);
    }
    if (vmax > A.mx) {  // rare after the first few vectors
        if (Z) {
            const float s = ex2_approx((A.mx - vmax) * c2);
            A.z0 *= s;
            A.z1 *= s;
        }
        int tt = N - 1;
#pragma unroll
        for (int t = N - 1; t >= 0; --t)
            if (x[t] == vmax) tt = t;
        A.mx = vmax;
        A.mi = e0 + (uint32_t)tt;
        A.nm = -vmax * c2;
    }
    if (Z) {
#pragma unroll
        for (int t = 0; t < N; t += 2) {
            A.z0 += ex2_approx(fmaf(x[t], c2, A.nm));
            if (t + 1 < N) A.z1 += ex2_approx(fmaf(x[t + 1], c2, A.nm));
        }
    }
    return vmax;
}

// Push every logit of the group that is >= theta.
template <int N>
__device__ __forceinline__ void push(const float *x, uint32_t e0, float vmax, const Ctx &cx) {
    if (!(vmax >= cx.theta)) return;
#pragma unroll
    for (int t = 0; t < N; ++t)
        if (x[t] >= cx.theta && x[t] > -INFINITY) {
            const uint32_t pos = atomicAdd(cx.ncand, 1u);
            if (pos < (uint32_t)kCandCap) cx.cand[pos] = rank_key(x[t], e0 + (uint32_t)t);
        }
}

// Unfiltered draw: the group's tokens that can still beat the thread's best
// perturbed score.
template <int N>
__device__ __forceinline__ void gumbel(const float *x, uint32_t e0, float vmax, const Ctx &cx, Acc &A) {
    if (!(vmax >= A.gcut)) return;
    uint32_t q_cached = 0xFFFFFFFFu;
    uint4 blk = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int t = 0; t < N; ++t) {
        const float xt = x[t];
        if (!(xt >= A.gcut) || !(xt > -INFINITY)) continue;
        const uint32_t e = e0 + (uint32_t)t;
        if ((e >> 2) != q_cached) {
            q_cached = e >> 2;
            blk = token_block(cx.seed, cx.offset, (uint32_t)cx.row, q_cached);
        }
        const uint32_t word = block_word(blk, e & 3);
        const float srel = (xt - cx.ref) * cx.invT;
        const float need = A.sbest - srel;  // the Gumbel value this token must beat
        if (need > kTopBitsMargin && (word >> 22) != 0x3FFu) continue;
        if (word_uniform(word) < gumbel_u_floor(need)) continue;
        const float sc = srel + gumbel_of(word);
        if (sc > A.sbest || (sc == A.sbest && e < A.sbi)) {
            A.sbest = sc;
            A.sbi = e;
            A.gcut = fmaf(sc - kGumbelMax, cx.T, cx.ref);
        }
    }
}

// One stage of this thread's vectors.  PASS 1 accumulates only, PASS 2 pushes
// / draws only, PASS 3 does both.
template <int DT, int MODE, int PASS>
__device__ __forceinline__ void run_stage(const uint4 *stage, const uint32_t *mw, int nvc, uint32_t e0, bool has_mask,
                                          bool straddle, const Ctx &cx, Acc &A) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    constexpr uint32_t kFull = (1u << AE) - 1u;
    constexpr bool kZ = MODE == kFilterZ || MODE == kZOnly;
    const uint32_t rel0 = e0 & 31u;
    // vectors are loaded kU at a time (two 4-element vectors, or one of 8),
    // which keeps the kernel within the registers of two CTAs per SM
    constexpr int kU = AE == 4 ? 2 : 1;
#pragma unroll 1
    for (int i0 = 0; i0 < kVecPerThread; i0 += kU) {
        float x[kU][AE];
        bool ok[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int j = (int)threadIdx.x + (i0 + u) * kCT;
            ok[u] = j < nvc;
            if (ok[u]) E::unpack(stage[j], x[u]);
        }
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            if (!ok[i]) continue;
            const int j = (int)threadIdx.x + (i0 + i) * kCT;
            if (has_mask) {
                const uint32_t rel = rel0 + (uint32_t)j * AE;
                const uint32_t k = rel >> 5, sh = rel & 31u;
                const uint32_t bits = (straddle ? __funnelshift_r(mw[k], mw[k + 1], sh) : (mw[k] >> sh)) & kFull;
#pragma unroll
                for (int t = 0; t < AE; ++t) x[i][t] = (bits >> t) & 1u ? x[i][t] : -INFINITY;
            }
            const uint32_t ej = e0 + (uint32_t)j * AE;
            float vmax;
            if (PASS & 1) {
                vmax = accumulate<AE, kZ>(x[i], ej, cx.c2, A);
            } else {
                vmax = x[i][0];
#pragma unroll
                for (int t = 1; t < AE; ++t) vmax = fmaxf(vmax, x[i][t]);
            }
            if (PASS & 2) {
                if (MODE == kFilter || MODE == kFilterZ) push<AE>(x[i], ej, vmax, cx);
                if (MODE == kUnfiltered) gumbel<AE>(x[i], ej, vmax, cx, A);
            }
        }
    }
}

template <int DT, int PASS>
__device__ __forceinline__ void run_stage_mode(int mode, const uint4 *stage, const uint32_t *mw, int nvc, uint32_t e0,
                                               bool has_mask, bool straddle, const Ctx &cx, Acc &A) {
    switch (mode) {
        case kGreedy:
            if (PASS & 1) run_stage<DT, kGreedy, 1>(stage, mw, nvc, e0, has_mask, straddle, cx, A);
            break;
        case kFilter: run_stage<DT, kFilter, PASS>(stage, mw, nvc, e0, has_mask, straddle, cx, A); break;
        case kFilterZ: run_stage<DT, kFilterZ, PASS>(stage, mw, nvc, e0, has_mask, straddle, cx, A); break;
        case kZOnly:
            if (PASS & 1) run_stage<DT, kZOnly, 1>(stage, mw, nvc, e0, has_mask, straddle, cx, A);
            break;
        default: run_stage<DT, kUnfiltered, PASS>(stage, mw, nvc, e0, has_mask, straddle, cx, A); break;
    }
}

// The warp's r-th largest thread maximum (as an order key; 0 if fewer than r
// lanes have one).
__device__ __forceinline__ uint32_t warp_rth_key(uint32_t kv, int r) {
    uint32_t kth = 0;
    const int lane = threadIdx.x & 31;
    for (int i = 0; i < r; ++i) {
        kth = __reduce_max_sync(0xFFFFFFFFu, kv);
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, kv == kth);
        if (lane == __ffs(hit) - 1) kv = 0;
    }
    return kth;
}

}  // namespace

__device__ unsigned int g_sample_row_status;

template <int DT>
__global__ void __launch_bounds__(kRowThreads, 2) sample_row_kernel(SampleArgs a) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint4 *stages = reinterpret_cast<uint4 *>(smem);
    uint32_t *masks = reinterpret_cast<uint32_t *>(smem + kStages * kStageVec * 16);
    uint64_t *cand = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(masks) + kStages * kStageWords * 4);
    Hist &hist = *reinterpret_cast<Hist *>(reinterpret_cast<uint8_t *>(cand) + kCandCap * 8);
    RowCtl &ctl = *reinterpret_cast<RowCtl *>(reinterpret_cast<uint8_t *>(&hist) + sizeof(Hist));

    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t V = (int32_t)a.V;
    const uint8_t *rp = reinterpret_cast<const uint8_t *>(a.logits) + (size_t)row * a.stride * E::SIZE;
    const int32_t *mrow = a.mask ? a.mask + (size_t)row * a.mstride : nullptr;
    const bool has_mask = mrow != nullptr;
    const Slice32 g = make_slice32<AE, E::SIZE>(rp, V, 0, 1);  // head, nvec, tail of the row
    const int nchunks = (g.nvec + kStageVec - 1) / kStageVec;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.full[s], 1 + 32);  // the producer's expect-tx + one cp.async arrival per lane
            mbar_init(&ctl.empty[s], kCW);
        }
        ctl.ncand = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kCW) {
        // ---------------------------------------------------------- producer
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % kStages, k = c / kStages;
            if (k > 0) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait_bounded(&ctl.empty[s], (uint32_t)(k - 1) & 1u, &g_sample_row_status);
                if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) break;
            }
            const int32_t v0 = c * kStageVec;
            const int32_t nvc = min(kStageVec, g.nvec - v0);
            const int32_t e0 = g.head + v0 * AE;
            if (lane == 0) {
                const uint32_t bytes = (uint32_t)nvc * 16u;
                mbar_arrive_expect_tx(&ctl.full[s], bytes);
                bulk_g2s(stages + (size_t)s * kStageVec, rp + (size_t)e0 * E::SIZE, bytes, &ctl.full[s]);
            }
            if (has_mask) {
                const int32_t w0 = e0 >> 5, nw = ((e0 + nvc * AE - 1) >> 5) - w0 + 1;
                uint32_t *dst = masks + s * kStageWords;
                for (int32_t w = lane; w < nw; w += 32) cp_async_4(dst + w, mrow + w0 + w);
            }
            cp_async_mbar_arrive(&ctl.full[s]);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const RowParams rpm = row_params(a, row);
    const bool tau_on = rpm.k_on && (rpm.K + kCW - 1) / kCW <= kTauMaxR;
    const bool push_on = rpm.filtered && (tau_on || rpm.m_on);
    int mode;
    if (rpm.greedy) mode = kGreedy;
    else if (rpm.unfiltered) mode = kUnfiltered;
    else if (push_on) mode = rpm.p_on ? kFilterZ : kFilter;
    else mode = kZOnly;
    const int r_tau = tau_on ? (rpm.K + kCW - 1) / kCW : 0;
    // a vector's AE mask bits cross a word boundary only when the row start is
    // not 16-byte aligned (AE divides 32)
    const bool straddle = g.head != 0;

    Ctx cx;
    cx.row = row;
    cx.T = rpm.T;
    cx.invT = rpm.invT;
    cx.c2 = rpm.c2;
    cx.theta = -INFINITY;
    cx.ref = 0.f;
    cx.seed = a.seed;
    cx.offset = a.offset;
    cx.cand = cand;
    cx.ncand = &ctl.ncand;
    Acc A = {-INFINITY, 0xFFFFFFFFu, 0.f, 0.f, 0.f, -INFINITY, 0xFFFFFFFFu, -INFINITY};

    // the row's unaligned head and tail elements (fewer than AE each): plain loads
    float hx = -INFINITY;
    uint32_t he = 0;
    {
        int32_t e = -1;
        if (tid < g.head) e = tid;
        else if (tid >= kCT - g.tail) e = g.head + g.nvec * AE + (tid - (kCT - g.tail));
        if (e >= 0) {
            float x = E::load1(rp, e);
            if (has_mask && !(((uint32_t)__ldg(mrow + (e >> 5)) >> (e & 31)) & 1u)) x = -INFINITY;
            hx = x;
            he = (uint32_t)e;
            const bool z = mode == kFilterZ || mode == kZOnly;
            if (z) accumulate<1, true>(&hx, he, cx.c2, A);
            else accumulate<1, false>(&hx, he, cx.c2, A);
        }
    }

    auto stage_ptr = [&](int s) { return stages + (size_t)s * kStageVec; };
    auto wait_full = [&](int c) {
        return mbar_wait_bounded(&ctl.full[c % kStages], (uint32_t)(c / kStages) & 1u, &g_sample_row_status);
    };
    auto release = [&](int c) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[c % kStages]);
    };
    // publish this warp's bound and maximum, then read everyone's
    auto refresh = [&]() {
        const uint32_t kv = A.mx > -INFINITY ? okey(A.mx) : 0u;
        const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, kv);
        if (tau_on) {
            const uint32_t kth = warp_rth_key(kv, r_tau);
            if (lane == 0) reinterpret_cast<volatile float *>(ctl.wtau)[warp] = kth ? okey_value(kth) : -INFINITY;
        }
        if (lane == 0) reinterpret_cast<volatile float *>(ctl.wmax)[warp] = wk ? okey_value(wk) : -INFINITY;
        __syncwarp();
        float t = INFINITY, mm = -INFINITY;
#pragma unroll
        for (int i = 0; i < kCW; ++i) {
            t = fminf(t, reinterpret_cast<volatile float *>(ctl.wtau)[i]);
            mm = fmaxf(mm, reinterpret_cast<volatile float *>(ctl.wmax)[i]);
        }
        float th = tau_on ? t : -INFINITY;
        if (rpm.m_on && mm > -INFINITY) th = fmaxf(th, min_p_cut(mm, rpm.T, rpm.MP));
        cx.theta = th;
        return mm;
    };

    bool ok = true;
    // ---- stage 0: accumulate, seed the threshold, then push / draw
    if (nchunks > 0) {
        ok = wait_full(0);
        const int nvc = min(kStageVec, g.nvec);
        run_stage_mode<DT, 1>(mode, stage_ptr(0), masks, nvc, (uint32_t)g.head, has_mask, straddle, cx, A);
    }
    if (tid == 0) {
        for (int i = 0; i < kCW; ++i) {
            ctl.wtau[i] = -INFINITY;
            ctl.wmax[i] = -INFINITY;
        }
    }
    CSync::sync();
    refresh();
    CSync::sync();
    const float ref = refresh();  // every warp has published: the first stage's maximum
    cx.ref = ref > -INFINITY ? ref : 0.f;
    if (mode == kFilter || mode == kFilterZ || mode == kUnfiltered) {
        if (nchunks > 0) {
            const int nvc = min(kStageVec, g.nvec);
            run_stage_mode<DT, 2>(mode, stage_ptr(0), masks, nvc, (uint32_t)g.head, has_mask, straddle, cx, A);
        }
        if (hx > -INFINITY) {  // this thread's head / tail element
            if (mode == kUnfiltered) gumbel<1>(&hx, he, hx, cx, A);
            else push<1>(&hx, he, hx, cx);
        }
    }
    if (nchunks > 0) release(0);

    // ---- the remaining stages: one pass each
    for (int c = 1; c < nchunks; ++c) {
        const int s = c % kStages;
        if (ok) ok = wait_full(c);
        const int32_t v0 = c * kStageVec;
        const int nvc = min(kStageVec, g.nvec - v0);
        run_stage_mode<DT, 3>(mode, stage_ptr(s), masks + s * kStageWords, nvc, (uint32_t)(g.head + v0 * AE), has_mask,
                              straddle, cx, A);
        release(c);
        if ((mode == kFilter || mode == kFilterZ) && (c % kRefresh) == 0) refresh();
    }

    // ---- end of the row: warp reductions, then one combine
    {
        const uint32_t kv = A.mx > -INFINITY ? okey(A.mx) : 0u;
        const uint32_t wkv = __reduce_max_sync(0xFFFFFFFFu, kv);
        const uint32_t wmi = __reduce_min_sync(0xFFFFFFFFu, (kv == wkv && wkv) ? A.mi : 0xFFFFFFFFu);
        const float wm = wkv ? okey_value(wkv) : -INFINITY;
        float wz = 0.f;
        if (mode == kFilterZ || mode == kZOnly)
            wz = warp_sum_f32(A.mx > -INFINITY ? (A.z0 + A.z1) * ex2_approx((A.mx - wm) * rpm.c2) : 0.f);
        uint64_t wb = 0;
        if (mode == kUnfiltered) wb = warp_max_u64(A.sbest > -INFINITY ? rank_key(A.sbest, A.sbi) : 0ull);
        uint32_t kth = 0;
        if (tau_on) kth = warp_rth_key(kv, r_tau);
        if (lane == 0) {
            ctl.wkey[warp] = wkv ? (((uint64_t)wkv << 32) | (uint64_t)(0xFFFFFFFFu - wmi)) : 0ull;
            ctl.wz[warp] = wz;
            ctl.wbest[warp] = wb;
            ctl.wtau[warp] = kth ? okey_value(kth) : -INFINITY;
        }
    }
    CSync::sync();
    uint64_t gkey = 0, best = 0;
    float tau = INFINITY;
#pragma unroll
    for (int i = 0; i < kCW; ++i) {
        gkey = ctl.wkey[i] > gkey ? ctl.wkey[i] : gkey;
        best = ctl.wbest[i] > best ? ctl.wbest[i] : best;
        tau = fminf(tau, ctl.wtau[i]);
    }
    const float m = gkey ? rank_key_value(gkey) : -INFINITY;
    const uint32_t amax = gkey ? rank_key_index(gkey) : 0u;
    float Z = 0.f;
    if (mode == kFilterZ || mode == kZOnly) {
#pragma unroll
        for (int i = 0; i < kCW; ++i)
            if (ctl.wkey[i]) Z += ctl.wz[i] * ex2_approx((rank_key_value(ctl.wkey[i]) - m) * rpm.c2);
    }
    int64_t token = -1;
    float vstar = -INFINITY;
    if (!ok) {
        token = -1;  // a bounded wait ran out: the status flag is set
        vstar = __int_as_float(0x7FC00000);
    } else if (!gkey) {
        vstar = __int_as_float(0x7FC00000);
    } else if (mode == kGreedy) {
        token = amax;
        vstar = m;
    } else if (mode == kUnfiltered) {
        token = rank_key_index(best);
    } else {
        const float v_m = rpm.m_on ? min_p_cut(m, rpm.T, rpm.MP) : -INFINITY;
        bool done = false;
        const uint32_t n_all = ctl.ncand;
        if (mode != kZOnly && n_all <= (uint32_t)kCandCap && Z == Z) {
            const float theta = fmaxf(tau_on ? tau : -INFINITY, v_m);
            // ordered in-place compaction of the candidates >= theta
            uint32_t written = 0;
            for (uint32_t t0 = 0; t0 < n_all; t0 += kCT) {
                const uint32_t i = t0 + (uint32_t)tid;
                uint64_t key = 0;
                bool keep = false;
                if (i < n_all) {
                    key = cand[i];
                    keep = rank_key_value(key) >= theta;
                }
                uint32_t tile_total = 0;
                const uint32_t pos = written + block_excl_scan_u32<CSync>(keep ? 1u : 0u, ctl.sel.sc, tile_total);
                CSync::sync();
                if (keep) cand[pos] = key;
                written += tile_total;
            }
            CSync::sync();
            done = select_from_candidates<CSync>(a, row, rpm, cand, written, (uint32_t)kCandCap, theta, v_m, m,
                                                 (double)Z, hist, ctl.sel, token, vstar);
        }
        if (!done) {
            if (!(Z == Z)) {  // a NaN logit reached the normaliser: recompute it with NaN as -inf
                float zt = 0.f;
                for (int32_t i = tid; i < V; i += kCT) {
                    float x = E::load1(rp, i);
                    if (has_mask && !(((uint32_t)__ldg(mrow + (i >> 5)) >> (i & 31)) & 1u)) x = -INFINITY;
                    if (x == x && x > -INFINITY) zt += ex2_approx((x - m) * rpm.c2);
                }
                Z = block_sum_f32<CSync>(zt, ctl.sel.sc);
            }
            general_path<DT, CSync>(a, row, rpm, m, amax, (double)Z, v_m, hist, ctl.sel, token, vstar);
        }
    }
    if (tid == 0) {
        a.tokens[row] = token;
        if (a.vstar_out) a.vstar_out[row] = vstar;
    }
}

unsigned int *sample_row_status_ptr() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sample_row_status) != cudaSuccess) return nullptr;
    return reinterpret_cast<unsigned int *>(p);
}

size_t sample_row_smem_bytes() {
    return (size_t)kStages * kStageVec * 16 + (size_t)kStages * kStageWords * 4 + (size_t)kCandCap * 8 + sizeof(Hist) +
           sizeof(RowCtl);
}

int sample_row_launch(const SampleArgs &args, int dtype, cudaStream_t st) {
    const void *fns[3] = {(const void *)sample_row_kernel<0>, (const void *)sample_row_kernel<1>,
                          (const void *)sample_row_kernel<2>};
    const void *fn = fns[dtype];
    const size_t smem = sample_row_smem_bytes();
    if (prepare_kernel(fn, smem, 1) != 0) return -1;
    SampleArgs a = args;
    void *params[] = {&a};
    return cudaLaunchKernel(fn, dim3((unsigned)args.B), dim3(kRowThreads), params, smem, st) == cudaSuccess ? 0 : -1;
}

}  // namespace tsa
