// sample, one CTA per row (logits-processor, "API" and "Method";
// logits-mask-xpu, "Method" for top_k == 1), for batches with enough rows to
// occupy the GPU.
//
// A producer warp streams the row through a ring of shared-memory stages: each
// stage is one 1-D bulk copy (cp.async.bulk) of up to kStageVec 16-byte
// vectors plus the mask words that cover them (4-byte cp.async), both
// completing on the stage's "full" mbarrier; the eleven consumer warps release
// a stage on its "empty" mbarrier.  Every logit is read from HBM once.  A
// row's time is set by the latency of its warps' dependent instructions more
// than by the SM's issue rate, so the CTA is made as wide as two CTAs per SM
// allow: eleven consumers and one producer (384 threads, at most 85 registers
// a thread), with four 22 KB stages.  The row's short last stage is padded
// with -inf by the producer, so that every stage runs the same code, and a
// row whose first stage is read twice asks for the rest of the row only once
// that stage has landed.
//
// Each consumer thread keeps, over the vectors it reads (vector j of a stage
// goes to consumer thread j mod 352): the maximum (and its lowest index, where
// no candidate list will hold it), and the sum of 2^((l - ref) log2(e) / T)
// against a reference ref that starts at the first stage's maximum and moves
// only when a term would pass 2^8, so the largest terms have small exponents
// (and small rounding).  Each term's exponent is one fma, l c2 + RN(-ref c2);
// the rounding of ref c2 scales every term alike, and is removed exactly when
// the sums are combined.  A keep-threshold lower bound theta rises as the row
// streams by:
//   - top-k: each warp's r-th largest thread maximum, r = ceil(k / 11), is a
//     logit with at least r - 1 larger ones among distinct thread maxima in
//     that warp, so the minimum over the 11 warps has at least k logits of
//     the row at or above it (skipped while the min-p cut dominates it);
//   - min-p: the cut m + T ln(min_p) at the largest maximum seen so far,
//     which is below the cut at the row maximum.
// Both only grow, so reading another warp's published value late is safe.
// Every allowed logit >= theta at the time it is read is pushed as a rank key
// into a shared candidate list; since the final threshold is at least every
// earlier one, the list holds every logit >= the final theta.  The first
// stage is read twice (once to seed theta, once to push).  Unfiltered rows
// draw Gumbel-max in the stream instead, each thread pruning tokens that
// cannot beat its own or its warp's best score.  At the end the warps reduce
// the row's maximum, argmax and normaliser, and the first 256 threads resolve
// the exact keep-threshold and the draw from the candidates; a row with no
// usable threshold (top-p alone), an overflowing list or a NaN in the
// normaliser takes the general path, which re-reads the row.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "tsa_device.cuh"
#include "tsa_host.h"
#include "tsa_sample_common.cuh"
#include "tsa_select.cuh"

namespace tsa {

using namespace sample_detail;

// each translation unit that includes this header has its own status word
static __device__ unsigned int g_sample_row_status;

namespace {
constexpr int kRowWarps = 12;
constexpr int kCW = kRowWarps - 1;           // consumer warps
constexpr int kCT = kCW * 32;                // consumer threads (threadIdx.x < kCT)
constexpr int kRowThreads = kRowWarps * 32;  // plus the producer warp
// the selection steps after the stream run on the first kThreads threads
static_assert(kRowThreads >= kThreads, "the selection steps need kThreads threads");
using SSync = NamedSync<2, kThreads>;
constexpr int kStages = 4;
constexpr int kVecPerThread = 4;
constexpr int kStageVec = kCT * kVecPerThread;  // 16-byte vectors per stage
static_assert(kStages * kStageVec * 16 >= (int)(sizeof(GHist) + sizeof(Hist)), "the selection's histograms reuse the stage ring");
// mask words one stage may span (8 elements per vector, unaligned start), plus
// one spare word read by the straddling bit extraction
constexpr int kStageWords = (kStageVec * 8 / 32 + 2 + 7) & ~7;
constexpr int kCandCap = 2048;
// the window path's first pass lists keys in the candidate list's first
// kRelistCap slots while its bin counts (kWinBins 32-bit words) take the rest
constexpr int kRelistCap = kCandCap - kWinBins / 2;
static_assert(kRelistCap >= 512, "the window bins leave the listing too little room");
static_assert(kCandCap * 8 >= kCW * 32 * kVecPerThread * 2, "the unfiltered draw queues reuse the candidate list");
// rows that read their first stage twice request this many stages before the
// first one lands, the rest after it
constexpr int kIssueAhead = 1;
constexpr int kEarly = 4;    // the threshold is refreshed after each of the first kEarly stages,
constexpr int kRefresh = 8;  // then after every kRefresh-th
// The normaliser sums 2^((l - rf) c2) against a reference rf that moves up
// only when a value passes it by kZSpan in the exponent: terms stay below
// 2^kZSpan, so a term's exponent, rounded once, is off by at most 2^-22 and
// the term by at most 1.7e-7 of itself.  rf starts at the first stage's block
// maximum, so the rescale is rare.
constexpr float kZSpan = 8.f;
constexpr int kTauMaxR = 32;  // largest r = ceil(k / kCW) for which the top-k bound is formed

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
    uint32_t ubest[kCW];  // unfiltered rows: each warp's best perturbed score so far (order key, 0 for none)
    // the window path
    uint32_t win_bk, win_plo, win_lfirst;  // first bins: top-k cut; U >= p Z; L >= p Z
    uint32_t win_lo, win_hi, win_clo, win_cnt, win_fail, win_all, win_gather;
    uint32_t win_nr, win_nb, win_nw;  // keys pass A and pass B listed; window keys of a gathered list
    float wmh[kCW], wml[kCW], wmin[kCW];
    float win_l[kWarps], win_u[kWarps];
    uint32_t win_c[kWarps], win_n[kWarps];
};

struct Acc {
    float mx;                // running maximum
    uint32_t mi;             // its lowest index
    unsigned long long zp;   // sum of 2^((l - rf) c2 + dz): two fp32 partial sums, packed
    float nm;                // RN(-rf c2); -inf while no reference is set (terms add 0)
    float dz;                // rf c2 + nm, exact: the bias every term of zp carries
    float rf;                // the normaliser's reference
    float rhi;               // rf + kZSpan / c2: the reference moves up only past this
    float sbest;   // unfiltered: best score (l - ref) / T + G of the tokens this thread drew
    uint32_t sbi;
    float gcut;    // unfiltered: logits below it cannot beat sbest
    float wbest, wcut;  // unfiltered: the same for the warp's best score (a prune bound only)
    bool full;          // a push of this thread found the candidate list full
};

struct Ctx {
    int64_t row;
    float T, invT, c2, theta, ref;
    float zspan;  // kZSpan / c2
    float mm;  // the row maximum as last read from the warps' published ones
    uint64_t seed, offset;
    uint64_t *cand;
    uint32_t ncand_s;  // shared-memory address of the candidate counter
    uint16_t *gq;      // this warp's draw queue
    const float4 *mtab;  // this lane's copy of the mask bias table (f32 rows)
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Two fp32 lanes in one 64-bit register, for the packed f32x2 arithmetic.
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The mask as an addition on the FMA pipe (f32 rows): the four mask bits of a
// 16-byte vector select a float4 of biases, -0.0 for an allowed element (x +
// -0.0 is x, bit for bit) and -inf for a disallowed one (a finite x becomes
// -inf; a disallowed NaN or +inf becomes NaN, which no maximum, candidate or
// draw takes, and which sends the normaliser to the exact recomputation).
// Two packed adds per vector replace a bit test and a select per element on
// the ALU pipe.  The table holds 16 entries in 8 interleaved copies (entry e
// of copy c at float4 8 e + c), and lane l reads copy l mod 8, so the eight
// lanes of each 128-bit load phase always hit different banks.
constexpr int kMaskTabCopies = 8;
constexpr int kMaskTabEntries = 16 * kMaskTabCopies;
__device__ __forceinline__ void init_mask_tab(float4 *tab) {
    for (int i = threadIdx.x; i < kMaskTabEntries; i += blockDim.x) {
        const int e = i / kMaskTabCopies;
        const float on = -0.0f, off = -INFINITY;
        tab[i] = make_float4(e & 1 ? on : off, e & 2 ? on : off, e & 4 ? on : off, e & 8 ? on : off);
    }
}
__device__ __forceinline__ void add_bias(uint4 &v, const float4 *mtab, uint32_t bits4) {
    const float4 b = mtab[(bits4 & 15u) * kMaskTabCopies];
    unsigned long long lo = f2_pack(__uint_as_float(v.x), __uint_as_float(v.y));
    unsigned long long hi = f2_pack(__uint_as_float(v.z), __uint_as_float(v.w));
    lo = f2_add(lo, f2_pack(b.x, b.y));
    hi = f2_add(hi, f2_pack(b.z, b.w));
    float a0, a1, a2, a3;
    f2_unpack(lo, a0, a1);
    f2_unpack(hi, a2, a3);
    v = make_uint4(__float_as_uint(a0), __float_as_uint(a1), __float_as_uint(a2), __float_as_uint(a3));
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (the arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Set the normaliser's reference to v (the first stage's block maximum, or
// -inf if it had no allowed finite logit) and clear the sums.
__device__ __forceinline__ void set_ref(float v, float c2, float zspan, Acc &A) {
    A.zp = 0ull;
    if (v > -INFINITY) {
        A.rf = v;
        A.nm = __fmul_rn(-v, c2);
        A.dz = fmaf(v, c2, A.nm);
        A.rhi = v + zspan;
    } else {  // the first finite value moves the reference
        A.rf = -INFINITY;
        A.nm = -INFINITY;
        A.dz = 0.f;
        A.rhi = -INFINITY;
    }
}

// Move the normaliser's reference up to v when v passes rf + kZSpan / c2:
// the sums so far are rescaled by 2^((rf - v) c2 + dz' - dz), which also
// moves them onto the new bias dz'.
__device__ __forceinline__ void move_ref(float v, float c2, float zspan, Acc &A) {
    const float nm = __fmul_rn(-v, c2);
    const float dz = fmaf(v, c2, nm);
    if (A.rf > -INFINITY) {
        const float s = ex2_diff(A.rf, v, c2, dz - A.dz);
        A.zp = f2_mul(A.zp, f2_pack(s, s));
    } else {
        A.zp = 0ull;
    }
    A.rf = v;
    A.nm = nm;
    A.dz = dz;
    A.rhi = v + zspan;
}

// The running maximum and its lowest index over one element (the row's
// unaligned head or tail element of this thread).
__device__ __forceinline__ void accumulate1(float x, uint32_t e, Acc &A) {
    if (x > A.mx) {
        A.mx = x;
        A.mi = e;
    }
}
// That element's normaliser term (-inf adds 0; NaN poisons the sum, which
// sends the row to the exact recomputation).
__device__ __forceinline__ void z_one(float x, float c2, float zspan, Acc &A) {
    if (x > A.rhi) move_ref(x, c2, zspan, A);
    float z0, z1;
    f2_unpack(A.zp, z0, z1);
    z0 += ex2_approx(fmaf(x, c2, A.nm));
    A.zp = f2_pack(z0, z1);
}

__device__ __forceinline__ uint32_t atomic_add_shared(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}

// Push every logit of the group that is >= theta: one shared atomic per
// candidate, by the (few) lanes that have one.
template <int N>
// A thread whose push lands past the list's capacity stops pushing (the list
// is incomplete from then on, and the count already shows it): a flat row
// would otherwise send every token through the counter's atomic.
__device__ __forceinline__ void push(const float *x, uint32_t e0, float vmax, const Ctx &cx, Acc &A) {
    if (!(vmax >= cx.theta) || A.full) return;
#pragma unroll
    for (int t = 0; t < N; ++t)
        if (x[t] >= cx.theta && x[t] > -INFINITY) {
            const uint32_t pos = atomic_add_shared(cx.ncand_s, 1u);
            if (pos < (uint32_t)kCandCap) cx.cand[pos] = rank_key(x[t], e0 + (uint32_t)t);
            else A.full = true;
        }
}

// Unfiltered draw: the group's tokens that can still beat the thread's best
// perturbed score.
template <int N>
__device__ __forceinline__ void gumbel(const float *x, uint32_t e0, float vmax, const Ctx &cx, Acc &A) {
    const float cut0 = fmaxf(A.gcut, A.wcut);
    if (!(vmax >= cut0)) return;
    uint32_t bits = 0;  // the elements that can still win
#pragma unroll
    for (int t = 0; t < N; ++t) bits |= (x[t] >= cut0 && x[t] > -INFINITY) ? 1u << t : 0u;
    if (N >= 4 && (e0 & 3u) == 0u) {
        // an aligned vector (every vector of a row whose start is 16-byte
        // aligned): whole groups of four tokens, slots known at compile time
#pragma unroll
        for (int gq = 0; gq < N / 4; ++gq) {
            const uint32_t gm = (bits >> (4 * gq)) & 0xFu;
            if (!gm) continue;
            const uint32_t q = (e0 >> 2) + (uint32_t)gq;
            const uint4 blk = token_block(cx.seed, cx.offset, (uint32_t)cx.row, q);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (!((gm >> k) & 1u)) continue;
                const float xt = x[4 * gq + k];
                if (!(xt >= fmaxf(A.gcut, A.wcut))) continue;  // the cut may have risen in this vector
                const uint32_t e = q * 4u + (uint32_t)k;
                const uint32_t word = k == 0 ? blk.x : (k == 1 ? blk.y : (k == 2 ? blk.z : blk.w));
                const float srel = (xt - cx.ref) * cx.invT;
                const float need = fmaxf(A.sbest, A.wbest) - srel;  // the Gumbel value this token must beat
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
        return;
    }
    // otherwise the vector's groups of four consecutive tokens, one Philox
    // block each, in a rolled loop (one copy of the block code)
    const uint32_t q0 = e0 >> 2;
    const int ng = (int)(((e0 + (uint32_t)N - 1u) >> 2) - q0) + 1;
#pragma unroll 1
    for (int gq = 0; gq < ng; ++gq) {
        const uint32_t q = q0 + (uint32_t)gq;
        const int tq = (int)(q * 4u) - (int)e0;  // slot of the group's first token (> -4)
        const uint32_t gm = bits & (tq >= 0 ? 0xFu << tq : 0xFu >> -tq);
        if (!gm) continue;
        const uint4 blk = token_block(cx.seed, cx.offset, (uint32_t)cx.row, q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int t = tq + k;
            if (t < 0 || t >= N || !((gm >> t) & 1u)) continue;
            float xt = x[0];
#pragma unroll
            for (int u = 1; u < N; ++u) xt = t == u ? x[u] : xt;
            if (!(xt >= fmaxf(A.gcut, A.wcut))) continue;  // the cut may have risen in this vector
            const uint32_t e = q * 4u + (uint32_t)k;
            const uint32_t word = k == 0 ? blk.x : (k == 1 ? blk.y : (k == 2 ? blk.z : blk.w));
            const float srel = (xt - cx.ref) * cx.invT;
            const float need = fmaxf(A.sbest, A.wbest) - srel;  // the Gumbel value this token must beat
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
}

// Maximum of n floats (NaN never wins unless all are NaN).
template <int N>
__device__ __forceinline__ float max_n(const float *x) {
    if (N == 4) return fmaxf(fmax3(x[0], x[1], x[2]), x[3]);
    float m = x[0];
#pragma unroll
    for (int t = 1; t < N; ++t) m = fmaxf(m, x[t]);
    return m;
}

// The maximum of 16 floats in eight 3-input max instructions (NaN never wins
// unless all are NaN).
__device__ __forceinline__ float max16(const float *f) {
    const float a0 = fmax3(f[0], f[1], f[2]), a1 = fmax3(f[3], f[4], f[5]), a2 = fmax3(f[6], f[7], f[8]);
    const float a3 = fmax3(f[9], f[10], f[11]), a4 = fmax3(f[12], f[13], f[14]);
    return fmaxf(fmax3(a0, a1, a2), fmax3(a3, a4, f[15]));
}
static_assert(kVecPerThread * 4 == 16, "a group is 16 elements: four f32 vectors or two 16-bit ones");

// This thread's masked 16-byte vectors of one stage (vector i is stage vector
// threadIdx.x + i kCT).  FULL stages hold kStageVec vectors; in the row's
// last stage a vector past its end reads as -inf, so that the lanes of a warp
// stay together (push and the draw queue are warp-collective).
template <int DT, bool FULL, int MASK>
__device__ __forceinline__ void load_vecs(const uint4 *stage, const uint32_t *mw, int nvc, uint32_t e0,
                                          const float4 *mtab, uint4 (&v)[kVecPerThread]) {
    constexpr int AE = Elem<DT>::AE;
    constexpr uint32_t kFull = (1u << AE) - 1u;
    constexpr uint32_t kNinf = DT == 0 ? 0xFF800000u : (DT == 1 ? 0xFC00FC00u : 0xFF80FF80u);
    // consecutive vectors of a thread are kCT * AE elements apart, a whole
    // number of mask words, so they share the bit offset within their word
    constexpr int kWordStep = kCT * AE / 32;
    static_assert(kCT * AE % 32 == 0, "vector stride must be whole mask words");
    const uint32_t rel = (e0 & 31u) + threadIdx.x * AE;
    const uint32_t k0 = rel >> 5, sh = rel & 31u;
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
        const int j = (int)threadIdx.x + i * kCT;
        if (FULL || j < nvc) {
            v[i] = stage[j];
            if (MASK && DT == 0) {
                // f32: the vector's four bits sit at sh .. sh + 3 of one word
                // (an aligned row start) or straddle two (MASK == 2)
                const uint32_t k = k0 + (uint32_t)(i * kWordStep);
                add_bias(v[i], mtab, MASK == 2 ? __funnelshift_r(mw[k], mw[k + 1], sh) : (mw[k] >> sh));
            } else if (MASK) {
                const uint32_t k = k0 + (uint32_t)(i * kWordStep);
                // MASK == 2: the row start is not 16-byte aligned and a
                // vector's bits may continue into the next word
                mask_vec<DT>(v[i], (MASK == 2 ? __funnelshift_r(mw[k], mw[k + 1], sh) : (mw[k] >> sh)) & kFull);
            }
        } else {
            v[i] = make_uint4(kNinf, kNinf, kNinf, kNinf);
        }
    }
}

// One stage's vectors of this thread, already masked in registers, kU at a
// time (four 4-element vectors, or two of 8).  PASS 1 accumulates only, PASS
// 2 pushes / draws only, PASS 3 does both.  A group's vectors are in
// increasing index order, so the first element equal to a new maximum is its
// lowest index.  The unfiltered draw queue re-reads its vectors from the
// stage, which must still be held.
template <int DT, int MODE, int PASS, int MASK>
__device__ __forceinline__ void run_groups(const uint4 (&v)[kVecPerThread], const uint4 *stage, const uint32_t *mw,
                                           uint32_t e0, const Ctx &cx, Acc &A) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    constexpr uint32_t kFull = (1u << AE) - 1u;
    constexpr bool kZ = MODE == kFilterZ || MODE == kZOnly;
    constexpr int kU = AE == 4 ? 4 : 2;
#pragma unroll
    for (int i0 = 0; i0 < kVecPerThread; i0 += kU) {
        float x[kU][AE];
        float vm[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) E::unpack(v[i0 + u], x[u]);
        float gm;
        if (MODE == kUnfiltered) {  // the draw queue needs every vector's maximum
#pragma unroll
            for (int u = 0; u < kU; ++u) vm[u] = max_n<AE>(x[u]);
            gm = vm[0];
#pragma unroll
            for (int u = 1; u < kU; ++u) gm = fmaxf(gm, vm[u]);
        } else {
            gm = max16(&x[0][0]);
        }
        const uint32_t eb = e0 + (uint32_t)((int)threadIdx.x + i0 * kCT) * AE;  // index of x[0][0]
        constexpr bool kPush = (PASS & 2) && (MODE == kFilter || MODE == kFilterZ);
        // The argmax is tracked only where no candidate list holds it (the
        // row maximum is always at or above theta, so a filtered row pushes
        // it); elsewhere the running maximum is one max instruction, since a
        // new maximum for some lane of a warp is not rare at all.
        constexpr bool kIdx = MODE == kGreedy || MODE == kZOnly;
        if (PASS & 1) {
            if (kIdx && gm > A.mx) {
                uint32_t off = 0xFFFFFFFFu;
#pragma unroll
                for (int u = kU - 1; u >= 0; --u)
#pragma unroll
                    for (int t = AE - 1; t >= 0; --t)
                        if (x[u][t] == gm) off = (uint32_t)(u * kCT * AE + t);
                A.mi = eb + off;
            }
            A.mx = fmaxf(A.mx, gm);
            if (kZ && gm > A.rhi) move_ref(gm, cx.c2, cx.zspan, A);  // rare: a lane's first values
        }
        if (kPush && gm >= cx.theta) {
#pragma unroll
            for (int u = 0; u < kU; ++u) push<AE>(x[u], eb + (uint32_t)(u * kCT * AE), max_n<AE>(x[u]), cx, A);
        }
        if ((PASS & 1) && kZ) {
            // 2^(x c2 - mx c2) in pairs: packed fma and add around the SFU
            const unsigned long long c2p = f2_pack(cx.c2, cx.c2), nmp = f2_pack(A.nm, A.nm);
#pragma unroll
            for (int u = 0; u < kU; ++u)
#pragma unroll
                for (int t = 0; t < AE; t += 2) {
                    float a0, a1;
                    f2_unpack(f2_fma(f2_pack(x[u][t], x[u][t + 1]), c2p, nmp), a0, a1);
                    A.zp = f2_add(A.zp, f2_pack(ex2_approx(a0), ex2_approx(a1)));
                }
        }
        if ((PASS & 2) && MODE == kUnfiltered) {
            // the vectors that can still beat the warp's best go to a queue
            // that the warp then draws densely, one vector a lane (a lane's
            // vectors rarely all qualify, but some lane's almost always does)
            const int lane = threadIdx.x & 31;
            const float cut = fmaxf(A.gcut, A.wcut);
            uint32_t nq = 0;
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const bool pred = vm[u] >= cut && vm[u] > -INFINITY;
                const uint32_t bal = __ballot_sync(0xFFFFFFFFu, pred);
                if (pred) cx.gq[nq + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)((int)threadIdx.x + (i0 + u) * kCT);
                nq += __popc(bal);
            }
            __syncwarp();
            for (uint32_t qi = lane; qi < nq; qi += 32) {
                const int j = cx.gq[qi];
                uint4 v = stage[j];
                if (MASK) {
                    const uint32_t rj = (e0 & 31u) + (uint32_t)j * AE;
                    const uint32_t k = rj >> 5, s2 = rj & 31u;
                    const uint32_t bits = MASK == 2 ? __funnelshift_r(mw[k], mw[k + 1], s2) : (mw[k] >> s2);
                    if (DT == 0) add_bias(v, cx.mtab, bits);
                    else mask_vec<DT>(v, bits & kFull);
                }
                float xx[AE];
                E::unpack(v, xx);
                gumbel<AE>(xx, e0 + (uint32_t)j * AE, max_n<AE>(xx), cx, A);
            }
            __syncwarp();
            const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, A.sbest > -INFINITY ? okey(A.sbest) : 0u);
            if (wk) {
                A.wbest = okey_value(wk);
                A.wcut = fmaf(A.wbest - kGumbelMax, cx.T, cx.ref);
            }
        }
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

// Threshold refresh: publish this warp's top-k bound and maximum, then set
// theta from every warp's latest published values (stale ones are lower).
struct Bound {
    bool tau_on, m_on;
    int r_tau;
    float tlnmp;  // T ln(min_p)
};
// The min-p cut at maximum m (min_p_cut): the same function serves the running
// cut and the final one; it is monotone in m, so the running cut never exceeds
// the final.
__device__ __forceinline__ float cut_at(float m, float tlnmp) { return min_p_cut(m, tlnmp); }
// The warp's top-k bound as an order key (0: none).  mref is a maximum of
// the row seen so far (the warp's own, or a later one read from the other
// warps).  When fewer than r lanes hold a maximum above the min-p cut at
// mref, the warp's
// r-th largest thread maximum is at or below that cut, which is at or below
// the row's final min-p cut, so it can never raise the keep-threshold and the
// r-step search is skipped.  The bound a warp publishes only has to be at or
// below its true r-th largest, which never falls; a warp that skips keeps its
// last published bound, so every threshold built from the bounds stays at or
// below the final one and the candidate list stays complete.
__device__ __forceinline__ uint32_t warp_tau_key(uint32_t kv, float mref, const Bound &bd) {
    if (!bd.tau_on) return 0u;
    if (bd.m_on && mref > -INFINITY) {
        const uint32_t ck = okey(cut_at(mref, bd.tlnmp));
        if (__popc(__ballot_sync(0xFFFFFFFFu, kv > ck)) < bd.r_tau) return 0u;
    }
    return warp_rth_key(kv, bd.r_tau);
}
__device__ __forceinline__ void publish_bound(RowCtl &ctl, const Acc &A, const Bound &bd, float mm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t kv = A.mx > -INFINITY ? okey(A.mx) : 0u;
    const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, kv);
    if (bd.tau_on) {
        // a warp that forms no bound keeps the one it published before: bounds
        // only grow, so an earlier one is still at or below its r-th largest
        const uint32_t kth = warp_tau_key(kv, fmaxf(wk ? okey_value(wk) : -INFINITY, mm), bd);
        if (lane == 0 && kth) reinterpret_cast<volatile float *>(ctl.wtau)[warp] = okey_value(kth);
    }
    if (lane == 0) reinterpret_cast<volatile float *>(ctl.wmax)[warp] = wk ? okey_value(wk) : -INFINITY;
}
__device__ __forceinline__ float read_bound(RowCtl &ctl, const Bound &bd, Ctx &cx) {
    float t = INFINITY, mm = -INFINITY;
#pragma unroll
    for (int i = 0; i < kCW; ++i) {
        t = fminf(t, reinterpret_cast<volatile float *>(ctl.wtau)[i]);
        mm = fmaxf(mm, reinterpret_cast<volatile float *>(ctl.wmax)[i]);
    }
    float th = bd.tau_on ? t : -INFINITY;
    if (bd.m_on && mm > -INFINITY) th = fmaxf(th, cut_at(mm, bd.tlnmp));
    cx.theta = th;
    cx.mm = mm;
    return mm;
}

// The row's stages, for one mode and mask layout.  Stage 0 is loaded into
// registers and its slot released at once; it is accumulated, theta is seeded
// from every consumer warp's maximum, and then it is pushed / drawn from the
// registers (unfiltered rows hold the slot: their draw queue re-reads it).
// The thread's head / tail element (hx at he, or -inf) goes with stage 0.
// Stages 1 .. nchunks-1 take one pass each.  A warp returns a stage's slot as
// soon as its vectors are in registers, so a CTA that shares its SM (and
// processes a stage more slowly) keeps as many bytes in flight as one that
// does not; unfiltered rows return it after the draw queue, greedy rows
// after their few instructions.
// Unfiltered rows: publish this warp's best perturbed score and take the
// best of every warp's as the prune bound.  Any score some token reaches
// bounds the row's best from below, so a token that cannot pass it cannot
// win (the bound is strict), and a late read of another warp's entry is only
// a weaker bound.
__device__ __forceinline__ void share_best(RowCtl &ctl, Acc &A, const Ctx &cx) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    volatile uint32_t *ub = ctl.ubest;
    if (lane == 0 && A.wbest > -INFINITY) ub[warp] = okey(A.wbest);
    const uint32_t k = __reduce_max_sync(0xFFFFFFFFu, lane < kCW ? ub[lane] : 0u);
    if (k && okey_value(k) > A.wbest) {
        A.wbest = okey_value(k);
        A.wcut = fmaf(A.wbest - kGumbelMax, cx.T, cx.ref);
    }
}

template <int DT, int MODE, int MK>
__device__ __forceinline__ bool stream_row(const uint4 *stages, const uint32_t *masks, RowCtl &ctl, int nchunks,
                                           int32_t nvec, int32_t head, const Bound &bd, Ctx &cx, Acc &A, bool ok,
                                           float hx, uint32_t he) {
    constexpr int AE = Elem<DT>::AE;
    constexpr bool kFilt = MODE == kFilter || MODE == kFilterZ;
    constexpr bool kTwo = kFilt || MODE == kUnfiltered;
    constexpr bool kZ = MODE == kFilterZ || MODE == kZOnly;
    // the unfiltered draw queue re-reads the stage; greedy rows measured
    // faster holding it through their (short) processing
    constexpr bool kEarlyFree = MODE != kUnfiltered && MODE != kGreedy;
    const int lane = threadIdx.x & 31;
    if (kFilt && nchunks > 0) {
        // Filtered rows read stage 0 twice through the loop's own stage code
        // (code run only once per row is fetched cold): iteration -1 with a
        // NaN theta (no logit, +inf included, compares >= it) and no
        // normaliser reference (its terms add 0) finds the stage's maximum;
        // theta is seeded and the reference set from every consumer warp's
        // maximum, and iteration 0 pushes it and sums its normaliser terms
        // (the maximum is idempotent).  Stage 0's slot is held until then.
        for (int c = -1; c < nchunks; ++c) {
            const int cs = c < 0 ? 0 : c;
            const int s = cs % kStages;
            if (c != 0 && ok) ok = mbar_wait_bounded(&ctl.full[s], (uint32_t)(cs / kStages) & 1u, &g_sample_row_status);
            const int32_t v0 = cs * kStageVec;
            const uint4 *st = stages + (size_t)s * kStageVec;
            const uint32_t *mw = masks + s * kStageWords;
            const uint32_t e0 = (uint32_t)(head + v0 * AE);
            const float th = cx.theta;
            if (c < 0) cx.theta = __int_as_float(0x7FFFFFFF);
            uint4 v[kVecPerThread];
            load_vecs<DT, true, MK>(st, mw, min(kStageVec, nvec - v0), e0, cx.mtab, v);
            if (c >= 0) {  // the stage is in registers: its slot goes back to the producer now
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.empty[s]);
            }
            run_groups<DT, MODE, 3, MK>(v, st, mw, e0, cx, A);
            cx.theta = th;
            if (c == 0) {
                if (hx > -INFINITY) push<1>(&hx, he, hx, cx, A);
                if (kZ) z_one(hx, cx.c2, cx.zspan, A);
            }
            if (c < 0 || (c > 0 && (c < kEarly || (c % kRefresh) == 0))) {
                publish_bound(ctl, A, bd, cx.mm);
                if (c < 0) CSync::sync();
                const float mm = read_bound(ctl, bd, cx);
                if (c < 0) {  // the first stage's maximum
                    cx.ref = mm > -INFINITY ? mm : 0.f;
                    if (kZ) set_ref(mm, cx.c2, cx.zspan, A);
                }
            }
        }
        return ok;
    }
    {
        uint4 v[kVecPerThread];
        const int nvc0 = min(kStageVec, nvec);
        if (nchunks > 0) {
            ok = mbar_wait_bounded(&ctl.full[0], 0u, &g_sample_row_status);
            if (nvc0 == kStageVec) load_vecs<DT, true, MK>(stages, masks, nvc0, (uint32_t)head, cx.mtab, v);
            else load_vecs<DT, false, MK>(stages, masks, nvc0, (uint32_t)head, cx.mtab, v);
            if (MODE != kUnfiltered) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.empty[0]);
            }
            run_groups<DT, MODE, 1, MK>(v, stages, masks, (uint32_t)head, cx, A);
        }
        publish_bound(ctl, A, bd, -INFINITY);
        CSync::sync();
        const float ref = read_bound(ctl, bd, cx);  // the first stage's maximum
        cx.ref = ref > -INFINITY ? ref : 0.f;
        if (kZ) {
            // the normaliser from the first stage's maximum on: stage 0's terms
            // again from the registers (they added 0 before), then the head /
            // tail element's
            set_ref(ref, cx.c2, cx.zspan, A);
            if (nchunks > 0) run_groups<DT, MODE, 1, MK>(v, stages, masks, (uint32_t)head, cx, A);
            z_one(hx, cx.c2, cx.zspan, A);
        }
        if (kTwo) {
            if (nchunks > 0) run_groups<DT, MODE, 2, MK>(v, stages, masks, (uint32_t)head, cx, A);
            if (hx > -INFINITY) {
                if (MODE == kUnfiltered) gumbel<1>(&hx, he, hx, cx, A);
                else push<1>(&hx, he, hx, cx, A);
            }
        }
        if (MODE == kUnfiltered && nchunks > 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[0]);
        }
    }
    for (int c = 1; c < nchunks; ++c) {
        const int s = c % kStages;
        if (ok) ok = mbar_wait_bounded(&ctl.full[s], (uint32_t)(c / kStages) & 1u, &g_sample_row_status);
        const int32_t v0 = c * kStageVec;
        const int nvc = min(kStageVec, nvec - v0);
        const uint4 *st = stages + (size_t)s * kStageVec;
        const uint32_t *mw = masks + s * kStageWords;
        const uint32_t e0 = (uint32_t)(head + v0 * AE);
        uint4 v[kVecPerThread];
        load_vecs<DT, true, MK>(st, mw, nvc, e0, cx.mtab, v);  // a short last stage is padded with -inf
        if (kEarlyFree) {  // the stage is in registers: its slot goes back to the producer now
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[s]);
        }
        run_groups<DT, MODE, 3, MK>(v, st, mw, e0, cx, A);
        if (!kEarlyFree) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[s]);
        }
        if (MODE == kUnfiltered) share_best(ctl, A, cx);
        if (kFilt && (c < kEarly || (c % kRefresh) == 0)) {
            publish_bound(ctl, A, bd, cx.mm);
            read_bound(ctl, bd, cx);
        }
    }
    return ok;
}


// The producer warp: request the row's stages into the ring as ring stages
// cbase .. cbase + nchunks - 1 (the ring's slots and barrier phases follow the
// ring stage), with the row's mask words.  A first read whose first stage is
// read twice (ahead) requests kIssueAhead stages, then the rest once the first
// has landed.  Returns false if a bounded wait ran out.
template <int DT>
__device__ __forceinline__ bool produce_row(uint4 *stages, uint32_t *masks, RowCtl &ctl, const uint8_t *rp,
                                            const int32_t *mrow, const Slice32 &g, int nchunks, int cbase, bool ahead) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    const int lane = threadIdx.x & 31;
    for (int c = 0; c < nchunks; ++c) {
        const int cg = cbase + c;
        const int s = cg % kStages, k = cg / kStages;
        if (k > 0) {
            bool w_ok = true;
            if (lane == 0) w_ok = mbar_wait_bounded(&ctl.empty[s], (uint32_t)(k - 1) & 1u, &g_sample_row_status);
            if (!__shfl_sync(0xFFFFFFFFu, w_ok ? 1 : 0, 0)) return false;
        }
        const int32_t v0 = c * kStageVec;
        if (ahead && c == kIssueAhead) {
            // rows whose first stage is read twice: let it land before the
            // rest of the row is requested, so that it is not queued behind
            // every row's later stages
            if (lane == 0) mbar_wait_bounded(&ctl.full[0], 0u, &g_sample_row_status);
            __syncwarp();
        }
        const int32_t nvc = min(kStageVec, g.nvec - v0);
        const int32_t e0 = g.head + v0 * AE;
        if (nvc < kStageVec) {
            // the row's last stage: the rest of the slot reads as -inf, so
            // that the consumers run the same code as for a full stage; the
            // proxy fence orders these stores before later bulk copies into
            // the same slot
            constexpr uint32_t kN = DT == 0 ? 0xFF800000u : (DT == 1 ? 0xFC00FC00u : 0xFF80FF80u);
            uint4 *dst = stages + (size_t)s * kStageVec;
            for (int32_t j = nvc + lane; j < kStageVec; j += 32) dst[j] = make_uint4(kN, kN, kN, kN);
            fence_proxy_async_smem();
            __syncwarp();  // ordered before lane 0's arrival (release) on the full barrier
        }
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)nvc * 16u;
            mbar_arrive_expect_tx(&ctl.full[s], bytes);
            bulk_g2s(stages + (size_t)s * kStageVec, rp + (size_t)e0 * E::SIZE, bytes, &ctl.full[s]);
        }
        if (mrow) {
            const int32_t w0 = e0 >> 5, nw = ((e0 + nvc * AE - 1) >> 5) - w0 + 1;
            uint32_t *dst = masks + s * kStageWords;
            for (int32_t w = lane; w < nw; w += 32) cp_async_4(dst + w, mrow + w0 + w);
        }
        cp_async_mbar_arrive(&ctl.full[s]);
    }
    return true;
}

// One more read of the row by the consumer warps, as ring stages cbase ..
// cbase + nchunks - 1.  f(x, eb, live, i) is called by the 32 lanes of a
// warp together, once per step over the threads' 16-byte vectors: x is the
// thread's vector i of the stage (masked elements and the last stage's
// padding read as -inf; NaN stays NaN), eb its first element's index, and
// live whether its maximum is >= thr; steps where no lane of the warp is live
// are skipped.  fe(st, mw, e0) runs on the whole warp after its steps of a
// stage, while the stage is still held.  A last call of f passes the thread's
// head or tail element (hx at he, the other slots -inf, i = -1).  Written for code size: one copy serves every mask layout (mk:
// 0 none, 1 aligned, 2 straddling), and the loop over the thread's vectors is
// not unrolled (these passes run after the stream, for rows with no usable
// candidate list, and large unrolled copies of them ran out of the
// instruction cache).
template <int DT, class F, class FE>
__device__ __forceinline__ bool consume_pass(const uint4 *stages, const uint32_t *masks, RowCtl &ctl, int nchunks,
                                             int32_t head, int cbase, int mk, const float4 *mtab, bool ok, float hx,
                                             uint32_t he, float thr, F &&f, FE &&fe) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    constexpr uint32_t kFull = (1u << AE) - 1u;
    const int lane = threadIdx.x & 31;
    for (int c = 0; c < nchunks; ++c) {
        const int cg = cbase + c, s = cg % kStages;
        if (ok) ok = mbar_wait_bounded(&ctl.full[s], (uint32_t)(cg / kStages) & 1u, &g_sample_row_status);
        const uint32_t e0 = (uint32_t)(head + c * kStageVec * AE);
        const uint4 *st = stages + (size_t)s * kStageVec;
        const uint32_t *mw = masks + s * kStageWords;
        const uint32_t rel = (e0 & 31u) + threadIdx.x * AE;
#pragma unroll 1
        for (int i = 0; i < kVecPerThread; ++i) {
            const int j = (int)threadIdx.x + i * kCT;
            uint4 v = st[j];
            if (mk) {
                const uint32_t k = (rel >> 5) + (uint32_t)(i * (kCT * AE / 32)), sh = rel & 31u;
                const uint32_t bits = mk == 2 ? __funnelshift_r(mw[k], mw[k + 1], sh) : (mw[k] >> sh);
                if (DT == 0) add_bias(v, mtab, bits);
                else mask_vec<DT>(v, bits & kFull);
            }
            float x[AE];
            E::unpack(v, x);
            const bool live = max_n<AE>(x) >= thr;
            if (!__any_sync(0xFFFFFFFFu, live)) continue;
            f(x, e0 + (uint32_t)j * AE, live, i);
        }
        fe(st, mw, e0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.empty[s]);
    }
    if (__any_sync(0xFFFFFFFFu, hx >= thr)) {
        float x[AE];
        x[0] = hx;
#pragma unroll
        for (int t = 1; t < AE; ++t) x[t] = -INFINITY;
        f(x, he, hx >= thr, -1);
    }
    return ok;
}

// Element t of a thread's vector, t known only at run time, without indexing
// the register array (which would move it to local memory).
template <int AE>
__device__ __forceinline__ float vec_elem(const float (&x)[AE], int t) {
    float r = x[0];
#pragma unroll
    for (int k = 1; k < AE; ++k) r = t == k ? x[k] : r;
    return r;
}

// Push the rank keys of the elements whose bits are set in this lane's
// vector, for the whole warp with one shared atomic (all 32 lanes call it
// together; positions in lane order, then element order).  Keys at positions
// >= cap are counted but not stored.  Returns, on every lane, whether the
// list has passed cap.
template <int AE>
__device__ __forceinline__ bool push_bits_warp(uint32_t bits, const float (&x)[AE], uint32_t eb, uint64_t *cand,
                                               uint32_t *ncand, uint32_t cap) {
    const int lane = threadIdx.x & 31;
    const uint32_t below = (1u << lane) - 1u;
    const uint32_t n = (uint32_t)__popc(bits);
    // the warp's exclusive prefix and total of n (n <= AE), bit plane by bit plane
    uint32_t pre = 0, tot = 0;
#pragma unroll
    for (int k = 0; (1 << k) <= AE; ++k) {
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, (n >> k) & 1u);
        pre += (uint32_t)__popc(bal & below) << k;
        tot += (uint32_t)__popc(bal) << k;
    }
    if (tot == 0u) return false;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(ncand, tot);
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    uint32_t pos = base + pre;
#pragma unroll
    for (int t = 0; t < AE; ++t)
        if ((bits >> t) & 1u) {
            if (pos < cap) cand[pos] = rank_key(x[t], eb + (uint32_t)t);
            ++pos;
        }
    return base + tot > cap;
}

// A filtered row with no complete candidate list, run by the whole CTA after
// the stream: the window path (see win_bin), two more reads of the row, the
// producer warp streaming it through the ring.  Pass A: the consumer warps
// count the tokens per bin; when theta_list is a number (the stream pushed
// candidates, and its list overflowed while its threshold was still low), the
// same read lists every allowed logit >= theta_list at the start of the
// candidate list, and if they fit there, listed is set and the caller
// resolves them.  Otherwise the first 256 threads find the window from the
// bins, and pass B gathers it (with every token above it, when all of them
// fit the list; else the tokens above it are summed and drawn from in the
// pass) for an exact resolution.  It recomputes the row's geometry rather
// than keep values from the stream alive, so that inlining it costs the
// stream loop no registers.  done and listed both false: the window cannot be
// resolved (it reaches the deep bin or holds more than the list), and the
// radix path runs.
struct WinOut {
    int64_t token;
    float vstar;
    uint32_t nlist;  // keys listed when listed is set
    bool done, listed;
};
template <int DT>
__device__ __forceinline__ WinOut window_path(const SampleArgs &a, const RowParams &rpm, float m, float Z, float v_m,
                                              float theta_list) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint4 *stages = reinterpret_cast<uint4 *>(smem);
    uint32_t *masks = reinterpret_cast<uint32_t *>(smem + kStages * kStageVec * 16);
    uint64_t *cand = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(masks) + kStages * kStageWords * 4);
    RowCtl &ctl = *reinterpret_cast<RowCtl *>(reinterpret_cast<uint8_t *>(cand) + kCandCap * 8);
    const float4 *mtab = reinterpret_cast<const float4 *>(reinterpret_cast<uint8_t *>(&ctl) + sizeof(RowCtl));
    uint32_t *whist = reinterpret_cast<uint32_t *>(cand + kRelistCap);  // the list's tail
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;
    const int32_t V = (int32_t)a.V;
    const uint8_t *rp = reinterpret_cast<const uint8_t *>(a.logits) + (size_t)row * a.stride * E::SIZE;
    const int32_t *mrow = a.mask ? a.mask + (size_t)row * a.mstride : nullptr;
    WinOut out{-1, -INFINITY, 0u, false, false};
    const Slice32 g = make_slice32<AE, E::SIZE>(rp, V, 0, 1);
    const int nchunks = (g.nvec + kStageVec - 1) / kStageVec;
    // the bins: e in [0, e_range) over kWinBins - 2 bins (deeper tokens weigh
    // < (1 - p) Z / (V + 1) with top-p on, and top-p drops them)
    float e_range = 62.f;
    if (rpm.p_on && rpm.P > 0.f) e_range = fminf(e_range, log2f((float)V + 1.f) - log2f(1.f - rpm.P) - log2f(Z) + 1.f);
    if (rpm.m_on) e_range = fminf(e_range, (m - v_m) * rpm.c2 + 1.f);
    e_range = fmaxf(e_range, 0.25f);
    const float S = (float)(kWinBins - 2) / e_range;
    const float c2S = rpm.c2 * S;
    const bool p_on = rpm.p_on;
    const bool relist = theta_list == theta_list;
    int cb = nchunks;  // the next ring stage
    const int mk = !mrow ? 0 : (g.head != 0 ? 2 : 1);
    const float4 *mtab_l = mtab + (lane & (kMaskTabCopies - 1));
    // this thread's head or tail element, as the stream read it (consumer
    // threads only: the tail index is formed from tid < kCT)
    float hx = -INFINITY;
    uint32_t he = 0;
    if (tid < kCT) {
        int32_t e = -1;
        if (tid < g.head) e = tid;
        else if (tid >= kCT - g.tail) e = g.head + g.nvec * AE + (tid - (kCT - g.tail));
        if (e >= 0) {
            float x = E::load1(rp, e);
            if (mrow && !(((uint32_t)__ldg(mrow + (e >> 5)) >> (e & 31)) & 1u)) x = -INFINITY;
            hx = x;
            he = (uint32_t)e;
        }
    }
    bool wok = true;
    // pass A: count the tokens >= the min-p cut per bin (with top-p, the deep
    // bin's tokens are dropped; else they are counted once a thread), and with
    // theta_list a number, list the logits >= theta_list
    for (int i = tid; i < kWinBins; i += kRowThreads) whist[i] = 0u;
    if (tid == 0) {
        ctl.win_bk = ctl.win_plo = ctl.win_lfirst = (uint32_t)kWinBins;
        ctl.win_fail = 0u;
        ctl.win_nr = 0u;
        ctl.win_nb = 0u;
    }
    __syncthreads();
    if (warp == kCW) {
        if (!produce_row<DT>(stages, masks, ctl, rp, mrow, g, nchunks, cb, false)) atomicOr(&g_sample_row_status, kStatusTimeout);
    } else {
        // groups below the min-p cut, and with top-p those whose tokens all
        // lie in the deep bin (one bin of slack for rounding), count nothing
        const float x_count = p_on ? fmaxf(v_m, m - (float)(kWinBins - 1) / c2S) : v_m;
        // the argmax class and the deep bin are counted in registers (a flat
        // row would otherwise send every token to one atomic)
        uint32_t top = 0, deep = 0;
        bool over = !relist;  // no listing, or this warp saw the list pass its share
        auto count = [&](const float (&x)[AE], uint32_t eb, bool live, int) {
            if (!over) {
                uint32_t bits = 0;
#pragma unroll
                for (int t = 0; t < AE; ++t) bits |= (x[t] >= theta_list && x[t] > -INFINITY) ? 1u << t : 0u;
                over = push_bits_warp<AE>(bits, x, eb, cand, &ctl.win_nr, (uint32_t)kRelistCap);
            }
            if (!live) return;
#pragma unroll
            for (int t = 0; t < AE; ++t) {
                const float xt = x[t];
                if (!(xt >= v_m) || !(xt > -INFINITY)) continue;
                const uint32_t b = win_bin(xt, m, c2S);
                if (b == 0u) {
                    ++top;
                } else if (b == (uint32_t)kWinBins - 1u) {
                    deep += p_on ? 0u : 1u;
                } else {
                    atomicAdd(&whist[b], 1u);
                }
            }
        };
        wok = consume_pass<DT>(stages, masks, ctl, nchunks, g.head, cb, mk, mtab_l, wok, hx, he,
                               relist ? fminf(theta_list, x_count) : x_count, count,
                               [](const uint4 *, const uint32_t *, uint32_t) {});
        top = __reduce_add_sync(0xFFFFFFFFu, top);
        deep = __reduce_add_sync(0xFFFFFFFFu, deep);
        if (lane == 0 && top) atomicAdd(&whist[0], top);
        if (lane == 0 && deep) atomicAdd(&whist[kWinBins - 1], deep);
    }
    cb += nchunks;
    __syncthreads();
    if (relist && ctl.win_nr <= (uint32_t)kRelistCap) {
        if (!wok) atomicOr(&g_sample_row_status, kStatusTimeout);
        out.listed = true;
        out.nlist = ctl.win_nr;
        return out;
    }
    if (warp == kCW) {
        if (!produce_row<DT>(stages, masks, ctl, rp, mrow, g, nchunks, cb, false)) atomicOr(&g_sample_row_status, kStatusTimeout);
        return out;
    }
    // the window: first 256 threads, 16 consecutive bins each, in fp32 (each
    // bound carries a relative margin of 1e-4, well above the rounding of the
    // sums and of e, so bounds stay bounds)
    if (tid < kThreads) {
        constexpr int kPer = kWinBins / kThreads;
        const uint32_t b0 = (uint32_t)tid * kPer;
        uint32_t c[kPer];
#pragma unroll
        for (int j = 0; j < kPer; j += 4) {
            const uint4 q = *reinterpret_cast<const uint4 *>(whist + b0 + j);
            c[j] = q.x;
            c[j + 1] = q.y;
            c[j + 2] = q.z;
            c[j + 3] = q.w;
        }
        // one token of bin b >= 1 weighs in (2^(-b / S), 2^(-(b - 1) / S)];
        // bin 0 (the argmax class) exactly 1; the deep bin at most 2^(-(kWinBins - 2) / S)
        const float r = exp2f(-1.f / S);
        const float w0 = exp2f(-(float)b0 / S);  // 2^(-b0 / S)
        uint32_t ct = 0;
        float lt = 0.f, ut = 0.f;
        {
            float wb = w0;  // 2^(-b / S)
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const uint32_t b = b0 + j;
                const float wl = b == 0 ? 1.f : (b == (uint32_t)kWinBins - 1u ? 0.f : wb);
                const float wh = b == 0 ? 1.f : wb / r;
                ct += c[j];
                lt += (float)c[j] * wl;
                ut += (float)c[j] * wh;
                wb *= r;
            }
        }
        uint32_t ci = ct;
        float li = lt, ui = ut;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t c2v = __shfl_up_sync(0xFFFFFFFFu, ci, o);
            const float l2 = __shfl_up_sync(0xFFFFFFFFu, li, o), u2 = __shfl_up_sync(0xFFFFFFFFu, ui, o);
            if (lane >= o) {
                ci += c2v;
                li += l2;
                ui += u2;
            }
        }
        if (lane == 31) {
            ctl.win_c[warp] = ci;
            ctl.win_l[warp] = li;
            ctl.win_u[warp] = ui;
        }
        SSync::sync();
        uint32_t cP = ci - ct;
        float LP = li - lt, UP = ui - ut;
        for (int q = 0; q < warp; ++q) {
            cP += ctl.win_c[q];
            LP += ctl.win_l[q];
            UP += ctl.win_u[q];
        }
        const uint32_t c_start = cP;
        const float pz = rpm.P * Z;
        uint32_t f_bk = kWinBins, f_plo = kWinBins, f_lf = kWinBins;
        {
            float wb = w0;
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                const uint32_t b = b0 + j, cb = c[j];
                const float wl = b == 0 ? 1.f : (b == (uint32_t)kWinBins - 1u ? 0.f : wb);
                const float wh = b == 0 ? 1.f : wb / r;
                if (rpm.k_on && f_bk == (uint32_t)kWinBins && cP < (uint32_t)rpm.K && cP + cb >= (uint32_t)rpm.K) f_bk = b;
                if (p_on && f_lf == (uint32_t)kWinBins && LP * (1.f - 1e-4f) >= pz) f_lf = b;
                cP += cb;
                LP += (float)cb * wl;
                UP += (float)cb * wh;
                if (p_on && f_plo == (uint32_t)kWinBins && UP * (1.f + 1e-4f) >= pz) f_plo = b;
                wb *= r;
            }
        }
        if (tid == kThreads - 1) ctl.win_all = cP;  // every counted token
        if (f_bk < (uint32_t)kWinBins) atomicMin(&ctl.win_bk, f_bk);
        if (f_plo < (uint32_t)kWinBins) atomicMin(&ctl.win_plo, f_plo);
        if (f_lf < (uint32_t)kWinBins) atomicMin(&ctl.win_lfirst, f_lf);
        SSync::sync();
        // bins < lo are kept by every filter; the window is [lo, hi]
        uint32_t plo = (uint32_t)kWinBins, phi = (uint32_t)kWinBins;
        if (p_on) {
            if (!(rpm.P > 0.f)) {
                plo = 1u;  // the argmax class alone
                phi = 0u;
            } else {
                plo = max(ctl.win_plo, 1u);  // the argmax class is always kept
                phi = ctl.win_lfirst - 1u;
            }
        }
        const uint32_t bk = ctl.win_bk;
        const uint32_t wlo_b = min(bk, plo), whi_b = min(bk, phi);
        uint32_t cnt = 0, before = c_start;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const uint32_t b = b0 + j;
            if (b >= wlo_b && b <= whi_b) cnt += c[j];
            if (b < wlo_b) before += c[j];
        }
        cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
        if (lane == 0) ctl.win_n[warp] = cnt;
        if (wlo_b < (uint32_t)kWinBins && wlo_b >= b0 && wlo_b < b0 + kPer) ctl.win_clo = before;
        SSync::sync();
        if (tid == 0) {
            uint32_t total = 0;
            for (int q = 0; q < kWarps; ++q) total += ctl.win_n[q];
            const bool nonempty = wlo_b <= whi_b;
            ctl.win_lo = wlo_b;
            ctl.win_hi = whi_b;
            ctl.win_cnt = total;
            ctl.win_nw = 0u;
            const bool fail = nonempty && (whi_b >= (uint32_t)kWinBins - 1u || total > (uint32_t)kCandCap);
            ctl.win_fail = fail ? 1u : 0u;
            // when the tokens above the window and the window's own fit the
            // list, pass B gathers them all and the list is resolved as a
            // whole; else the tokens above the window are summed in the pass
            const uint32_t n_gather = (wlo_b < (uint32_t)kWinBins ? ctl.win_clo : ctl.win_all) + (nonempty ? total : 0u);
            ctl.win_gather = (!fail && n_gather <= (uint32_t)kCandCap) ? 1u : 0u;
        }
    }
    CSync::sync();
    const uint32_t w_lo = ctl.win_lo, w_hi = ctl.win_hi;
    const bool w_fail = ctl.win_fail != 0u;
    const bool w_gather = ctl.win_gather != 0u;
    // pass B: the window's tokens to the list; above it, the exact mass, the
    // smallest value and a Gumbel-max draw (all of them are kept).  In gather
    // mode every token down to the window's end goes to the list instead.
    const float c2 = rpm.c2, invT = rpm.invT, T = rpm.T;
    const uint64_t seed = a.seed, offset = a.offset;
    F2 mass{0.f, 0.f};
    float msure = INFINITY, best_sc = -INFINITY, gcut = -INFINITY;
    uint32_t bi = 0xFFFFFFFFu, ntop = 0u;
    uint32_t top_u = 0u, top_i = 0xFFFFFFFFu;  // the argmax class's best: lattice index of u, token
    {
        // groups below every bin up to the window's end (one bin of slack for
        // rounding) hold no token this pass takes
        const uint32_t b_end = w_lo <= w_hi ? w_hi + 1u : w_lo;  // bins < b_end matter
        const float x_gather = (w_fail || b_end >= (uint32_t)kWinBins - 1u) ? v_m
                                                                            : fmaxf(v_m, m - (float)(b_end + 1u) / c2S);
        // the draw above the window, one Philox block per group of four
        // consecutive tokens; an argmax-class token weighs only its u
        auto take = [&](uint32_t word, uint32_t i, float xt, bool top) {
            if (top) {
                // every score of the argmax class is G(u) alone: its best
                // is the largest u (lowest index on ties), and no
                // logarithm is taken here
                const uint32_t u = word >> 9;
                if (u > top_u || (u == top_u && i < top_i)) {
                    top_u = u;
                    top_i = i;
                }
                return;
            }
            // Gumbel-max with the unfiltered draw's prune
            const float srel = (xt - m) * invT;
            const float need = best_sc - srel;  // the Gumbel value this token must beat
            if (need > kTopBitsMargin && (word >> 22) != 0x3FFu) return;
            if (word_uniform(word) < gumbel_u_floor(need)) return;
            const float sc = srel + gumbel_of(word);
            if (sc > best_sc || (sc == best_sc && i < bi)) {
                best_sc = sc;
                bi = i;
                gcut = fmaf(sc - kGumbelMax, T, m);
            }
        };
        // the draw over one vector's marked tokens: tbits of the argmax
        // class, gbits above the window
        auto draw = [&](const float (&x)[AE], uint32_t eb, uint32_t tbits, uint32_t gbits) {
            if ((eb & 3u) == 0u) {
                // an aligned vector: whole groups, slots known at compile time
#pragma unroll
                for (int gq = 0; gq < AE / 4; ++gq) {
                    if (!(((tbits | gbits) >> (4 * gq)) & 0xFu)) continue;
                    const uint32_t q = (eb >> 2) + (uint32_t)gq;
                    const uint4 blk = token_block(seed, offset, (uint32_t)row, q);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int t = 4 * gq + k;
                        if (!(((tbits | gbits) >> t) & 1u)) continue;
                        const uint32_t word = k == 0 ? blk.x : (k == 1 ? blk.y : (k == 2 ? blk.z : blk.w));
                        take(word, q * 4u + (uint32_t)k, x[t], ((tbits >> t) & 1u) != 0u);
                    }
                }
                return;
            }
            // otherwise the vector's groups in a rolled loop
            const uint32_t q0 = eb >> 2;
            const int ng = (int)(((eb + (uint32_t)AE - 1u) >> 2) - q0) + 1;
#pragma unroll 1
            for (int gq = 0; gq < ng; ++gq) {
                const uint32_t q = q0 + (uint32_t)gq;
                const int tq = (int)(q * 4u) - (int)eb;  // slot of the group's first token (> -4)
                const uint32_t gmask = tq >= 0 ? 0xFu << tq : 0xFu >> -tq;
                if (!((tbits | gbits) & gmask)) continue;
                const uint4 blk = token_block(seed, offset, (uint32_t)row, q);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int t = tq + k;
                    if (t < 0 || t >= AE) continue;
                    if (!(((tbits | gbits) >> t) & 1u)) continue;
                    const uint32_t word = k == 0 ? blk.x : (k == 1 ? blk.y : (k == 2 ? blk.z : blk.w));
                    take(word, q * 4u + (uint32_t)k, vec_elem<AE>(x, t), ((tbits >> t) & 1u) != 0u);
                }
            }
        };
        // which tokens of a vector the draw takes (see the gather step)
        auto marks = [&](const float (&x)[AE], uint32_t &tbits, uint32_t &gbits) {
#pragma unroll
            for (int t = 0; t < AE; ++t) {
                const float xt = x[t];
                if (!(xt >= v_m) || !(xt > -INFINITY)) continue;
                if (xt == m) {
                    if (w_lo > 0u) tbits |= 1u << t;
                    continue;
                }
                const uint32_t b = win_bin(xt, m, c2S);
                if (p_on && b == (uint32_t)kWinBins - 1u) continue;
                gbits |= (b < w_lo && xt >= gcut) ? 1u << t : 0u;
            }
        };
        // On a step where few lanes have tokens to draw, a lane's vectors are
        // marked in dmask and drawn at the stage's end by the whole warp, one
        // marked vector a lane, so that a Philox block runs on all lanes at
        // once: on rows where a few tokens in a hundred are kept, a warp step
        // rarely has more than a handful of lanes with one.
        uint32_t dmask = 0;
        auto gather = [&](const float (&x)[AE], uint32_t eb, bool live, int vi) {
            // elements to the list; of the argmax class (above the window);
            // above the window and able to win the draw
            uint32_t wbits = 0, tbits = 0, gbits = 0;
            if (live && !w_fail) {
#pragma unroll
                for (int t = 0; t < AE; ++t) {
                    const float xt = x[t];
                    if (!(xt >= v_m) || !(xt > -INFINITY)) continue;
                    if (w_gather) {
                        const uint32_t b = win_bin(xt, m, c2S);
                        if (p_on && b == (uint32_t)kWinBins - 1u) continue;  // below the top-p bound
                        wbits |= b < b_end ? 1u << t : 0u;
                        continue;
                    }
                    if (xt == m) {  // bin 0: above the window unless the window starts there
                        if (w_lo > 0u) tbits |= 1u << t;
                        else wbits |= 1u << t;
                        continue;
                    }
                    const uint32_t b = win_bin(xt, m, c2S);
                    if (p_on && b == (uint32_t)kWinBins - 1u) continue;  // below the top-p bound
                    if (b < w_lo) {
                        mass = f2_add(mass, F2{ex2_approx((xt - m) * c2), 0.f});
                        msure = fminf(msure, xt);
                        gbits |= xt >= gcut ? 1u << t : 0u;
                    }
                    wbits |= (b >= w_lo && b <= w_hi) ? 1u << t : 0u;
                }
            }
            push_bits_warp<AE>(wbits, x, eb, cand, &ctl.win_nb, (uint32_t)kCandCap);
            ntop += (uint32_t)__popc(tbits);  // each weighs exactly 1
            const bool want = (tbits | gbits) != 0u;
            const uint32_t nwant = (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, want));
            if (!want) return;
            // a step where at least half the lanes draw is drawn in place
            // (flat rows); the head or tail element always is
            if (vi >= 0 && nwant < 16u) dmask |= 1u << vi;
            else draw(x, eb, tbits, gbits);
        };
        auto drain = [&](const uint4 *st, const uint32_t *mw, uint32_t e0) {
            uint32_t bal[kVecPerThread], pre[kVecPerThread + 1];
            pre[0] = 0u;
#pragma unroll
            for (int i = 0; i < kVecPerThread; ++i) {
                bal[i] = __ballot_sync(0xFFFFFFFFu, (dmask >> i) & 1u);
                pre[i + 1] = pre[i] + (uint32_t)__popc(bal[i]);
            }
            dmask = 0u;
            const uint32_t total = pre[kVecPerThread];
            for (uint32_t e = (uint32_t)lane; e < ((total + 31u) & ~31u); e += 32u) {
                if (e >= total) continue;
                // marked vector e: vector i of lane src
                int i = 0;
                uint32_t bl = bal[0], pr = 0u;
#pragma unroll
                for (int ii = 1; ii < kVecPerThread; ++ii)
                    if (e >= pre[ii]) {
                        i = ii;
                        bl = bal[ii];
                        pr = pre[ii];
                    }
                const uint32_t src = __fns(bl, 0u, (int)(e - pr) + 1);
                const int j = (warp * 32 + (int)src) + i * kCT;
                uint4 v = st[j];
                if (mk) {
                    const uint32_t rj = (e0 & 31u) + (uint32_t)j * AE;
                    const uint32_t k = rj >> 5, sh = rj & 31u;
                    const uint32_t bits = mk == 2 ? __funnelshift_r(mw[k], mw[k + 1], sh) : (mw[k] >> sh);
                    if (DT == 0) add_bias(v, mtab_l, bits);
                    else mask_vec<DT>(v, bits & ((1u << AE) - 1u));
                }
                float x[AE];
                E::unpack(v, x);
                uint32_t tbits = 0, gbits = 0;
                marks(x, tbits, gbits);
                if (tbits | gbits) draw(x, e0 + (uint32_t)j * AE, tbits, gbits);
            }
        };
        wok = consume_pass<DT>(stages, masks, ctl, nchunks, g.head, cb, mk, mtab_l, wok, hx, he, x_gather, gather,
                               drain);
    }
    {
        // the argmax class joins the sums: mass ntop, smallest value m, and its
        // best token's full score
        if (ntop) {
            mass = f2_add(mass, F2{(float)ntop, 0.f});
            msure = fminf(msure, m);
        }
        if (top_i != 0xFFFFFFFFu) {  // this lane drew argmax-class tokens (its own or another lane's)
            const float sc = gumbel_of(top_u << 9);
            if (sc > best_sc || (sc == best_sc && top_i < bi)) {
                best_sc = sc;
                bi = top_i;
            }
        }
        F2 wm2 = mass;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            wm2 = f2_add(wm2, F2{__shfl_xor_sync(0xFFFFFFFFu, wm2.hi, o), __shfl_xor_sync(0xFFFFFFFFu, wm2.lo, o)});
        float mn = msure;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
        const uint64_t wb = warp_max_u64(bi != 0xFFFFFFFFu ? rank_key(best_sc, bi) : 0ull);
        if (lane == 0) {
            ctl.wmh[warp] = wm2.hi;
            ctl.wml[warp] = wm2.lo;
            ctl.wmin[warp] = mn;
            ctl.wbest[warp] = wb;
        }
        if (!wok) atomicOr(&g_sample_row_status, kStatusTimeout);
    }
    CSync::sync();
    if (tid >= kThreads) return out;
    if (w_gather && ctl.win_nb <= (uint32_t)kCandCap) {
        // the list holds every token down to the window's end.  Those above
        // the window need no order: they are summed, and their smallest value
        // and best draw kept, while the window's keys move to the start of the
        // idle stage ring, the only keys that get sorted.
        uint64_t *wk = reinterpret_cast<uint64_t *>(stages);
        const uint32_t n = ctl.win_nb;
        F2 bm{0.f, 0.f};
        float bmin = INFINITY;
        uint64_t bbest = 0ull;
        uint32_t nsure = 0;
        for (uint32_t i = tid; i < n; i += kThreads) {
            const uint64_t key = cand[i];
            const float x = rank_key_value(key);
            if (win_bin(x, m, c2S) < w_lo) {
                ++nsure;
                bm = f2_add(bm, F2{ex2_approx((x - m) * c2), 0.f});
                bmin = fminf(bmin, x);
                const uint32_t idx = rank_key_index(key);
                const uint4 blk = token_block(seed, offset, (uint32_t)row, idx >> 2);
                const uint64_t sk = rank_key((x - m) * invT + gumbel_of(block_word(blk, idx & 3u)), idx);
                bbest = sk > bbest ? sk : bbest;
            } else {
                wk[atomicAdd(&ctl.win_nw, 1u)] = key;
            }
        }
        nsure = __reduce_add_sync(0xFFFFFFFFu, nsure);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            bm = f2_add(bm, F2{__shfl_xor_sync(0xFFFFFFFFu, bm.hi, o), __shfl_xor_sync(0xFFFFFFFFu, bm.lo, o)});
            bmin = fminf(bmin, __shfl_xor_sync(0xFFFFFFFFu, bmin, o));
        }
        bbest = warp_max_u64(bbest);
        if (lane == 0) {
            ctl.wmh[warp] = bm.hi;
            ctl.wml[warp] = bm.lo;
            ctl.wmin[warp] = bmin;
            ctl.wbest[warp] = bbest;
            ctl.win_n[warp] = nsure;
        }
        SSync::sync();
        F2 base{0.f, 0.f};
        float mins = INFINITY;
        uint64_t bsure = 0ull;
        uint32_t cnt = 0;
        for (int q = 0; q < kWarps; ++q) {
            base = f2_add(base, F2{ctl.wmh[q], ctl.wml[q]});
            mins = fminf(mins, ctl.wmin[q]);
            bsure = ctl.wbest[q] > bsure ? ctl.wbest[q] : bsure;
            cnt += ctl.win_n[q];
        }
        select_window<SSync>(seed, offset, row, rpm, wk, ctl.win_nw, cnt, base, v_m, mins, bsure, m, Z, ctl.sel,
                             out.token, out.vstar);
        out.done = true;
    } else if (!w_fail && ctl.win_nb <= (uint32_t)kCandCap) {
        F2 base{0.f, 0.f};
        float mins = INFINITY;
        uint64_t bsure = 0ull;
        for (int q = 0; q < kCW; ++q) {
            base = f2_add(base, F2{ctl.wmh[q], ctl.wml[q]});
            mins = fminf(mins, ctl.wmin[q]);
            bsure = ctl.wbest[q] > bsure ? ctl.wbest[q] : bsure;
        }
        const uint32_t clo = w_lo <= w_hi ? ctl.win_clo : 0u;
        select_window<SSync>(seed, offset, row, rpm, cand, ctl.win_nb, clo, base, v_m, mins, bsure, m, Z, ctl.sel,
                             out.token, out.vstar);
        out.done = true;
    }
    return out;
}

// The end of a filtered row on one warp: compact the candidate list to the
// keys >= theta (in place, in order) and, when at most 32 remain, resolve the
// keep-threshold and the draw in registers.
struct SmallOut {
    int64_t token;
    float vstar;
    uint32_t n;  // keys >= theta; the result is valid only if n <= 32
};
__device__ __forceinline__ SmallOut settle_small(uint64_t seed, uint64_t offset, int64_t row, const RowParams &rpm,
                                                uint64_t *cand, uint32_t n_all, float theta, float v_m, float m,
                                                float Z) {
    const int lane = threadIdx.x & 31;
    uint32_t written = 0;
    for (uint32_t b0 = 0; b0 < n_all; b0 += 32) {
        const uint32_t i = b0 + (uint32_t)lane;
        const uint64_t key = i < n_all ? cand[i] : 0ull;
        const bool keep = i < n_all && rank_key_value(key) >= theta;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
        if (keep) cand[written + __popc(bal & ((1u << lane) - 1u))] = key;
        written += __popc(bal);
    }
    __syncwarp();
    SmallOut o{-1, -INFINITY, written};
    if (written <= 32u) warp_select_small(seed, offset, row, rpm, cand, written, theta, v_m, m, Z, o.token, o.vstar);
    return o;
}

}  // namespace

// The keep-threshold and the draw from a complete candidate list (every
// allowed logit >= theta, n_all keys, possibly more than theta needs): warp 0
// compacts the keys >= theta in place, in order, and settles the row alone
// when at most 32 remain; otherwise the block steps.  On the first 256
// threads; false if the list cannot decide (the radix path then runs).
template <class Sync>
__device__ __forceinline__ bool resolve_list(const SampleArgs &a, int64_t row, const RowParams &rpm, uint64_t *cand,
                                             uint32_t n_all, float theta, float v_m, float m, float Z, Hist &hist,
                                             SelCtl &sel, int64_t &token, float &vstar) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp == 0) {
        const SmallOut o = settle_small(a.seed, a.offset, row, rpm, cand, n_all, theta, v_m, m, Z);
        if (o.n <= 32u) {
            token = o.token;
            vstar = o.vstar;
        }
        if (lane == 0) sel.n = o.n;
    }
    Sync::sync();
    const uint32_t n = sel.n;
    if (n <= 32u) return true;  // warp 0 holds the result
    return select_from_candidates<Sync>(a, row, rpm, cand, n, (uint32_t)kCandCap, theta, v_m, m, Z, hist, sel, token,
                                        vstar);
}

// SPEC < 0: every row's mode and mask layout found at run time.  SPEC =
// 4 mode + mk: every row has that mode and mask layout (scalar sampling
// parameters, 16-byte aligned rows), and only its code is compiled in.
template <int DT, int SPEC>
__global__ void __launch_bounds__(kRowThreads, 2) sample_row_kernel(SampleArgs a) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint4 *stages = reinterpret_cast<uint4 *>(smem);
    uint32_t *masks = reinterpret_cast<uint32_t *>(smem + kStages * kStageVec * 16);
    uint64_t *cand = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(masks) + kStages * kStageWords * 4);
    RowCtl &ctl = *reinterpret_cast<RowCtl *>(reinterpret_cast<uint8_t *>(cand) + kCandCap * 8);
    float4 *mtab = reinterpret_cast<float4 *>(reinterpret_cast<uint8_t *>(&ctl) + sizeof(RowCtl));
    // the selection's digit histogram is needed only after the stream: it
    // takes the end of the stage ring (the general path's histograms take its
    // start)
    Hist &hist = *reinterpret_cast<Hist *>(smem + kStages * kStageVec * 16 - sizeof(Hist));

    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t V = (int32_t)a.V;
    const uint8_t *rp = reinterpret_cast<const uint8_t *>(a.logits) + (size_t)row * a.stride * E::SIZE;
    const int32_t *mrow = a.mask ? a.mask + (size_t)row * a.mstride : nullptr;
    const bool has_mask = mrow != nullptr;
    const Slice32 g = make_slice32<AE, E::SIZE>(rp, V, 0, 1);  // head, nvec, tail of the row
    const int nchunks = (g.nvec + kStageVec - 1) / kStageVec;

    // Programmatic dependent launch: the next kernel on the stream may be
    // scheduled now (its CTAs take SM slots as they free up and wait for this
    // grid to finish before they read memory), and this grid's prologue below
    // may overlap the previous kernel.  No global memory is read before the
    // wait, so logits written by the previous kernel are always seen.
    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.full[s], 1 + 32);  // the producer's expect-tx + one cp.async arrival per lane
            mbar_init(&ctl.empty[s], kCW);
        }
        ctl.ncand = 0;
        for (int i = 0; i < kCW; ++i) {
            ctl.wtau[i] = -INFINITY;
            ctl.wmax[i] = -INFINITY;
            ctl.ubest[i] = 0u;
        }
        mbar_init_fence();
    }
    if (DT == 0 && a.mask) init_mask_tab(mtab);
    __syncthreads();
    pdl_wait_primary();

    const RowParams rpm = row_params(a, row);
    const bool tau_on = rpm.k_on && (rpm.K + kCW - 1) / kCW <= kTauMaxR;
    const bool push_on = rpm.filtered && (tau_on || rpm.m_on);
    int mode_rt;
    if (rpm.greedy) mode_rt = kGreedy;
    else if (rpm.unfiltered) mode_rt = kUnfiltered;
    else if (push_on) mode_rt = rpm.p_on ? kFilterZ : kFilter;
    else mode_rt = kZOnly;
    const int mode = SPEC >= 0 ? SPEC / 4 : mode_rt;
    const int r_tau = tau_on ? (rpm.K + kCW - 1) / kCW : 0;
    const float tlnmp = rpm.tlnmp;
    Acc A;
    A.mx = -INFINITY;
    A.mi = 0xFFFFFFFFu;
    A.zp = 0ull;
    A.nm = -INFINITY;  // until the reference is set, normaliser terms add 0
    A.dz = 0.f;
    A.rf = -INFINITY;
    A.rhi = INFINITY;  // and never move it
    A.sbest = -INFINITY;
    A.sbi = 0xFFFFFFFFu;
    A.gcut = -INFINITY;
    A.wbest = -INFINITY;
    A.wcut = -INFINITY;
    A.full = false;
    bool ok = true;
    Ctx cx;
    cx.mm = -INFINITY;
    Bound bd;
    bd.tau_on = tau_on;
    bd.m_on = rpm.m_on;
    bd.r_tau = r_tau;
    bd.tlnmp = tlnmp;

    if (warp == kCW) {
        // ---------------------------------------------------------- producer
        ok = produce_row<DT>(stages, masks, ctl, rp, mrow, g, nchunks, 0, push_on || rpm.unfiltered);
    } else {
        // ---------------------------------------------------------- consumers
        // a vector's AE mask bits cross a word boundary only when the row start
        // is not 16-byte aligned (AE divides 32)
        const int mk = !has_mask ? 0 : (g.head != 0 ? 2 : 1);
        cx.row = row;
        cx.T = rpm.T;
        cx.invT = rpm.invT;
        cx.c2 = rpm.c2;
        cx.zspan = kZSpan / rpm.c2;
        cx.theta = -INFINITY;
        cx.ref = 0.f;
        cx.seed = a.seed;
        cx.offset = a.offset;
        cx.cand = cand;
        cx.ncand_s = smem_u32(&ctl.ncand);
        cx.gq = reinterpret_cast<uint16_t *>(cand) + warp * (32 * kVecPerThread);  // unfiltered rows push no candidates
        cx.mtab = mtab + (lane & (kMaskTabCopies - 1));

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
                accumulate1(hx, he, A);
            }
        }

        // ---- the row's stages, in a loop made for the mode and the mask layout
        auto rest = [&](auto mode_c) {
            constexpr int M = decltype(mode_c)::value;
            if (mk == 0) ok = stream_row<DT, M, 0>(stages, masks, ctl, nchunks, g.nvec, g.head, bd, cx, A, ok, hx, he);
            else if (mk == 1) ok = stream_row<DT, M, 1>(stages, masks, ctl, nchunks, g.nvec, g.head, bd, cx, A, ok, hx, he);
            else ok = stream_row<DT, M, 2>(stages, masks, ctl, nchunks, g.nvec, g.head, bd, cx, A, ok, hx, he);
        };
        if constexpr (SPEC >= 0) {
            ok = stream_row<DT, SPEC / 4, SPEC % 4>(stages, masks, ctl, nchunks, g.nvec, g.head, bd, cx, A, ok, hx,
                                                    he);
        } else {
            switch (mode) {
                case kGreedy: rest(std::integral_constant<int, kGreedy>()); break;
                case kFilter: rest(std::integral_constant<int, kFilter>()); break;
                case kFilterZ: rest(std::integral_constant<int, kFilterZ>()); break;
                case kZOnly: rest(std::integral_constant<int, kZOnly>()); break;
                default: rest(std::integral_constant<int, kUnfiltered>()); break;
            }
        }
    }

    // ---- end of the row, on the whole CTA: warp reductions, then one combine
    if (warp < kCW) {
        const uint32_t kv = A.mx > -INFINITY ? okey(A.mx) : 0u;
        const uint32_t wkv = __reduce_max_sync(0xFFFFFFFFu, kv);
        const uint32_t wmi = __reduce_min_sync(0xFFFFFFFFu, (kv == wkv && wkv) ? A.mi : 0xFFFFFFFFu);
        const float wm = wkv ? okey_value(wkv) : -INFINITY;
        float wz = 0.f;
        if (mode == kFilterZ || mode == kZOnly) {
            // each thread's sums moved from its reference and bias onto the
            // warp maximum: 2^((rf - wm) c2 - dz), with compensated rounding
            float z0, z1;
            f2_unpack(A.zp, z0, z1);
            const bool has = A.rf > -INFINITY && wm > -INFINITY;
            wz = warp_sum_f32(has ? (z0 + z1) * ex2_diff(A.rf, wm, rpm.c2, -A.dz) : 0.f);
        }
        uint64_t wb = 0;
        if (mode == kUnfiltered) wb = warp_max_u64(A.sbest > -INFINITY ? rank_key(A.sbest, A.sbi) : 0ull);
        // the last top-k bound search is made only for rows without min-p:
        // with min-p the bound of the last refresh is kept (the search costs
        // more at the row's end than the few extra candidates it removes)
        uint32_t kth = 0;
        if (tau_on && !rpm.m_on) kth = warp_tau_key(kv, fmaxf(wm, cx.mm), bd);
        if (lane == 0) {
            ctl.wkey[warp] = wkv ? (((uint64_t)wkv << 32) | (uint64_t)(0xFFFFFFFFu - wmi)) : 0ull;
            ctl.wz[warp] = wz;
            ctl.wbest[warp] = wb;
            if (kth) ctl.wtau[warp] = okey_value(kth);  // else the last published bound stands
        }
    }
    // the producer joins here; a bounded wait that ran out anywhere counts for all
    const bool all_ok = __syncthreads_and(ok ? 1 : 0) != 0;
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
    const float v_m = rpm.m_on ? cut_at(m, tlnmp) : -INFINITY;
    const uint32_t n_all = ctl.ncand;
    // filtered rows: the candidate list when it is complete and can be
    // resolved, else the window path (which needs Z only for top-p), else
    // the radix path
    const bool filt = all_ok && gkey && (mode == kFilter || mode == kFilterZ || mode == kZOnly);
    const bool fast = filt && mode != kZOnly && n_all <= (uint32_t)kCandCap &&
                      (n_all <= (uint32_t)kSortCap || rpm.k_on) && Z == Z;
    const bool win = filt && !fast && (!rpm.p_on || Z == Z);
    int64_t token = -1;
    float vstar = -INFINITY;
    bool done = false;
    if (!win) {
        if (kRowThreads > kThreads && tid >= kThreads) return;
        if (!all_ok) {
            vstar = __int_as_float(0x7FC00000);  // a bounded wait ran out: the status flag is set
        } else if (!gkey) {
            vstar = __int_as_float(0x7FC00000);
        } else if (mode == kGreedy) {
            token = amax;
            vstar = m;
        } else if (mode == kUnfiltered) {
            token = rank_key_index(best);
        } else {
            if (fast) {
                const float theta = fmaxf(tau_on ? tau : -INFINITY, v_m);
                done = resolve_list<SSync>(a, row, rpm, cand, n_all, theta, v_m, m, Z, hist, ctl.sel, token, vstar);
            }
            if (!done) {
                if (!(Z == Z)) {  // a NaN logit reached the normaliser: recompute it with NaN as -inf
                    float zt = 0.f;
                    for (int32_t i = tid; i < V; i += kThreads) {
                        float x = E::load1(rp, i);
                        if (has_mask && !(((uint32_t)__ldg(mrow + (i >> 5)) >> (i & 31)) & 1u)) x = -INFINITY;
                        if (x == x && x > -INFINITY) zt += ex2_approx((x - m) * rpm.c2);
                    }
                    Z = block_sum_f32<SSync>(zt, ctl.sel.sc);
                }
                general_path<DT, SSync>(a, row, rpm, m, amax, (double)Z, v_m, smem, ctl.sel, token, vstar);
            }
        }
        if (tid == 0) {
            a.tokens[row] = token;
            if (a.vstar_out) a.vstar_out[row] = vstar;
        }
        return;
    }
    // ---- a filtered row with no complete candidate list: one more read
    // collects the list at the final threshold when the stream pushed
    // candidates (its list overflowed before the threshold rose), else or
    // if that list would overflow too, the window path
    const float theta = fmaxf(tau_on ? tau : -INFINITY, v_m);
    const WinOut w = window_path<DT>(a, rpm, m, Z, v_m, mode != kZOnly ? theta : __int_as_float(0x7FC00000));
    if (kRowThreads > kThreads && tid >= kThreads) return;
    if (w.done) {
        token = w.token;
        vstar = w.vstar;
    } else {
        if (w.listed) done = resolve_list<SSync>(a, row, rpm, cand, w.nlist, theta, v_m, m, Z, hist, ctl.sel, token, vstar);
        if (!done) general_path<DT, SSync>(a, row, rpm, m, amax, (double)Z, v_m, smem, ctl.sel, token, vstar);
    }
    if (tid == 0) {
        a.tokens[row] = token;
        if (a.vstar_out) a.vstar_out[row] = vstar;
    }
}

constexpr size_t kRowSmemBytes = (size_t)kStages * kStageVec * 16 + (size_t)kStages * kStageWords * 4 +
                                 (size_t)kCandCap * 8 + sizeof(RowCtl) + (size_t)kMaskTabEntries * sizeof(float4);
// two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(2 * (kRowSmemBytes + 1024) <= 233472, "two row CTAs must fit one SM's shared memory");

// This translation unit's status word (see g_sample_row_status).
static unsigned int *row_status_word() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sample_row_status) != cudaSuccess) return nullptr;
    return reinterpret_cast<unsigned int *>(p);
}

}  // namespace tsa
