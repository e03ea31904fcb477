// Pieces of `sample` shared by its kernels (logits-processor, "API" and
// "Method"): the per-row parameters, the exact keep-threshold and Gumbel-max
// draw over a candidate list, and the general path that re-reads a row when
// no candidate list is complete.  Block-level steps take a barrier policy so
// that a kernel whose other warps do different work can run them on its
// consumer warps alone; those threads are threadIdx.x 0 .. 255.
#pragma once

#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_host.h"
#include "tsa_select.cuh"

namespace tsa {
namespace sample_detail {

constexpr int kThreads = kSelThreads;
constexpr int kWarps = kSelWarps;
constexpr int kSortCap = 1024;  // largest candidate set sorted directly
// Fixed-point scale of token masses in the general path's histograms: masses
// are <= 1 and rows have < 2^23 tokens, so sums stay below 2^63.
constexpr float kMassScale = 1099511627776.0f;  // 2^40
constexpr float kLog2e = 1.4426950408889634f;
// Unless the top 10 bits of a word's 23-bit lattice index are all ones, its
// uniform is below 1 - 2^-10, so -ln u > 2^-10 and G = -ln(-ln u) < 10 ln 2:
// such a word cannot beat a needed margin above 6.9315 (plus rounding slack).
constexpr float kTopBitsMargin = 6.94f;

struct RowParams {
    float T, P, MP, invT, c2;
    float tlnmp;  // T ln(min_p), rounded once (0 when min-p is off)
    int32_t K;
    bool greedy, k_on, p_on, m_on, filtered, unfiltered;
};
__device__ __forceinline__ RowParams row_params(const SampleArgs &a, int64_t row) {
    RowParams r;
    r.T = a.temperature ? __ldg(a.temperature + row) : a.temperature_s;
    r.K = a.top_k ? __ldg(a.top_k + row) : a.top_k_s;
    r.P = a.top_p ? __ldg(a.top_p + row) : a.top_p_s;
    r.MP = a.min_p ? __ldg(a.min_p + row) : a.min_p_s;
    r.greedy = !(r.T > 0.f) || r.K == 1;
    r.k_on = !r.greedy && r.K > 1;
    r.p_on = !r.greedy && r.P < 1.f;
    r.m_on = !r.greedy && r.MP > 0.f;
    r.filtered = r.k_on || r.p_on || r.m_on;
    r.unfiltered = !r.greedy && !r.filtered;
    r.invT = r.greedy ? 1.f : 1.f / r.T;
    r.c2 = r.invT * kLog2e;  // log2(e) / T
    r.tlnmp = r.m_on ? __fmul_rn(r.T, logf(r.MP)) : 0.f;
    return r;
}

// The min-p cut at row maximum m: min-p keeps l when p_l >= min_p p_max, that
// is l - m >= T ln(min_p).  For a float l that holds exactly when l is at or
// above the smallest float c >= m + tlnmp, so c is taken from the rounded sum
// and its exact rounding error (two-sum): no logit ends up on the wrong side
// of the cut through the rounding of m + tlnmp, whatever the size of m.  It
// is capped at m (the argmax class is always kept), and it is monotone in m,
// so a cut formed at a running maximum never exceeds the final one.
__device__ __forceinline__ float min_p_cut(float m, float tlnmp) {
    const float s = __fadd_rn(m, tlnmp);
    const float bp = __fsub_rn(s, m);
    const float err = __fadd_rn(__fsub_rn(m, __fsub_rn(s, bp)), __fsub_rn(tlnmp, bp));  // m + tlnmp = s + err
    const float c = err > 0.f ? nextafterf(s, INFINITY) : s;
    return fminf(c, m);
}

constexpr float kLn2 = 0.693147181f;
// 2^((a - b) c2 + extra) for finite a and b, the exponent's own roundings
// compensated: a - b = d + derr exactly (two-sum), d c2 = e + (its rounding,
// recovered by an fma), and the small remainder elo is applied through the
// series of 2^elo rather than a second ex2.approx.  Its error is that of one
// ex2.approx, whatever the size of (a - b) c2.  Rare paths only.
__device__ __forceinline__ float ex2_diff(float a, float b, float c2, float extra) {
    const float d = __fsub_rn(a, b);
    const float bp = __fsub_rn(d, a);
    const float derr = __fadd_rn(__fsub_rn(a, __fsub_rn(d, bp)), __fsub_rn(-b, bp));
    const float e = __fmul_rn(d, c2);
    const float elo = __fadd_rn(fmaf(d, c2, -e), fmaf(derr, c2, extra));
    const float t = elo * kLn2;
    const float corr = fabsf(t) < 0x1p-6f ? fmaf(t, fmaf(t, 0.5f, 1.f), 1.f) : ex2_approx(elo);
    return ex2_approx(e) * corr;
}

// Smallest uniform u whose Gumbel variate can exceed c, slightly lowered so
// the test never rejects a winner: G(u) > c needs u > exp(-exp(-c)).
__device__ __forceinline__ float gumbel_u_floor(float c) {
    const float e1 = ex2_approx(-c * kLog2e);
    return ex2_approx(-e1 * kLog2e) * (1.0f - 1.0e-5f) - 1.0e-6f;
}
__device__ __forceinline__ float word_uniform(uint32_t w) { return (float)(2u * (w >> 9) + 1u) * 0x1p-24f; }

// Shared-memory control block of the selection steps.
struct SelCtl {
    Scratch sc;
    float whi[kWarps], wlo[kWarps];  // per-warp compensated mass sums
    uint32_t wlast[kWarps];
    uint32_t n;
    float vs;
    uint32_t tok;
};

// Compensated fp32 sums: a value is hi + lo with |lo| << |hi|; adding two
// keeps the rounding error of the high parts (Knuth's two-sum) in lo.  Prefix
// masses of up to a few thousand terms then stay within about 1e-7 of Z,
// well inside the comparison band of the top-p boundary, with no FP64.
struct F2 {
    float hi, lo;
};
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    const float s = a.hi + b.hi, bp = s - a.hi;
    const float err = (a.hi - (s - bp)) + (b.hi - bp);
    return F2{s, a.lo + b.lo + err};
}
// Inclusive warp prefix of a compensated value.
__device__ __forceinline__ F2 warp_incl_scan_f2(F2 v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        F2 t;
        t.hi = __shfl_up_sync(0xFFFFFFFFu, v.hi, o);
        t.lo = __shfl_up_sync(0xFFFFFFFFu, v.lo, o);
        if (lane >= o) v = f2_add(t, v);
    }
    return v;
}

// Bitonic sort of n rank keys in shared memory, descending (pads with 0 up to
// the next power of two, which must fit the buffer).
template <class Sync>
__device__ __forceinline__ void block_sort_desc(uint64_t *keys, uint32_t n) {
    uint32_t n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (uint32_t i = n + threadIdx.x; i < n2; i += kThreads) keys[i] = 0ull;
    Sync::sync();
    for (uint32_t kk = 2; kk <= n2; kk <<= 1)
        for (uint32_t jj = kk >> 1; jj > 0; jj >>= 1) {
            for (uint32_t i = threadIdx.x; i < n2; i += kThreads) {
                const uint32_t pp = i ^ jj;
                if (pp > i) {
                    const uint64_t ki = keys[i], kp = keys[pp];
                    const bool desc = (i & kk) == 0;
                    if (desc ? (ki < kp) : (ki > kp)) {
                        keys[i] = kp;
                        keys[pp] = ki;
                    }
                }
            }
            Sync::sync();
        }
}

// Block-local radix digit (one bin per thread): the digit D holding the
// `need`-th largest key; `above` = keys in digits above D.
template <class Sync>
__device__ __forceinline__ uint32_t block_digit(const uint32_t *cnt_in, uint64_t need, Scratch &sc,
                                                uint64_t &above) {
    const int d = threadIdx.x;
    const uint32_t cnt = cnt_in[d];
    const int w = d >> 5, l = d & 31;
    uint32_t incl = cnt;  // suffix within the warp: lanes l .. 31
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (l + o < 32) incl += t;
    }
    Sync::sync();
    if (l == 0) sc.r64[w] = incl;
    Sync::sync();
    uint64_t later = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i)
        if (i > w) later += sc.r64[i];
    const uint64_t excl = incl - cnt + later;
    if (d == 0) sc.u0 = 0xFFFFFFFFu;
    Sync::sync();
    if (cnt > 0 && excl < need && need <= excl + cnt) {
        sc.u0 = (uint32_t)d;
        sc.above = excl;
    }
    Sync::sync();
    const uint32_t D = sc.u0;
    above = D < 256u ? sc.above : 0ull;
    Sync::sync();
    return D;
}

// Block-local mass digit: the lowest non-empty digit whose mass strictly above
// (base + digits above it) is still below pz.
template <class Sync>
__device__ __forceinline__ uint32_t block_mass_digit(const Hist &h, uint64_t base, double pz, Scratch &sc,
                                                     uint64_t &above) {
    const int d = threadIdx.x;
    const uint32_t cnt = h.cnt[d];
    const uint64_t mass = h.mass[d];
    const int w = d >> 5, l = d & 31;
    uint64_t incl = mass;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (l + o < 32) incl += t;
    }
    Sync::sync();
    if (l == 0) sc.r64[w] = incl;
    Sync::sync();
    uint64_t later = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i)
        if (i > w) later += sc.r64[i];
    const uint64_t excl = incl - mass + later;
    if (d == 0) sc.u0 = 0xFFFFFFFFu;
    Sync::sync();
    if (cnt > 0 && (double)(base + excl) < pz) atomicMin(&sc.u0, (uint32_t)d);
    Sync::sync();
    const uint32_t D = sc.u0;
    if (D < 256u && d == (int)D) sc.above = excl;
    Sync::sync();
    above = D < 256u ? sc.above : 0ull;
    Sync::sync();
    return D;
}

// The keep-threshold and the draw from at most 32 candidates, by one warp
// with no block barrier: cand[0 .. n) holds rank keys of every allowed logit
// >= theta of the row (theta >= the min-p cut v_m when min-p is on), in any
// order.  No sort: each lane takes one key and counts the keys above it (its
// sorted position; keys are distinct) while summing their masses in
// compensated fp32 (two TwoSum chains), unless neither top-k nor top-p needs
// the positions.  Top-k takes the key at position
// k - 1, top-p the last position whose mass strictly above is < p Z, and the
// Gumbel-max draw, whose Philox words every lane computes up front, runs over
// the keys >= v*.  Every lane returns the same token and v*.
__device__ __forceinline__ void warp_select_small(uint64_t seed, uint64_t offset, int64_t row, const RowParams &rpm,
                                                  const uint64_t *cand, uint32_t n, float theta, float v_m, float m,
                                                  float Z, int64_t &token, float &vstar) {
    const int lane = threadIdx.x & 31;
    const bool has = lane < (int)n;
    const uint64_t v = has ? cand[lane] : 0ull;
    const float x = rank_key_value(v);
    const uint32_t idx = rank_key_index(v);
    // the draw's score, before v* is known
    float score = -INFINITY;
    if (has) {
        const uint4 blk = token_block(seed, offset, (uint32_t)row, idx >> 2);
        score = (x - m) * rpm.invT + gumbel_of(block_word(blk, idx & 3));
    }
    const float wgt = (has && rpm.p_on) ? ex2_approx((x - m) * rpm.c2) : 0.f;
    const float pz = rpm.P * Z;
    // The ranks are needed for top-k when k <= n, and for top-p unless the
    // candidates' whole mass is below p Z (less a 1e-6 margin): then every
    // candidate has less than p Z above it, top-p keeps them all, and its cut
    // is the smallest candidate.
    bool ranked = rpm.k_on && (uint32_t)rpm.K <= n;
    bool p_all = false;
    if (!ranked && rpm.p_on) {
        F2 t{wgt, 0.f};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            t = f2_add(t, F2{__shfl_xor_sync(0xFFFFFFFFu, t.hi, o), __shfl_xor_sync(0xFFFFFFFFu, t.lo, o)});
        p_all = t.hi + t.lo < pz * (1.f - 1.0e-6f);
        ranked = !p_all;
    }
    uint32_t pos = 0;
    F2 e0{0.f, 0.f}, e1{0.f, 0.f};
    for (uint32_t q = 0; ranked && q < n; q += 2) {
        const uint64_t k0 = __shfl_sync(0xFFFFFFFFu, v, (int)q);
        const float w0 = __shfl_sync(0xFFFFFFFFu, wgt, (int)q);
        const uint64_t k1 = __shfl_sync(0xFFFFFFFFu, v, (int)(q + 1) & 31);
        const float w1 = __shfl_sync(0xFFFFFFFFu, wgt, (int)(q + 1) & 31);
        if (k0 > v) {
            ++pos;
            e0 = f2_add(e0, F2{w0, 0.f});
        }
        if (q + 1 < n && k1 > v) {
            ++pos;
            e1 = f2_add(e1, F2{w1, 0.f});
        }
    }
    float v_k = -INFINITY;
    if (rpm.k_on && (uint32_t)rpm.K <= n) {
        const uint32_t at = __ballot_sync(0xFFFFFFFFu, has && pos == (uint32_t)rpm.K - 1u);
        v_k = __shfl_sync(0xFFFFFFFFu, x, __ffs(at) - 1);
    }
    const float th2 = fmaxf(fmaxf(theta, v_k), v_m);
    float v_p = -INFINITY;
    if (rpm.p_on && rpm.P > 0.f && p_all) {
        const uint32_t lo = __reduce_min_sync(0xFFFFFFFFu, has ? okey(x) : 0xFFFFFFFFu);
        v_p = okey_value(lo);
    } else if (rpm.p_on) {
        const F2 excl = f2_add(e0, e1);
        const bool ok = has && (pos == 0 || excl.hi + excl.lo < pz);
        // the last sorted position kept (position 0 always is)
        const uint32_t last = __reduce_max_sync(0xFFFFFFFFu, ok ? pos : 0u);
        const uint32_t at = __ballot_sync(0xFFFFFFFFu, has && pos == last);
        v_p = (rpm.P > 0.f) ? __shfl_sync(0xFFFFFFFFu, x, __ffs(at) - 1) : m;
    }
    vstar = fmaxf(th2, v_p);
    const uint64_t best = warp_max_u64((has && x >= vstar) ? rank_key(score, idx) : 0ull);
    token = rank_key_index(best);
}

// The keep-threshold and the draw from a candidate list.  cand[0 .. n) holds
// rank keys of every allowed logit >= theta of the row (theta >= the min-p
// cut v_m when min-p is on), in any order; `cap` is the buffer's capacity (a
// power of two >= 32) and n may exceed it only if the list is incomplete.
// m is the row maximum and Z the row's sum of exp((l - m) / T).  On success
// the token and v* are set (by thread 0 for the token) and true returned;
// false means the list cannot decide and the general path must run.
template <class Sync>
__device__ bool select_from_candidates(const SampleArgs &a, int64_t row, const RowParams &rpm, uint64_t *cand,
                                       uint32_t n, uint32_t cap, float theta, float v_m, float m, float Z,
                                       Hist &hist, SelCtl &ctl, int64_t &token, float &vstar) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float invT = rpm.invT, c2 = rpm.c2;
    float v_k = -INFINITY;
    if (n <= cap && n > (uint32_t)kSortCap && rpm.k_on && (uint32_t)rpm.K < n) {
        // too many to sort: radix-select the k-th largest, keep >= it
        uint32_t prefix = 0;
        uint64_t need = (uint64_t)rpm.K;
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            hist.cnt[tid] = 0;
            Sync::sync();
            const uint32_t hmask = pass ? (0xFFFFFFFFu << (shift + 8)) : 0u;
            for (uint32_t i = tid; i < n; i += kThreads) {
                const uint32_t kk2 = (uint32_t)(cand[i] >> 32);
                if ((kk2 & hmask) == (prefix & hmask)) atomicAdd(&hist.cnt[(kk2 >> shift) & 255u], 1u);
            }
            Sync::sync();
            uint64_t above = 0;
            const uint32_t D = block_digit<Sync>(hist.cnt, need, ctl.sc, above);
            prefix |= D << shift;
            need -= above;
        }
        v_k = okey_value(prefix);
        const float th = fmaxf(theta, v_k);
        uint32_t written = 0;  // ordered in-place compaction
        for (uint32_t t0 = 0; t0 < n; t0 += kThreads) {
            const uint32_t i = t0 + tid;
            uint64_t key = 0;
            bool keep = false;
            if (i < n) {
                key = cand[i];
                keep = rank_key_value(key) >= th;
            }
            uint32_t tile_total = 0;
            const uint32_t pos = written + block_excl_scan_u32<Sync>(keep ? 1u : 0u, ctl.sc, tile_total);
            Sync::sync();
            if (keep) cand[pos] = key;
            written += tile_total;
        }
        Sync::sync();
        n = written;
    }
    if (n <= 32u) {
        if (warp == 0) {
            int64_t tk;
            float vs;
            warp_select_small(a.seed, a.offset, row, rpm, cand, n, theta, v_m, m, Z, tk, vs);
            if (lane == 0) {
                ctl.vs = vs;
                ctl.tok = (uint32_t)(tk >= 0 ? tk : 0xFFFFFFFFu);
            }
        }
        Sync::sync();
        vstar = ctl.vs;
        token = ctl.tok == 0xFFFFFFFFu ? -1 : (int64_t)ctl.tok;
        return true;
    }
    if (n <= (uint32_t)kSortCap) {
        // up to kThreads keys: thread t owns key t, and its perturbed score
        // (independent of v*) is formed before the ranking, so the Philox
        // rounds and logarithms overlap the rank loop instead of following
        // the top-p scan
        uint64_t own = 0ull;
        float own_score = -INFINITY;
        if (n <= (uint32_t)kThreads) {
            // rank sort: keys are distinct (the index is part of the key), so
            // the number of larger keys is each key's sorted position
            own = (uint32_t)tid < n ? cand[tid] : 0ull;
            if ((uint32_t)tid < n) {
                const uint32_t idx = rank_key_index(own);
                const uint4 blk = token_block(a.seed, a.offset, (uint32_t)row, idx >> 2);
                own_score = (rank_key_value(own) - m) * invT + gumbel_of(block_word(blk, idx & 3));
            }
            uint32_t rank = 0;
            if ((uint32_t)tid < n)
                for (uint32_t j = 0; j < n; ++j) rank += cand[j] > own ? 1u : 0u;
            Sync::sync();
            if ((uint32_t)tid < n) cand[rank] = own;
            Sync::sync();
        } else {
            block_sort_desc<Sync>(cand, n);
        }
        if (rpm.k_on && (uint32_t)rpm.K <= n) v_k = fmaxf(v_k, rank_key_value(cand[rpm.K - 1]));
        const float th2 = fmaxf(fmaxf(theta, v_k), v_m);
        float v_p = -INFINITY;
        if (rpm.p_on) {
            // last sorted position whose exclusive prefix mass is < p Z
            // (compensated fp32 block scan, tile by tile)
            const float pz = rpm.P * Z;
            F2 acc{0.f, 0.f};
            uint32_t last = 1;  // position 0 (the argmax) is always kept
            for (uint32_t t0 = 0; t0 < n; t0 += kThreads) {
                const uint32_t i = t0 + tid;
                float wgt = 0.f;
                if (i < n) wgt = ex2_approx((rank_key_value(cand[i]) - m) * c2);
                const F2 incl = warp_incl_scan_f2(F2{wgt, 0.f});
                Sync::sync();
                if (lane == 31) {
                    ctl.whi[warp] = incl.hi;
                    ctl.wlo[warp] = incl.lo;
                }
                Sync::sync();
                F2 before = acc;
                for (int qq = 0; qq < warp; ++qq) before = f2_add(before, F2{ctl.whi[qq], ctl.wlo[qq]});
                const F2 all = f2_add(before, incl);
                const bool ok = (i < n) && (i == 0 || (all.hi - wgt) + all.lo < pz);
                const uint32_t bal = __ballot_sync(0xFFFFFFFFu, ok);
                if (lane == 0) ctl.wlast[warp] = bal ? t0 + warp * 32 + (31 - __clz(bal)) + 1 : 0u;
                Sync::sync();
                for (int qq = 0; qq < kWarps; ++qq) {
                    last = max(last, ctl.wlast[qq]);
                    acc = f2_add(acc, F2{ctl.whi[qq], ctl.wlo[qq]});
                }
            }
            v_p = (rpm.P > 0.f) ? rank_key_value(cand[last - 1]) : m;
        }
        vstar = fmaxf(th2, v_p);
        uint64_t best = 0ull;
        if (n <= (uint32_t)kThreads) {
            if ((uint32_t)tid < n && rank_key_value(own) >= vstar) best = rank_key(own_score, rank_key_index(own));
        } else {
            for (uint32_t i = tid; i < n; i += kThreads) {
                const uint64_t kk2 = cand[i];
                const float x = rank_key_value(kk2);
                if (!(x >= vstar)) continue;
                const uint32_t idx = rank_key_index(kk2);
                const uint4 blk = token_block(a.seed, a.offset, (uint32_t)row, idx >> 2);
                const float sc = (x - m) * invT + gumbel_of(block_word(blk, idx & 3));
                const uint64_t key = rank_key(sc, idx);
                best = key > best ? key : best;
            }
        }
        best = block_max_u64<Sync>(best, ctl.sc);
        token = rank_key_index(best);
        return true;
    }
    return false;
}

// ---------------------------------------------------------------- window path
// Rows with no usable candidate bound (top-p alone, or a list that overflowed)
// are resolved from two more streamed reads.  The first counts the row's
// tokens in log-mass bins of e = (m - l) c2 (the exponent of the token's
// weight 2^-e): bin 0 holds the argmax class (l == m) exactly, bin b >= 1
// holds e * S in [b - 1, b), and the last bin every deeper token.  From the
// counts, the top-k cut lies in one known bin, and the top-p cut in a short
// range of bins whose mass bounds straddle p Z; those bins are the window.
// The second read gathers the window's tokens as rank keys, sums the exact
// mass of every token above the window, and draws Gumbel-max over those
// tokens, all of which are kept.  The window is then resolved exactly, as a
// candidate list whose counts and masses start from the sums above it.
constexpr int kWinBins = 2048;
__device__ __forceinline__ uint32_t win_bin(float x, float m, float c2S) {
    if (x == m) return 0u;
    const float es = __fmul_rn(__fsub_rn(m, x), c2S);  // the same rounding on every read
    // 1 + floor(es) for 0 <= es < 2^23: es + 2^23 rounded down holds floor(es)
    // in its low mantissa bits (an FMA-pipe add instead of a conversion)
    return es < (float)(kWinBins - 2) ? __float_as_uint(__fadd_rd(es, 8388608.f)) - 0x4AFFFFFFu
                                      : (uint32_t)(kWinBins - 1);
}

// The keep-threshold and the draw from a window: cand[0 .. n) holds the rank
// keys of every allowed token >= v_floor in the window bins, in any order; the
// tokens above the window number base_cnt (all allowed tokens, the argmax
// class included) and weigh base_mass (sum of 2^((l - m) c2)), their smallest
// kept value is min_sure and their best perturbed score key best_sure (0 when
// there are none); every one of them is kept.  n <= 2048 and cand has room
// for the next power of two.  Sets token (thread 0) and v*.
template <class Sync>
__device__ void select_window(uint64_t seed, uint64_t offset, int64_t row, const RowParams &rpm, uint64_t *cand, uint32_t n,
                              uint32_t base_cnt, F2 base_mass, float v_floor, float min_sure, uint64_t best_sure,
                              float m, float Z, SelCtl &ctl, int64_t &token, float &vstar) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float invT = rpm.invT, c2 = rpm.c2;
    uint64_t own = 0ull;
    float own_score = -INFINITY;
    if (n <= (uint32_t)kThreads) {
        own = (uint32_t)tid < n ? cand[tid] : 0ull;
        if ((uint32_t)tid < n) {
            const uint32_t idx = rank_key_index(own);
            const uint4 blk = token_block(seed, offset, (uint32_t)row, idx >> 2);
            own_score = (rank_key_value(own) - m) * invT + gumbel_of(block_word(blk, idx & 3));
        }
        uint32_t rank = 0;
        if ((uint32_t)tid < n)
            for (uint32_t j = 0; j < n; ++j) rank += cand[j] > own ? 1u : 0u;
        Sync::sync();
        if ((uint32_t)tid < n) cand[rank] = own;
        Sync::sync();
    } else {
        block_sort_desc<Sync>(cand, n);
    }
    // top-k: the k-th largest is in the window when base_cnt < K <= base_cnt + n
    float v_k = -INFINITY;
    if (rpm.k_on && (uint32_t)rpm.K > base_cnt && (uint32_t)rpm.K - base_cnt <= n)
        v_k = rank_key_value(cand[rpm.K - 1 - base_cnt]);
    // top-p: the last window position whose exclusive prefix mass (from the
    // mass above the window) is < p Z; none means the cut is the last token
    // above the window
    float v_p = -INFINITY;
    if (rpm.p_on) {
        if (!(rpm.P > 0.f)) {
            v_p = m;
        } else {
            const float pz = rpm.P * Z;
            F2 acc = base_mass;
            uint32_t last = 0;  // one past the last qualifying position
            for (uint32_t t0 = 0; t0 < n; t0 += kThreads) {
                const uint32_t i = t0 + tid;
                float wgt = 0.f;
                if (i < n) wgt = ex2_approx((rank_key_value(cand[i]) - m) * c2);
                const F2 incl = warp_incl_scan_f2(F2{wgt, 0.f});
                Sync::sync();
                if (lane == 31) {
                    ctl.whi[warp] = incl.hi;
                    ctl.wlo[warp] = incl.lo;
                }
                Sync::sync();
                F2 before = acc;
                for (int qq = 0; qq < warp; ++qq) before = f2_add(before, F2{ctl.whi[qq], ctl.wlo[qq]});
                const F2 all = f2_add(before, incl);
                const bool ok = (i < n) && ((all.hi - wgt) + all.lo < pz);
                const uint32_t bal = __ballot_sync(0xFFFFFFFFu, ok);
                if (lane == 0) ctl.wlast[warp] = bal ? t0 + warp * 32 + (31 - __clz(bal)) + 1 : 0u;
                Sync::sync();
                for (int qq = 0; qq < kWarps; ++qq) {
                    last = max(last, ctl.wlast[qq]);
                    acc = f2_add(acc, F2{ctl.whi[qq], ctl.wlo[qq]});
                }
            }
            v_p = last ? rank_key_value(cand[last - 1]) : min_sure;
        }
    }
    vstar = fmaxf(fmaxf(v_k, v_p), v_floor);
    uint64_t best = 0ull;
    if (n <= (uint32_t)kThreads) {
        if ((uint32_t)tid < n && rank_key_value(own) >= vstar) best = rank_key(own_score, rank_key_index(own));
    } else {
        for (uint32_t i = tid; i < n; i += kThreads) {
            const uint64_t kk2 = cand[i];
            const float x = rank_key_value(kk2);
            if (!(x >= vstar)) continue;
            const uint32_t idx = rank_key_index(kk2);
            const uint4 blk = token_block(seed, offset, (uint32_t)row, idx >> 2);
            const uint64_t key = rank_key((x - m) * invT + gumbel_of(block_word(blk, idx & 3)), idx);
            best = key > best ? key : best;
        }
    }
    best = block_max_u64<Sync>(best, ctl.sc);
    best = best > best_sure ? best : best_sure;
    token = best ? (int64_t)rank_key_index(best) : -1;
}

// Byte permute in sign-replicating mode: selector nibble 8 + t gives byte t's
// top bit copied into all 8 bits of that result byte.
__device__ __forceinline__ uint32_t prmt_sign(uint32_t a, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0u), "r"(sel));
    return d;
}
// Allowed words unchanged, disallowed ones replaced by the -inf pattern.
__device__ __forceinline__ uint32_t keep_or(uint32_t w, uint32_t allow, uint32_t ninf) {
    return (w & allow) | (ninf & ~allow);
}
// Apply a vector's mask bits (bit t <-> element t) to its raw 16 bytes.
// nibble * 0x10204080 moves bit t of a 4-bit nibble to bit 8t + 7, the top
// bit of byte t, from where one prmt spreads it over a 32-bit lane.
template <int DT>
__device__ __forceinline__ void mask_vec(uint4 &v, uint32_t bits) {
    if (DT == 0) {
        const uint32_t sp = bits * 0x10204080u;
        v.x = keep_or(v.x, prmt_sign(sp, 0x8888u), 0xFF800000u);
        v.y = keep_or(v.y, prmt_sign(sp, 0x9999u), 0xFF800000u);
        v.z = keep_or(v.z, prmt_sign(sp, 0xAAAAu), 0xFF800000u);
        v.w = keep_or(v.w, prmt_sign(sp, 0xBBBBu), 0xFF800000u);
    } else {
        // two 16-bit elements per word: element 2j in the low half
        const uint32_t ninf = DT == 1 ? 0xFC00FC00u : 0xFF80FF80u;
        const uint32_t lo = (bits & 0xFu) * 0x10204080u, hi = (bits >> 4) * 0x10204080u;
        v.x = keep_or(v.x, prmt_sign(lo, 0x9988u), ninf);
        v.y = keep_or(v.y, prmt_sign(lo, 0xBBAAu), ninf);
        v.z = keep_or(v.z, prmt_sign(hi, 0x9988u), ninf);
        v.w = keep_or(v.w, prmt_sign(hi, 0xBBAAu), ninf);
    }
}

// Every allowed, finite-or-infinite (not NaN) logit of the row, read straight
// from global memory: f(x, i) for each, by all kThreads threads.  The aligned
// part is read as 16-byte vectors, four in flight per thread, each masked as a
// whole; the unaligned head and tail element by element.
template <int DT, class F>
__device__ __forceinline__ void scan_row(const uint8_t *rp, const int32_t *mrow, int32_t V, F &&f) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    const int tid = threadIdx.x;
    const Slice32 g = make_slice32<AE, E::SIZE>(rp, V, 0, 1);
    auto scalar = [&](int32_t i) {
        float x = E::load1(rp, i);
        if (mrow && !(((uint32_t)__ldg(mrow + (i >> 5)) >> (i & 31)) & 1u)) x = -INFINITY;
        if (x == x && x > -INFINITY) f(x, (uint32_t)i);
    };
    if (tid < g.head) scalar(tid);
    if (tid < g.tail) scalar(g.head + g.nvec * AE + tid);
    constexpr int kU = 4;
    for (int32_t v0 = 0; v0 < g.nvec; v0 += kThreads * kU) {
        uint4 w[kU];
        uint32_t bits[kU];
        int32_t e[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t v = v0 + tid + u * kThreads;
            e[u] = v < g.nvec ? g.head + v * AE : -1;
            bits[u] = (1u << AE) - 1u;
            if (e[u] >= 0) {
                w[u] = __ldcs(reinterpret_cast<const uint4 *>(rp + (size_t)e[u] * E::SIZE));
                if (mrow) {
                    const uint32_t lo = (uint32_t)__ldg(mrow + (e[u] >> 5));
                    const uint32_t hi = ((e[u] & 31) + AE > 32) ? (uint32_t)__ldg(mrow + (e[u] >> 5) + 1) : 0u;
                    bits[u] = __funnelshift_r(lo, hi, (uint32_t)(e[u] & 31)) & ((1u << AE) - 1u);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (e[u] < 0) continue;
            if (mrow) mask_vec<DT>(w[u], bits[u]);
            float x[AE];
            E::unpack(w[u], x);
#pragma unroll
            for (int t = 0; t < AE; ++t)
                if (x[t] == x[t] && x[t] > -INFINITY) f(x[t], (uint32_t)(e[u] + t));
        }
    }
}

// The same walk, warp-uniform: f(x, i, valid) is called by all 32 lanes of a
// warp together for every element slot (valid false for masked, NaN or absent
// ones), so that f may use warp collectives.
template <int DT, class F>
__device__ __forceinline__ void scan_row_warp(const uint8_t *rp, const int32_t *mrow, int32_t V, F &&f) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    const int tid = threadIdx.x;
    const Slice32 g = make_slice32<AE, E::SIZE>(rp, V, 0, 1);
    {  // the head and tail elements (fewer than AE each), in the first warp
        float x = -INFINITY;
        int32_t i = -1;
        if (tid < g.head) i = tid;
        else if (tid >= 8 && tid < 8 + g.tail) i = g.head + g.nvec * AE + (tid - 8);
        if (i >= 0) {
            x = E::load1(rp, i);
            if (mrow && !(((uint32_t)__ldg(mrow + (i >> 5)) >> (i & 31)) & 1u)) x = -INFINITY;
        }
        if (tid < 32) f(x, (uint32_t)(i >= 0 ? i : 0), i >= 0 && x == x && x > -INFINITY);
    }
    constexpr int kU = 4;
    for (int32_t v0 = 0; v0 < g.nvec; v0 += kThreads * kU) {
        uint4 w[kU];
        uint32_t bits[kU];
        int32_t e[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int32_t v = v0 + tid + u * kThreads;
            e[u] = v < g.nvec ? g.head + v * AE : -1;
            bits[u] = (1u << AE) - 1u;
            w[u] = make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
            if (e[u] >= 0) {
                w[u] = __ldcs(reinterpret_cast<const uint4 *>(rp + (size_t)e[u] * E::SIZE));
                if (mrow) {
                    const uint32_t lo = (uint32_t)__ldg(mrow + (e[u] >> 5));
                    const uint32_t hi = ((e[u] & 31) + AE > 32) ? (uint32_t)__ldg(mrow + (e[u] >> 5) + 1) : 0u;
                    bits[u] = __funnelshift_r(lo, hi, (uint32_t)(e[u] & 31)) & ((1u << AE) - 1u);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (e[u] >= 0 && mrow) mask_vec<DT>(w[u], bits[u]);
            float x[AE];
            E::unpack(w[u], x);
#pragma unroll
            for (int t = 0; t < AE; ++t)
                f(x[t], (uint32_t)(e[u] + t), e[u] >= 0 && x[t] == x[t] && x[t] > -INFINITY);
        }
    }
}

// Exact 64-bit add into shared memory as two native 32-bit atomics (the low
// word, then the high word plus the carry out of this add): every wrap of the
// low word is counted once.  Much faster here than a 64-bit shared atomic add.
__device__ __forceinline__ void atomic_add_u64_split(unsigned long long *p, unsigned long long v) {
    uint32_t *w = reinterpret_cast<uint32_t *>(p);
    const uint32_t lo = (uint32_t)v, old = atomicAdd(w, lo);
    const uint32_t hi = (uint32_t)(v >> 32) + ((uint32_t)(old + lo) < old ? 1u : 0u);
    if (hi) atomicAdd(w + 1, hi);
}

// 2,048-bin histograms of one 11-bit digit of the order key (24 KB).
constexpr int kGBins = 2048;
struct GHist {
    uint32_t cnt[kGBins];
    unsigned long long mass[kGBins];
};
constexpr int kGPerThread = kGBins / kThreads;  // bins owned by each thread in the selection

// The digit D holding the `need`-th largest key (counting from 1, within the
// current prefix); `above` = keys in digits above D.
template <class Sync>
__device__ __forceinline__ uint32_t ghist_count_digit(const GHist &h, uint64_t need, Scratch &sc, uint64_t &above) {
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    uint32_t c[kGPerThread];
    uint64_t mine = 0;
#pragma unroll
    for (int b = 0; b < kGPerThread; ++b) {
        c[b] = h.cnt[tid * kGPerThread + b];
        mine += c[b];
    }
    // suffix over threads (higher threads own higher digits)
    uint64_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (l + o < 32) incl += t;
    }
    Sync::sync();
    if (l == 0) sc.r64[w] = incl;
    if (tid == 0) sc.u0 = 0xFFFFFFFFu;
    Sync::sync();
    uint64_t run = incl - mine;
#pragma unroll
    for (int i = 0; i < kWarps; ++i)
        if (i > w) run += sc.r64[i];
#pragma unroll
    for (int b = kGPerThread - 1; b >= 0; --b) {
        if (c[b] > 0 && run < need && need <= run + c[b]) {
            sc.u0 = (uint32_t)(tid * kGPerThread + b);
            sc.above = run;
        }
        run += c[b];
    }
    Sync::sync();
    const uint32_t D = sc.u0;
    above = D < (uint32_t)kGBins ? sc.above : 0ull;
    Sync::sync();
    return D;
}

// The lowest non-empty digit D whose mass strictly above (base + digits above
// D) is still below pz; `above` = mass in digits above D.  0xFFFFFFFF if none.
template <class Sync>
__device__ __forceinline__ uint32_t ghist_mass_digit(const GHist &h, uint64_t base, double pz, Scratch &sc,
                                                     uint64_t &above) {
    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    uint64_t ms[kGPerThread];
    uint64_t mine = 0;
#pragma unroll
    for (int b = 0; b < kGPerThread; ++b) {
        ms[b] = h.mass[tid * kGPerThread + b];
        mine += ms[b];
    }
    uint64_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (l + o < 32) incl += t;
    }
    Sync::sync();
    if (l == 0) sc.r64[w] = incl;
    if (tid == 0) sc.u0 = 0xFFFFFFFFu;
    Sync::sync();
    uint64_t run = incl - mine;
#pragma unroll
    for (int i = 0; i < kWarps; ++i)
        if (i > w) run += sc.r64[i];
    uint32_t lowest = 0xFFFFFFFFu;
    uint64_t low_above = 0;
#pragma unroll
    for (int b = kGPerThread - 1; b >= 0; --b) {
        const uint32_t d = (uint32_t)(tid * kGPerThread + b);
        if (h.cnt[d] > 0 && (double)(base + run) < pz) {
            lowest = d;
            low_above = run;
        }
        run += ms[b];
    }
    if (lowest != 0xFFFFFFFFu) atomicMin(&sc.u0, lowest);
    Sync::sync();
    const uint32_t D = sc.u0;
    if (D != 0xFFFFFFFFu && lowest == D) sc.above = low_above;
    Sync::sync();
    above = D != 0xFFFFFFFFu ? sc.above : 0ull;
    Sync::sync();
    return D;
}

// General path over the whole row (re-read from global memory): exact radix
// selects of the k-th largest logit (counts) and of the top-p boundary
// (fixed-point masses) on order-preserving keys, 11 bits a pass, then the
// Gumbel-max draw over the kept tokens.  m, its index amax (0xFFFFFFFF if the
// caller did not track it) and Z come from the caller; v_m is the min-p cut
// (or -inf).  NaN logits count as -inf here.
// `scratch` is at least sizeof(GHist) bytes of shared memory, 8-byte aligned,
// free for the duration.
template <int DT, class Sync>
__device__ void general_path(const SampleArgs &a, int64_t row, const RowParams &rpm, float m, uint32_t amax,
                             double Z, float v_m, uint8_t *scratch, SelCtl &ctl, int64_t &token, float &vstar) {
    using E = Elem<DT>;
    GHist &gh = *reinterpret_cast<GHist *>(scratch);
    const int tid = threadIdx.x;
    const int32_t V = (int32_t)a.V;
    const float T = rpm.T, invT = rpm.invT, c2 = rpm.c2;
    const uint8_t *rp = reinterpret_cast<const uint8_t *>(a.logits) + (size_t)row * a.stride * E::SIZE;
    const int32_t *mrow = a.mask ? a.mask + (size_t)row * a.mstride : nullptr;
    // digits: key bits [31:21], [20:10], [9:0]; widened bf16 / f16 keys end in
    // at least 13 zero bits, so two passes resolve them
    constexpr int kPasses = DT == 0 ? 3 : 2;
    auto digit_shift = [](int p) { return p == 0 ? 21 : (p == 1 ? 10 : 0); };
    auto digit_mask = [](int p) { return p == 2 ? 1023u : (uint32_t)(kGBins - 1); };
    // the value of a resolved key prefix: for bf16 / f16 the unresolved low
    // bits of a key are all zero (positive values) or all one (negative ones,
    // whose keys are inverted)
    auto prefix_value = [](uint32_t prefix) {
        return okey_value(kPasses == 3 ? prefix : (prefix | ((prefix & 0x80000000u) ? 0u : 0x3FFu)));
    };
    auto clear_hist = [&](bool mass) {
        for (int i = tid; i < kGBins; i += kThreads) {
            gh.cnt[i] = 0;
            if (mass) gh.mass[i] = 0ull;
        }
        Sync::sync();
    };
    float lo_v = v_m;
    float v_k = -INFINITY;
    if (rpm.k_on) {
        uint32_t prefix = 0;
        uint64_t need = (uint64_t)rpm.K;
        bool all_kept = false;
        for (int p = 0; p < kPasses; ++p) {
            const int shift = digit_shift(p);
            const uint32_t hmask = p ? (0xFFFFFFFFu << (shift + (p == 1 ? 11 : 10))) : 0u;
            clear_hist(false);
            // lanes holding the same key add together, through one lane
            scan_row_warp<DT>(rp, mrow, V, [&](float x, uint32_t, bool valid) {
                const uint32_t kk = okey(x);
                const bool on = valid && x >= lo_v && (kk & hmask) == (prefix & hmask);
                if (!__any_sync(0xFFFFFFFFu, on)) return;
                const uint32_t same = __match_any_sync(0xFFFFFFFFu, on ? kk : 0u);
                if (on && (threadIdx.x & 31) == __ffs(same) - 1)
                    atomicAdd(&gh.cnt[(kk >> shift) & digit_mask(p)], (uint32_t)__popc(same));
            });
            Sync::sync();
            if (p == 0) {  // no more than k candidates: top-k keeps them all
                uint32_t tot = 0;
                for (int i = tid; i < kGBins; i += kThreads) tot += gh.cnt[i];
                if (block_sum_f32<Sync>((float)tot, ctl.sc) <= (float)rpm.K) {
                    all_kept = true;
                    break;
                }
            }
            uint64_t above = 0;
            const uint32_t D = ghist_count_digit<Sync>(gh, need, ctl.sc, above);
            prefix |= D << shift;
            need -= above;
        }
        if (!all_kept) v_k = prefix_value(prefix);
    }
    lo_v = fmaxf(lo_v, v_k);
    float v_p = -INFINITY;
    if (rpm.p_on) {
        if (!(rpm.P > 0.f)) {
            v_p = m;
        } else {
            const double pz = (double)rpm.P * Z * (double)kMassScale;
            uint32_t prefix = 0;
            uint64_t mass_above = 0;
            bool found = true;
            for (int p = 0; p < kPasses; ++p) {
                const int shift = digit_shift(p);
                const uint32_t hmask = p ? (0xFFFFFFFFu << (shift + (p == 1 ? 11 : 10))) : 0u;
                clear_hist(true);
                // lanes holding the same key (hence the same mass) add together,
                // through one lane: count and count * mass, exact in fixed point
                scan_row_warp<DT>(rp, mrow, V, [&](float x, uint32_t, bool valid) {
                    const uint32_t kk = okey(x);
                    const bool on = valid && x >= lo_v && (kk & hmask) == (prefix & hmask);
                    if (!__any_sync(0xFFFFFFFFu, on)) return;
                    const uint32_t same = __match_any_sync(0xFFFFFFFFu, on ? kk : 0u);
                    if (on && (threadIdx.x & 31) == __ffs(same) - 1) {
                        const uint32_t d = (kk >> shift) & digit_mask(p);
                        const uint32_t n = (uint32_t)__popc(same);
                        atomicAdd(&gh.cnt[d], n);
                        atomic_add_u64_split(&gh.mass[d], (unsigned long long)n *
                                             (unsigned long long)(ex2_approx((x - m) * c2) * kMassScale));
                    }
                });
                Sync::sync();
                uint64_t above = 0;
                const uint32_t D = ghist_mass_digit<Sync>(gh, mass_above, pz, ctl.sc, above);
                if (D == 0xFFFFFFFFu) {  // unreachable for p > 0: the top digit has no mass above
                    found = false;
                    break;
                }
                prefix |= D << shift;
                mass_above += above;
            }
            v_p = found ? fminf(prefix_value(prefix), m) : m;
        }
    }
    vstar = fmaxf(lo_v, v_p);
    // Gumbel-max over the row's kept tokens; each thread's elements arrive in
    // increasing index order within a vector, so a Philox block is computed
    // once for up to four consecutive tokens
    // the argmax is always kept, so its score seeds the pruning; an unknown
    // argmax (0xFFFFFFFF) starts from no token
    float best_sc = -INFINITY;
    uint32_t bi = 0xFFFFFFFFu;
    if (amax != 0xFFFFFFFFu) {
        const uint4 blk_a = token_block(a.seed, a.offset, (uint32_t)row, amax >> 2);
        best_sc = gumbel_of(block_word(blk_a, amax & 3));
        bi = amax;
    }
    float cut = fmaf(best_sc - kGumbelMax, T, m);
    uint32_t q_cached = 0xFFFFFFFFu;
    uint4 blk = make_uint4(0, 0, 0, 0);
    const float vs = vstar;
    scan_row<DT>(rp, mrow, V, [&](float x, uint32_t i) {
        if (!(x >= vs) || !(x >= cut)) return;
        if ((i >> 2) != q_cached) {
            q_cached = i >> 2;
            blk = token_block(a.seed, a.offset, (uint32_t)row, q_cached);
        }
        const uint32_t word = block_word(blk, i & 3);
        const float srel = (x - m) * invT;
        const float need = best_sc - srel;
        if (need > kTopBitsMargin && (word >> 22) != 0x3FFu) return;
        if (word_uniform(word) < gumbel_u_floor(need)) return;
        const float sc = srel + gumbel_of(word);
        if (sc > best_sc || (sc == best_sc && i < bi)) {
            best_sc = sc;
            bi = i;
            cut = fmaf(best_sc - kGumbelMax, T, m);
        }
    });
    token = rank_key_index(block_max_u64<Sync>(rank_key(best_sc, bi), ctl.sc));
}

}  // namespace sample_detail
}  // namespace tsa
