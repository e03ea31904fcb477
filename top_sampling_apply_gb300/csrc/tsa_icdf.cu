// logits-mask-xpu, "Usage" (bitmask_from_allowed: a bool allow-set packed one
// bit per token) and "Method" (the inverse-CDF draw from a caller uniform:
// chunk masses, a scan over them to the chunk holding the target, and a walk
// of that chunk alone).
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_host.h"

namespace tsa {

namespace {

// Packing: a warp forms one 32-bit word per step, lane j reading token 32 w + j
// of the row (32 consecutive bytes per step) and the ballot giving the word.
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *allowed, int64_t B, int64_t V, int64_t astride,
                                                   int32_t *bits, int64_t wstride, int64_t W) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t g = warp0; g < B * W; g += nwarps) {
        const int64_t b = g / W, w = g - b * W;
        const int64_t i = w * 32 + lane;
        const bool on = i < V && __ldg(allowed + b * astride + i) != 0;
        const uint32_t word = __ballot_sync(0xFFFFFFFFu, on);
        if (lane == 0) bits[b * wstride + w] = (int32_t)word;
    }
}

// Packing, rows 4-byte aligned and V a multiple of 4: a warp forms four words
// per step, lane l reading tokens 128 s + 4 l .. 4 l + 3 in one 4-byte load;
// each lane makes their four bits, and eight lanes OR theirs into a word.
// Blocks are laid out (steps of a row, rows); a warp takes kPackU consecutive
// steps of one row and issues all their loads before it packs any.
constexpr int kPackU = 8;
__global__ void __launch_bounds__(256) pack4_kernel(const uint8_t *allowed, int64_t B, int64_t V, int64_t astride,
                                                    int32_t *bits, int64_t wstride, int64_t W) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t steps = (W + 3) / 4;
    const int64_t s0 = ((int64_t)blockIdx.x * 8 + warp) * kPackU;
    if (s0 >= steps) return;  // the whole warp
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        const uint8_t *row = allowed + b * astride;
        uint32_t v[kPackU];
#pragma unroll
        for (int u = 0; u < kPackU; ++u) {
            const int64_t t0 = (s0 + u) * 128 + lane * 4;
            v[u] = t0 < V ? __ldg(reinterpret_cast<const uint32_t *>(row + t0)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kPackU; ++u) {
            uint32_t x = ((v[u] & 0xFFu) ? 1u : 0u) | ((v[u] & 0xFF00u) ? 2u : 0u) |
                         ((v[u] & 0xFF0000u) ? 4u : 0u) | ((v[u] & 0xFF000000u) ? 8u : 0u);
            x <<= 4 * (lane & 7);
            x |= __shfl_xor_sync(0xFFFFFFFFu, x, 1);
            x |= __shfl_xor_sync(0xFFFFFFFFu, x, 2);
            x |= __shfl_xor_sync(0xFFFFFFFFu, x, 4);
            const int64_t w = (s0 + u) * 4 + (lane >> 3);
            if ((lane & 7) == 0 && w < W) bits[b * wstride + w] = (int32_t)x;
        }
    }
}

constexpr int kIcdfThreads = 512;
constexpr int kIcdfWarps = kIcdfThreads / 32;
constexpr int kIcdfBlocks = 64;  // recorded blocks of batches per warp chunk
constexpr float kIcdfLog2e = 1.4426950408889634f;

// Compensated fp32 sum (two-sum): hi + lo carries the sum to about 2^-44.
struct Sum2 {
    float hi, lo;
};
__device__ __forceinline__ Sum2 sum2_add(Sum2 a, float b) {
    const float s = a.hi + b;
    const float bb = s - a.hi;
    const float err = (a.hi - (s - bb)) + (b - bb);
    return Sum2{s, a.lo + err};
}

struct IcdfShared {
    float bm[kIcdfWarps][kIcdfBlocks];  // per recorded block: its warp's running maximum at the block's end
    float bs[kIcdfWarps][kIcdfBlocks];  // and the block's mass against that maximum
    float wm[kIcdfWarps];               // each warp's maximum kept logit
    float M;                            // the row's maximum kept logit
    float target, before_hi, before_lo;  // u W; the mass before the chosen block
    int chunk, block;                   // the warp chunk and its block holding the target
};

// One CTA per row.  Warp w owns the contiguous chunk [w C, (w + 1) C) of the
// row.  A step of the warp covers 32 NE consecutive tokens, NE to a lane (NE =
// a 16-byte vector's worth when every row is 16-byte aligned and V a multiple
// of it, else 1), and an iteration a batch of kIcdfBatch steps whose loads are
// in flight together.  One read forms the mass of every block of batches (at
// most kIcdfBlocks a chunk) against the warp's running maximum; thread 0 then
// scans chunks and blocks in index order for the block holding u W, and one
// warp walks that block again, a step at a time with a warp scan over the
// lanes' sums, to the first kept token whose running mass passes u W.  Kept:
// allowed, finite, logit >= v* (the keep-threshold of the sample call that ran
// before).
template <int DT, bool MASK, bool VEC>
__global__ void __launch_bounds__(kIcdfThreads, 2) icdf_kernel(IcdfArgs a) {
    using E = Elem<DT>;
    constexpr int NE = VEC ? E::AE : 1;
    // steps a batch, their loads in flight together: 32 values a lane (eight
    // 16-byte loads for f32, four for 16-bit types, eight single tokens)
    constexpr int kIcdfBatch = VEC ? 32 / NE : 8;
    __shared__ IcdfShared sh;
    const int64_t row = blockIdx.x;
    const float T = a.temperature ? a.temperature[row] : a.temperature_s;
    const int32_t K = a.top_k ? a.top_k[row] : a.top_k_s;
    const float vs = a.vstar[row];
    // greedy rows (their token is the argmax) and empty rows (-1) keep what the
    // sample call wrote
    if (!(T > 0.f) || K == 1 || vs != vs) return;
    const float c2 = (1.f / T) * kIcdfLog2e;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t V = a.V;
    const uint8_t *rp = reinterpret_cast<const uint8_t *>(a.logits) + (size_t)row * a.stride * E::SIZE;
    const int32_t *mrow = a.mask ? a.mask + (size_t)row * a.mstride : nullptr;
    constexpr int64_t kStep = 32 * NE, kB = kStep * kIcdfBatch;
    const int64_t C = ((V + kIcdfWarps - 1) / kIcdfWarps + kB - 1) / kB * kB;  // whole batches a chunk
    const int64_t nbat = C / kB;
    const int64_t bpb = (nbat + kIcdfBlocks - 1) / kIcdfBlocks;  // batches a recorded block
    // this lane's NE tokens of the step at s0 (kept logits, else -inf); the
    // loads are unconditional within the row, so a batch of them is in flight
    // together
    struct Step {
        float x[NE];
    };
    auto load_step = [&](int64_t s0) -> Step {
        Step r;
        float *x = r.x;
        const int64_t e = s0 + (int64_t)lane * NE;
        if (VEC) {
            // V is a multiple of NE: a vector is wholly inside or outside the row
            if (e < V) {
                E::unpack(__ldg(reinterpret_cast<const uint4 *>(rp + (size_t)e * E::SIZE)), x);
                uint32_t bits = (1u << NE) - 1u;
                if (MASK) bits = ((uint32_t)__ldg(mrow + (e >> 5)) >> (e & 31)) & ((1u << NE) - 1u);
#pragma unroll
                for (int t = 0; t < NE; ++t)
                    x[t] = (((bits >> t) & 1u) && x[t] >= vs && x[t] < INFINITY) ? x[t] : -INFINITY;
            } else {
#pragma unroll
                for (int t = 0; t < NE; ++t) x[t] = -INFINITY;
            }
        } else {
            float v = -INFINITY;
            if (e < V) {
                v = E::load1(rp, e);
                bool keep = v >= vs && v < INFINITY;
                if (MASK) keep = keep & ((((uint32_t)__ldg(mrow + (e >> 5))) >> (e & 31)) & 1u);
                if (!keep) v = -INFINITY;
            }
            x[0] = v;
        }
        return r;
    };
    const int64_t c0 = (int64_t)warp * C;
    for (int b = lane; b < kIcdfBlocks; b += 32) {
        sh.bm[warp][b] = -INFINITY;
        sh.bs[warp][b] = 0.f;
    }
    __syncwarp();
    // one read: the warp's running maximum m (warp-uniform) and each recorded
    // block's mass against it (rescaled when m grows)
    float m = -INFINITY, blk = 0.f;
    for (int64_t bt = 0; bt < nbat && c0 + bt * kB < V; ++bt) {
        Step xs[kIcdfBatch];
#pragma unroll
        for (int u = 0; u < kIcdfBatch; ++u) xs[u] = load_step(c0 + bt * kB + u * kStep);
        float lm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kIcdfBatch; ++u)
#pragma unroll
            for (int t = 0; t < NE; ++t) lm = fmaxf(lm, xs[u].x[t]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lm = fmaxf(lm, __shfl_xor_sync(0xFFFFFFFFu, lm, o));
        if (lm > m) {
            if (m > -INFINITY) blk *= ex2_approx((m - lm) * c2);
            m = lm;
        }
        float ls = 0.f;
        if (m > -INFINITY) {
#pragma unroll
            for (int u = 0; u < kIcdfBatch; ++u)
#pragma unroll
                for (int t = 0; t < NE; ++t)
                    if (xs[u].x[t] > -INFINITY) ls += ex2_approx((xs[u].x[t] - m) * c2);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, o);
        blk += ls;
        if ((bt + 1) % bpb == 0 || bt + 1 == nbat || c0 + (bt + 1) * kB >= V) {
            if (lane == 0) {
                sh.bm[warp][bt / bpb] = m;
                sh.bs[warp][bt / bpb] = blk;
            }
            blk = 0.f;
        }
    }
    if (lane == 0) sh.wm[warp] = m;
    __syncthreads();
    if (warp == 0) {
        // Warp 0 finds the total W and the first block (index order: chunk,
        // then block) where the running mass passes u W, or the last block
        // with mass when rounding leaves it unpassed.  Lane l takes the 32
        // consecutive blocks from 32 l on; a warp scan of the lanes'
        // compensated sums places each lane's run.
        static_assert(kIcdfWarps * kIcdfBlocks == 32 * 32, "32 recorded blocks a lane");
        float M = -INFINITY;
        for (int w = 0; w < kIcdfWarps; ++w) M = fmaxf(M, sh.wm[w]);
        auto mass_of = [&](int e) -> float {
            const int w = e / kIcdfBlocks, b = e % kIcdfBlocks;
            return sh.bm[w][b] > -INFINITY ? sh.bs[w][b] * ex2_approx((sh.bm[w][b] - M) * c2) : 0.f;
        };
        Sum2 mine{0.f, 0.f};
        bool any = false;
        for (int j = 0; j < 32; ++j) {
            const float ms = mass_of(32 * lane + j);
            if (ms > 0.f) {
                mine = sum2_add(mine, ms);
                any = true;
            }
        }
        Sum2 incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float hi = __shfl_up_sync(0xFFFFFFFFu, incl.hi, o), lo = __shfl_up_sync(0xFFFFFFFFu, incl.lo, o);
            if (lane >= o) {
                incl = sum2_add(incl, hi);
                incl.lo += lo;
            }
        }
        const float tot = __shfl_sync(0xFFFFFFFFu, incl.hi + incl.lo, 31);
        const float th = a.uniform[row] * tot;
        Sum2 excl{__shfl_up_sync(0xFFFFFFFFu, incl.hi, 1), __shfl_up_sync(0xFFFFFFFFu, incl.lo, 1)};
        if (lane == 0) excl = Sum2{0.f, 0.f};
        const uint32_t passes = __ballot_sync(0xFFFFFFFFu, any && incl.hi + incl.lo > th);
        const uint32_t with_mass = __ballot_sync(0xFFFFFFFFu, any);
        // the lane holding the block: the first that passes, else the last with mass
        const int L = passes ? __ffs(passes) - 1 : (with_mass ? 31 - __clz(with_mass) : -1);
        if (L < 0 && lane == 0) sh.chunk = -1;  // no kept mass at all
        if (lane == L) {
            Sum2 run = excl, before = excl, before_last = excl;
            int ce = -1, le = -1;
            for (int j = 0; j < 32; ++j) {
                const float ms = mass_of(32 * lane + j);
                if (!(ms > 0.f)) continue;
                const Sum2 next = sum2_add(run, ms);
                le = 32 * lane + j;
                before_last = run;
                if (next.hi + next.lo > th) {
                    ce = le;
                    before = run;
                    break;
                }
                run = next;
            }
            if (ce < 0) {
                ce = le;
                before = before_last;
            }
            sh.M = M;
            sh.chunk = ce / kIcdfBlocks;
            sh.block = ce % kIcdfBlocks;
            sh.target = th;
            sh.before_hi = before.hi;
            sh.before_lo = before.lo;
        }
    }
    __syncthreads();
    if (warp != sh.chunk) return;
    // the walk over the chosen block: a step at a time in index order, the
    // running mass starting from everything before the block
    const float M = sh.M, th = sh.target;
    Sum2 run{sh.before_hi, sh.before_lo};
    int64_t last_kept = -1;
    bool done = false;  // warp-uniform
    const int64_t bt0 = (int64_t)sh.block * bpb;
    for (int64_t bt = bt0; !done && bt < bt0 + bpb && bt < nbat && c0 + bt * kB < V; ++bt) {
        Step xs[kIcdfBatch];
#pragma unroll
        for (int u = 0; u < kIcdfBatch; ++u) xs[u] = load_step(c0 + bt * kB + u * kStep);
#pragma unroll
        for (int u = 0; u < kIcdfBatch; ++u) {
            const int64_t s0 = c0 + bt * kB + u * kStep;
            float w[NE], ls = 0.f;
            int last_t = -1;
#pragma unroll
            for (int t = 0; t < NE; ++t) {
                const bool has = xs[u].x[t] > -INFINITY;
                w[t] = has ? ex2_approx((xs[u].x[t] - M) * c2) : 0.f;
                ls += w[t];
                if (has) last_t = t;
            }
            float incl = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t2 = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += t2;
            }
            // the first lane with a kept token whose running mass passes the
            // target, then the token inside that lane
            const Sum2 mine = sum2_add(run, incl);
            const uint32_t pass = __ballot_sync(0xFFFFFFFFu, !done && last_t >= 0 && mine.hi + mine.lo > th);
            const uint32_t any = __ballot_sync(0xFFFFFFFFu, last_t >= 0);
            if (pass) {
                const int L = __ffs(pass) - 1;
                if (lane == L) {
                    Sum2 acc = sum2_add(run, incl - ls);
                    int pick = last_t;  // rounding may leave the target unpassed inside the lane
                    float cum = 0.f;
                    int found = -1;
#pragma unroll
                    for (int t = 0; t < NE; ++t) {
                        if (!(xs[u].x[t] > -INFINITY)) continue;
                        cum += w[t];
                        const Sum2 at = sum2_add(acc, cum);
                        if (found < 0 && at.hi + at.lo > th) found = t;
                    }
                    if (found >= 0) pick = found;
                    a.tokens[row] = s0 + (int64_t)L * NE + pick;
                }
                done = true;
            }
            if (!done && any) {
                const int L = 31 - __clz(any);
                const int lt = __shfl_sync(0xFFFFFFFFu, last_t, L);
                last_kept = s0 + (int64_t)L * NE + lt;
            }
            run = sum2_add(run, __shfl_sync(0xFFFFFFFFu, incl, 31));
        }
    }
    if (!done && lane == 0 && last_kept >= 0) a.tokens[row] = last_kept;
}

}  // namespace

int pack_launch(const uint8_t *allowed, int64_t B, int64_t V, int64_t astride, int32_t *bits, int64_t wstride,
                cudaStream_t st) {
    const int64_t W = (V + 31) / 32;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if ((reinterpret_cast<uintptr_t>(allowed) % 4) == 0 && astride % 4 == 0 && V % 4 == 0) {
        // (steps of a row / (8 warps x kPackU), rows), rows strided past 65,535
        const int64_t steps = (W + 3) / 4;
        const dim3 grid((unsigned)((steps + 8 * kPackU - 1) / (8 * kPackU)), (unsigned)(B < 65535 ? B : 65535));
        pack4_kernel<<<grid, 256, 0, st>>>(allowed, B, V, astride, bits, wstride, W);
    } else {
        int64_t blocks = (B * W + 7) / 8;  // a word per warp, 8 warps per block
        const int64_t cap = (int64_t)sms * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        pack_kernel<<<(unsigned)blocks, 256, 0, st>>>(allowed, B, V, astride, bits, wstride, W);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int icdf_launch(const IcdfArgs &args, int dtype, cudaStream_t st) {
    const dim3 grid((unsigned)args.B);
    const bool m = args.mask != nullptr;
    // vector loads when every row starts 16-byte aligned and holds whole vectors
    const int es = dtype == 0 ? 4 : 2, ae = 16 / es;
    const bool vec = (reinterpret_cast<uintptr_t>(args.logits) % 16) == 0 && (args.stride * es) % 16 == 0 &&
                     args.V % ae == 0;
#define TSA_ICDF(D) \
    (vec ? (m ? icdf_kernel<D, true, true><<<grid, kIcdfThreads, 0, st>>>(args) \
              : icdf_kernel<D, false, true><<<grid, kIcdfThreads, 0, st>>>(args)) \
         : (m ? icdf_kernel<D, true, false><<<grid, kIcdfThreads, 0, st>>>(args) \
              : icdf_kernel<D, false, false><<<grid, kIcdfThreads, 0, st>>>(args)))
    if (dtype == 0) TSA_ICDF(0);
    else if (dtype == 1) TSA_ICDF(1);
    else TSA_ICDF(2);
#undef TSA_ICDF
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tsa
