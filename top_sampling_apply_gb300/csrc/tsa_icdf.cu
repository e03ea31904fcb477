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

constexpr int kIcdfThreads = 256;
constexpr int kIcdfBatch = 8;  // loads in flight a lane
constexpr int kIcdfWarps = kIcdfThreads / 32;
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
__device__ __forceinline__ Sum2 sum2_scale(Sum2 a, float f) { return Sum2{a.hi * f, a.lo * f}; }
__device__ __forceinline__ Sum2 sum2_merge(Sum2 a, Sum2 b) {
    Sum2 r = sum2_add(a, b.hi);
    r.lo += b.lo;
    return r;
}

struct IcdfShared {
    float wm[kIcdfWarps];  // each warp's maximum kept logit
    float whi[kIcdfWarps], wlo[kIcdfWarps];  // and its kept mass against that maximum
    float M;           // the row's maximum kept logit
    float target_hi, target_lo, before_hi, before_lo;  // u W; the mass before the chosen chunk
    int chunk;         // the warp chunk holding the target (-1: none)
};

// One CTA per row.  Warp w owns the contiguous chunk [w C, (w + 1) C) of the
// row, its lanes reading 32 consecutive tokens per step.  One read forms each
// chunk's maximum and mass (online, against a running maximum); thread 0 then
// scans the chunks in index order for the one holding u W, and that warp walks
// its chunk again, 32 tokens a step with a warp scan, to the first kept token
// whose running mass passes u W.  Kept: allowed, finite, logit >= v* (the
// keep-threshold of the sample call that ran before).
template <int DT, bool MASK>
__global__ void __launch_bounds__(kIcdfThreads) icdf_kernel(IcdfArgs a) {
    using E = Elem<DT>;
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
    const int64_t C = ((V + kIcdfWarps - 1) / kIcdfWarps + 31) & ~(int64_t)31;
    const int64_t c0 = (int64_t)warp * C, c1 = c0 + C < V ? c0 + C : V;
    // the logit if kept, else -inf; both loads unconditional, so that a
    // batch of them is in flight together
    auto kept_value = [&](int64_t i) -> float {
        const float x = E::load1(rp, i);
        bool keep = x >= vs && x < INFINITY;
        if (MASK) keep = keep & ((((uint32_t)__ldg(mrow + (i >> 5))) >> (i & 31)) & 1u);
        return keep ? x : -INFINITY;
    };
    // one read: each lane's maximum and mass against it, merged over the
    // warp; kIcdfBatch loads in flight a lane (a step of the warp covers 32
    // consecutive tokens)
    float m = -INFINITY;
    Sum2 s{0.f, 0.f};
    for (int64_t i0 = c0 + lane; i0 < c1; i0 += 32 * kIcdfBatch) {
        float xs[kIcdfBatch];
#pragma unroll
        for (int u = 0; u < kIcdfBatch; ++u) {
            const int64_t i = i0 + 32 * u;
            xs[u] = i < c1 ? kept_value(i) : -INFINITY;
        }
        float bm = xs[0];
#pragma unroll
        for (int u = 1; u < kIcdfBatch; ++u) bm = fmaxf(bm, xs[u]);
        if (!(bm > -INFINITY)) continue;
        if (bm > m) {
            s = sum2_scale(s, m > -INFINITY ? ex2_approx((m - bm) * c2) : 0.f);
            m = bm;
        }
#pragma unroll
        for (int u = 0; u < kIcdfBatch; ++u)
            if (xs[u] > -INFINITY) s = sum2_add(s, ex2_approx((xs[u] - m) * c2));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        Sum2 s2{__shfl_xor_sync(0xFFFFFFFFu, s.hi, o), __shfl_xor_sync(0xFFFFFFFFu, s.lo, o)};
        const float mm = fmaxf(m, m2);
        if (mm > -INFINITY) {
            s = sum2_merge(sum2_scale(s, m > -INFINITY ? ex2_approx((m - mm) * c2) : 0.f),
                           sum2_scale(s2, m2 > -INFINITY ? ex2_approx((m2 - mm) * c2) : 0.f));
        }
        m = mm;
    }
    if (lane == 0) {
        sh.wm[warp] = m;
        sh.whi[warp] = s.hi;
        sh.wlo[warp] = s.lo;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = -INFINITY;
        for (int w = 0; w < kIcdfWarps; ++w) M = fmaxf(M, sh.wm[w]);
        Sum2 tot{0.f, 0.f}, part[kIcdfWarps];
        for (int w = 0; w < kIcdfWarps; ++w) {
            const float f = sh.wm[w] > -INFINITY ? ex2_approx((sh.wm[w] - M) * c2) : 0.f;
            part[w] = sum2_scale(Sum2{sh.whi[w], sh.wlo[w]}, f);
            tot = sum2_merge(tot, part[w]);
        }
        // the target u W, and the chunk where the running mass passes it (the
        // last chunk with mass when rounding leaves it unpassed)
        const float Wt = tot.hi + tot.lo;
        const float u = a.uniform[row];
        const float th = u * Wt;
        Sum2 run{0.f, 0.f};
        int chunk = -1, last = -1;
        Sum2 before{0.f, 0.f}, before_last{0.f, 0.f};
        for (int w = 0; w < kIcdfWarps; ++w) {
            if (!(part[w].hi > 0.f)) continue;
            const Sum2 next = sum2_merge(run, part[w]);
            last = w;
            before_last = run;
            if (chunk < 0 && next.hi + next.lo > th) {
                chunk = w;
                before = run;
            }
            run = next;
        }
        if (chunk < 0) {
            chunk = last;
            before = before_last;
        }
        sh.M = M;
        sh.chunk = chunk;
        sh.target_hi = th;
        sh.target_lo = 0.f;
        sh.before_hi = before.hi;
        sh.before_lo = before.lo;
    }
    __syncthreads();
    if (warp != sh.chunk) return;
    // the walk: 32 tokens a step, index order, running mass from the chunks
    // before; the loads of kIcdfBatch steps are issued together
    const float M = sh.M, th = sh.target_hi;
    Sum2 run{sh.before_hi, sh.before_lo};
    int64_t last_kept = -1;
    float xs[kIcdfBatch];
    for (int64_t b0 = c0; b0 < c1; b0 += 32) {
        const int step = (int)(((b0 - c0) >> 5) % kIcdfBatch);
        if (step == 0) {
#pragma unroll
            for (int u = 0; u < kIcdfBatch; ++u) {
                const int64_t i = b0 + 32 * u + lane;
                xs[u] = i < c1 ? kept_value(i) : -INFINITY;
            }
        }
        const int64_t i = b0 + lane;
        float x = xs[0];
#pragma unroll
        for (int u = 1; u < kIcdfBatch; ++u) x = step == u ? xs[u] : x;
        const bool has = x > -INFINITY;
        const float w = has ? ex2_approx((x - M) * c2) : 0.f;
        float incl = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t;
        }
        // first kept lane whose running mass passes the target
        const Sum2 mine = sum2_add(run, incl);
        const uint32_t pass = __ballot_sync(0xFFFFFFFFu, has && mine.hi + mine.lo > th);
        const uint32_t any = __ballot_sync(0xFFFFFFFFu, has);
        if (pass) {
            if (lane == 0) a.tokens[row] = b0 + (__ffs(pass) - 1);
            return;
        }
        if (any) last_kept = b0 + (31 - __clz(any));
        run = sum2_add(run, __shfl_sync(0xFFFFFFFFu, incl, 31));
    }
    if (lane == 0 && last_kept >= 0) a.tokens[row] = last_kept;
}

}  // namespace

int pack_launch(const uint8_t *allowed, int64_t B, int64_t V, int64_t astride, int32_t *bits, int64_t wstride,
                cudaStream_t st) {
    const int64_t W = (V + 31) / 32;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (B * W + 7) / 8;  // a word per warp, 8 warps per block
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    pack_kernel<<<(unsigned)blocks, 256, 0, st>>>(allowed, B, V, astride, bits, wstride, W);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int icdf_launch(const IcdfArgs &args, int dtype, cudaStream_t st) {
    const dim3 grid((unsigned)args.B);
    const bool m = args.mask != nullptr;
    if (dtype == 0) m ? icdf_kernel<0, true><<<grid, kIcdfThreads, 0, st>>>(args) : icdf_kernel<0, false><<<grid, kIcdfThreads, 0, st>>>(args);
    else if (dtype == 1) m ? icdf_kernel<1, true><<<grid, kIcdfThreads, 0, st>>>(args) : icdf_kernel<1, false><<<grid, kIcdfThreads, 0, st>>>(args);
    else m ? icdf_kernel<2, true><<<grid, kIcdfThreads, 0, st>>>(args) : icdf_kernel<2, false><<<grid, kIcdfThreads, 0, st>>>(args);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tsa
