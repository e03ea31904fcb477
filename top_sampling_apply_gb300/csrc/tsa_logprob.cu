// selective log-softmax (selective_log_softmax, "Selective Log Softmax" and
// "Online log-sum-exp"): one log-probability per row, the row's logit at a
// given index less the log-sum-exp of the row, here over the allowed tokens
// of the temperature-scaled row:
//     out[b] = (l[b, i_b] - m_b) / T_b - ln sum_{j allowed} exp((l[b, j] - m_b) / T_b)
// with m_b the row's largest allowed logit.  T_b <= 0 (greedy rows of
// sample) uses T = 1, the page's unscaled definition.  NaN logits count as
// -inf; a disallowed index gives -inf; an index outside [0, V) or a row with
// no allowed finite logit gives NaN.
//
// One CTA of 512 threads per row streams the row once with 16-byte vector
// loads, eight in flight per thread (64 KB a CTA; 256 threads with four loads
// a thread kept too few bytes in flight and reached a fifth of HBM).  Each
// thread sums 2^((l - ref) log2(e) / T) against a reference ref that moves
// only when a term would pass 2^64, so a new maximum costs nothing on the
// common path; block reductions then form the row maximum and the
// normaliser, and thread 0 reads the indexed logit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_host.h"
#include "tsa_sample_common.cuh"

namespace tsa {

using namespace sample_detail;

namespace {
constexpr float kLsmSpan = 64.f;   // the reference moves when a term would pass 2^kLsmSpan
constexpr int kLsmThreads = 512;   // a row's threads
constexpr int kLsmU = 8;           // 16-byte vectors in flight per thread (64 KB a CTA)
constexpr int kLsmWarps = kLsmThreads / 32;
}  // namespace

template <int DT>
__global__ void __launch_bounds__(kLsmThreads) logprob_kernel(const void *logits, int64_t V, int64_t stride,
                                                              const int32_t *mask, int64_t mstride,
                                                              const float *temperature, float temperature_s,
                                                              const int64_t *index, float *out) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    __shared__ float s_red[kLsmWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;
    const uint8_t *rp = reinterpret_cast<const uint8_t *>(logits) + (size_t)row * stride * E::SIZE;
    const int32_t *mrow = mask ? mask + (size_t)row * mstride : nullptr;
    float T = temperature ? temperature[row] : temperature_s;
    if (!(T > 0.f)) T = 1.f;
    const float c2 = kLog2e / T, span = kLsmSpan / c2;
    float mx = -INFINITY, ref = -INFINITY, rhi = -INFINITY, s = 0.f;
    auto take = [&](float x) {
        if (!(x == x) || !(x > -INFINITY)) return;  // NaN and disallowed (-inf) add nothing
        mx = fmaxf(mx, x);
        if (x > rhi) {  // rare: the thread's first values, or a jump of 2^64
            s *= ex2_approx((ref - x) * c2);
            ref = x;
            rhi = x + span;
        }
        s += ex2_approx((x - ref) * c2);
    };
    // a whole vector, without a branch per element: NaN becomes -inf, and the
    // reference check is made once on the vector's maximum.  The exponent is
    // (x - ref) c2, not x c2 - ref c2: the product ref c2 would be rounded once
    // and scale every term alike, by up to |ref c2| 2^-24.
    auto take_vec = [&](float (&x)[AE]) {
        float vmax = -INFINITY;
#pragma unroll
        for (int t = 0; t < AE; ++t) {
            x[t] = x[t] == x[t] ? x[t] : -INFINITY;
            vmax = fmaxf(vmax, x[t]);
        }
        mx = fmaxf(mx, vmax);
        if (vmax > rhi) {
            s *= ex2_approx((ref - vmax) * c2);
            ref = vmax;
            rhi = vmax + span;
        }
        if (ref > -INFINITY) {  // else the vector holds no allowed finite value yet
#pragma unroll
            for (int t = 0; t < AE; ++t) s += ex2_approx((x[t] - ref) * c2);
        }
    };
    const Slice32 g = make_slice32<AE, E::SIZE>(rp, (int32_t)V, 0, 1);
    auto scalar = [&](int32_t i) {
        float x = E::load1(rp, i);
        if (mrow && !(((uint32_t)__ldg(mrow + (i >> 5)) >> (i & 31)) & 1u)) x = -INFINITY;
        take(x);
    };
    if (tid < g.head) scalar(tid);
    if (tid < g.tail) scalar(g.head + g.nvec * AE + tid);
    for (int32_t v0 = 0; v0 < g.nvec; v0 += kLsmThreads * kLsmU) {
        uint4 w[kLsmU];
        uint32_t bits[kLsmU];
        int32_t e[kLsmU];
#pragma unroll
        for (int u = 0; u < kLsmU; ++u) {
            const int32_t v = v0 + tid + u * kLsmThreads;
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
        for (int u = 0; u < kLsmU; ++u) {
            if (e[u] < 0) continue;
            if (mrow) mask_vec<DT>(w[u], bits[u]);
            float x[AE];
            E::unpack(w[u], x);
            take_vec(x);
        }
    }
    // the row maximum, then the normaliser against it
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kLsmWarps; ++i) m = fmaxf(m, s_red[i]);
    __syncthreads();
    float part = (ref > -INFINITY && m > -INFINITY) ? s * ex2_approx((ref - m) * c2) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
    if (lane == 0) s_red[warp] = part;
    __syncthreads();
    if (tid == 0) {
        float Z = 0.f;
        for (int i = 0; i < kLsmWarps; ++i) Z += s_red[i];
        const int64_t i = index[row];
        float r = __int_as_float(0x7FC00000);
        if (i >= 0 && i < V && m > -INFINITY) {
            float x = E::load1(rp, (int32_t)i);
            if (mrow && !(((uint32_t)mrow[i >> 5] >> (i & 31)) & 1u)) x = -INFINITY;
            if (!(x == x)) x = -INFINITY;
            r = x > -INFINITY ? (x - m) / T - logf(Z) : -INFINITY;
        }
        out[row] = r;
    }
}

int logprob_launch(const void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                   int64_t mstride, const float *temperature, float temperature_s, const int64_t *index,
                   float *out, cudaStream_t st) {
    const dim3 grid((unsigned)B), block(kLsmThreads);
    if (dtype == 0)
        logprob_kernel<0><<<grid, block, 0, st>>>(logits, V, stride, mask, mstride, temperature, temperature_s,
                                                  index, out);
    else if (dtype == 1)
        logprob_kernel<1><<<grid, block, 0, st>>>(logits, V, stride, mask, mstride, temperature, temperature_s,
                                                  index, out);
    else
        logprob_kernel<2><<<grid, block, 0, st>>>(logits, V, stride, mask, mstride, temperature, temperature_s,
                                                  index, out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tsa
