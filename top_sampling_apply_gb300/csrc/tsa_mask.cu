// apply_token_bitmask (logits-processor, "API" and "Correctness"): disallowed
// logits become -inf in place; allowed logits are never written.  Its logits
// are never read: a word of all ones costs its 4-byte mask read and no write;
// a word with zero bits writes -inf to exactly those tokens.
//
// Also the bitmask of a per-row logit floor's survivors, the middle step of
// the sequential reading of top-p (logits-processor: the transformers chain).
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_host.h"

namespace tsa {

// A warp takes 32 consecutive mask words (1,024 tokens) of one row: lane l
// loads word l, then for each word j the warp broadcasts it and lane l writes
// -inf to token 32 j + l when its bit is 0, so each store instruction covers
// 32 consecutive tokens.
template <int DT>
__global__ void __launch_bounds__(256) mask_kernel(void *logits, int64_t B, int64_t V, int64_t stride,
                                                   const int32_t *mask, int64_t mstride, int64_t W,
                                                   int64_t chunks_per_row) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t total = B * chunks_per_row;
    for (int64_t g = warp0; g < total; g += nwarps) {
        const int64_t b = g / chunks_per_row, ch = g - b * chunks_per_row;
        const int64_t w0 = ch * 32;
        const int64_t wl = w0 + lane;
        // words past the row's last one read as all-allowed
        const uint32_t mine = wl < W ? (uint32_t)__ldg(mask + b * mstride + wl) : 0xFFFFFFFFu;
        if (__all_sync(0xFFFFFFFFu, mine == 0xFFFFFFFFu)) continue;
        const int64_t base = b * stride;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            const uint32_t word = __shfl_sync(0xFFFFFFFFu, mine, j);
            const int64_t i = (w0 + j) * 32 + lane;
            if (i < V && !((word >> lane) & 1u)) {  // bits at or beyond V are ignored
                if (DT == 0)
                    reinterpret_cast<uint32_t *>(logits)[base + i] = 0xFF800000u;
                else
                    reinterpret_cast<unsigned short *>(logits)[base + i] = (unsigned short)(DT == 1 ? 0xFC00u : 0xFF80u);
            }
        }
    }
}

int mask_launch(void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                int64_t mstride, cudaStream_t st) {
    const int64_t W = (V + 31) / 32;
    const int64_t chunks_per_row = (W + 31) / 32;
    const int64_t total = B * chunks_per_row;  // one warp each
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (total + 7) / 8;  // 8 warps per block
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (dtype == 0)
        mask_kernel<0><<<(unsigned)blocks, 256, 0, st>>>(logits, B, V, stride, mask, mstride, W, chunks_per_row);
    else if (dtype == 1)
        mask_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(logits, B, V, stride, mask, mstride, W, chunks_per_row);
    else
        mask_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(logits, B, V, stride, mask, mstride, W, chunks_per_row);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// The survivors of a per-row logit floor as a bitmask: word w of row b holds
// bit j set iff token 32 w + j is allowed by `mask` (all allowed when NULL),
// lies below V, and its logit is >= floor[b] (NaN never is; a NaN floor keeps
// nothing).  A warp forms one word per ballot: lane j compares token 32 w + j.
constexpr int kFloorU = 8;  // words a warp forms per pass
template <int DT>
__global__ void __launch_bounds__(256) floor_mask_kernel(const void *logits, int64_t B, int64_t V, int64_t stride,
                                                         const int32_t *mask, int64_t mstride, const float *floor,
                                                         int32_t *out, int64_t W) {
    // blocks are laid out (words of a row, rows); a warp takes kFloorU
    // consecutive words of one row and issues all their loads before its
    // ballots, so that each lane has kFloorU reads in flight
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t w0 = ((int64_t)blockIdx.x * 8 + warp) * kFloorU;
    if (w0 >= W) return;  // the whole warp
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        const uint8_t *row = reinterpret_cast<const uint8_t *>(logits) + (size_t)b * stride * E::SIZE;
        const float f = __ldg(floor + b);
        bool on[kFloorU];
#pragma unroll
        for (int u = 0; u < kFloorU; ++u) {
            const int64_t i = (w0 + u) * 32 + lane;
            on[u] = i < V && E::load1(row, i) >= f;
        }
        uint32_t mine = 0;  // lane u keeps word w0 + u
#pragma unroll
        for (int u = 0; u < kFloorU; ++u) {
            const uint32_t wd = __ballot_sync(0xFFFFFFFFu, on[u]);
            if (lane == u) mine = wd;
        }
        if (lane < kFloorU && w0 + lane < W) {
            if (mask) mine &= (uint32_t)__ldg(mask + b * mstride + w0 + lane);
            out[b * W + w0 + lane] = (int32_t)mine;
        }
    }
}

// Rows that start 16-byte aligned: a lane reads AE consecutive tokens in one
// 16-byte load, and the 32 / AE lanes that share a word OR their bits into it
// (three shuffles for f32, two for 16-bit).  A warp step covers AE words; a
// warp takes kFloorVU consecutive steps of one row, all loads in flight.  A
// vector that runs past V reads its in-row tokens one by one.
constexpr int kFloorVU = 4;
template <int DT>
__global__ void __launch_bounds__(256) floor_mask_vec_kernel(const void *logits, int64_t B, int64_t V, int64_t stride,
                                                             const int32_t *mask, int64_t mstride,
                                                             const float *floor, int32_t *out, int64_t W) {
    using E = Elem<DT>;
    constexpr int AE = E::AE;
    constexpr int kLanesPerWord = 32 / AE;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nsteps = (V + 32 * AE - 1) / (32 * AE);
    const int64_t s0 = ((int64_t)blockIdx.x * 8 + warp) * kFloorVU;
    if (s0 >= nsteps) return;  // the whole warp
    for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
        const uint8_t *row = reinterpret_cast<const uint8_t *>(logits) + (size_t)b * stride * E::SIZE;
        const float f = __ldg(floor + b);
        uint4 v[kFloorVU];
#pragma unroll
        for (int u = 0; u < kFloorVU; ++u) {
            const int64_t e = ((s0 + u) * 32 + lane) * AE;  // first token of this lane's vector
            v[u] = e + AE <= V ? __ldg(reinterpret_cast<const uint4 *>(row + (size_t)e * E::SIZE))
                               : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kFloorVU; ++u) {
            const int64_t e = ((s0 + u) * 32 + lane) * AE;
            float x[AE];
            E::unpack(v[u], x);
            uint32_t bits = 0;
#pragma unroll
            for (int t = 0; t < AE; ++t) {
                const float xt = e + AE <= V ? x[t] : (e + t < V ? E::load1(row, e + t) : -INFINITY);
                bits |= xt >= f ? 1u << t : 0u;
            }
            bits <<= AE * (lane % kLanesPerWord);
#pragma unroll
            for (int o = 1; o < kLanesPerWord; o <<= 1) bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, o);
            const int64_t w = (s0 + u) * AE + lane / kLanesPerWord;
            if (lane % kLanesPerWord == 0 && w < W) {
                if (mask) bits &= (uint32_t)__ldg(mask + b * mstride + w);
                out[b * W + w] = (int32_t)bits;
            }
        }
    }
}

int floor_mask_launch(const void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                      int64_t mstride, const float *floor, int32_t *out, cudaStream_t st) {
    const int64_t W = (V + 31) / 32;
    const int es = dtype == 0 ? 4 : 2, ae = 16 / es;
    if ((reinterpret_cast<uintptr_t>(logits) % 16) == 0 && (stride * es) % 16 == 0) {
        // (steps of a row / (8 warps x kFloorVU), rows), rows strided past 65,535
        const int64_t nsteps = (V + 32 * ae - 1) / (32 * ae);
        const dim3 grid((unsigned)((nsteps + 8 * kFloorVU - 1) / (8 * kFloorVU)), (unsigned)(B < 65535 ? B : 65535));
        if (dtype == 0)
            floor_mask_vec_kernel<0><<<grid, 256, 0, st>>>(logits, B, V, stride, mask, mstride, floor, out, W);
        else if (dtype == 1)
            floor_mask_vec_kernel<1><<<grid, 256, 0, st>>>(logits, B, V, stride, mask, mstride, floor, out, W);
        else
            floor_mask_vec_kernel<2><<<grid, 256, 0, st>>>(logits, B, V, stride, mask, mstride, floor, out, W);
        return cudaGetLastError() == cudaSuccess ? 0 : -1;
    }
    // (words of a row / (8 warps x kFloorU), rows), rows strided past 65,535
    const dim3 grid((unsigned)((W + 8 * kFloorU - 1) / (8 * kFloorU)), (unsigned)(B < 65535 ? B : 65535));
    if (dtype == 0)
        floor_mask_kernel<0><<<grid, 256, 0, st>>>(logits, B, V, stride, mask, mstride, floor, out, W);
    else if (dtype == 1)
        floor_mask_kernel<1><<<grid, 256, 0, st>>>(logits, B, V, stride, mask, mstride, floor, out, W);
    else
        floor_mask_kernel<2><<<grid, 256, 0, st>>>(logits, B, V, stride, mask, mstride, floor, out, W);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tsa
