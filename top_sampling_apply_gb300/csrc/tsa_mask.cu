// apply_token_bitmask (logits-processor, "API" and "Correctness"): disallowed
// logits become -inf in place; allowed logits are never written.
//
// Logits are never read: a word of all ones costs one 4-byte mask read and no
// write; a word with zero bits writes -inf to exactly those tokens.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_host.h"

namespace tsa {

template <int DT>
__global__ void __launch_bounds__(256) mask_kernel(void *logits, int64_t V, int64_t stride,
                                                   const int32_t *mask, int64_t mstride,
                                                   int64_t W, int64_t total_words) {
    // One warp per 32-bit mask word; lane t owns token 32 w + t, so the -inf
    // stores of a warp are coalesced into one 128-byte (or 64-byte) segment.
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t g = warp0; g < total_words; g += nwarps) {
        const int64_t b = g / W, w = g - b * W;
        const uint32_t word = (uint32_t)__ldg(mask + b * mstride + w);
        const int64_t i = w * 32 + lane;
        if (i >= V || ((word >> lane) & 1u)) continue;  // bits at or beyond V are ignored
        if (DT == 0)
            reinterpret_cast<uint32_t *>(logits)[b * stride + i] = 0xFF800000u;
        else
            reinterpret_cast<unsigned short *>(logits)[b * stride + i] =
                (unsigned short)(DT == 1 ? 0xFC00u : 0xFF80u);
    }
}

int mask_launch(void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                int64_t mstride, cudaStream_t st) {
    const int64_t W = (V + 31) / 32;
    const int64_t total = B * W;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (total + 7) / 8;  // 8 warps (words) per block
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (dtype == 0)
        mask_kernel<0><<<(unsigned)blocks, 256, 0, st>>>(logits, V, stride, mask, mstride, W, total);
    else if (dtype == 1)
        mask_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(logits, V, stride, mask, mstride, W, total);
    else
        mask_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(logits, V, stride, mask, mstride, W, total);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tsa
