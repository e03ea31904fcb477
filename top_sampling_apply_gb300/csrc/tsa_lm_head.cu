// lm-head-topk, "API", "Method" and "Correctness" (the dense head): the
// vocabulary projection scores = hidden . weight^T (+ bias) fused with exact
// top-k, so the score vector is never written.
//
// Pass 1 (one CTA per 512-entry chunk of the vocabulary): the CTA's eight
// warps each take one weight row at a time, the 32 lanes striding it in
// 16-byte loads (four in flight a lane) against the hidden rows held in
// shared memory, fp32 accumulation; the chunk's scores become rank keys
// (value desc, index asc), are sorted in shared memory, and the chunk writes
// its best min(k, 512) in that order.  The global top k may all lie in one
// chunk, which is why each chunk offers k candidates (or all it has).
// Pass 2: the exact top-k over the candidates (the library's top-k kernel);
// candidates are laid out chunk by chunk, so a lower position is a lower
// vocabulary index among equal scores, and that kernel's position ties give
// the page's index ties.  Pass 3 maps positions back to vocabulary indices.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_device.cuh"
#include "tsa_host.h"
#include "tsa_sample_common.cuh"

namespace tsa {

namespace {

using sample_detail::block_sort_desc;

constexpr int kLhThreads = 256;
static_assert(kLhThreads == sample_detail::kThreads, "the chunk sort runs on kThreads threads");
constexpr int kLhWarps = kLhThreads / 32;
constexpr int kLhChunk = 512;

struct BlockBarrier {
    __device__ static void sync() { __syncthreads(); }
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
}

template <int M>
__global__ void __launch_bounds__(kLhThreads) lm_head_chunk_kernel(LmHeadArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t *keys = reinterpret_cast<uint64_t *>(smem);                          // [M][kLhChunk]
    uint4 *hs = reinterpret_cast<uint4 *>(smem + (size_t)M * kLhChunk * 8);       // [M][H / 8]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t H8 = a.H / 8;
    for (int64_t i = tid; i < M * H8; i += kLhThreads) {
        const int64_t m = i / H8, j = i - m * H8;
        hs[i] = __ldg(reinterpret_cast<const uint4 *>(a.hidden + m * a.hstride) + j);
    }
    const int64_t c = blockIdx.x;
    const int64_t r0 = c * kLhChunk;
    const int n = (int)((a.V - r0) < kLhChunk ? (a.V - r0) : kLhChunk);
    __syncthreads();
    for (int r = warp; r < n; r += kLhWarps) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(a.weight + (r0 + r) * a.wstride);
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.f;
        int64_t j = lane;
        for (; j + 96 < H8; j += 128) {  // four 16-byte loads in flight a lane
            uint4 wv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) wv[u] = __ldcs(wrow + j + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float wf[8];
                bf16x8_to_f32(wv[u], wf);
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    float hf[8];
                    bf16x8_to_f32(hs[m * H8 + j + 32 * u], hf);
#pragma unroll
                    for (int t = 0; t < 8; ++t) acc[m] = fmaf(wf[t], hf[t], acc[m]);
                }
            }
        }
        for (; j < H8; j += 32) {
            float wf[8];
            bf16x8_to_f32(__ldcs(wrow + j), wf);
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float hf[8];
                bf16x8_to_f32(hs[m * H8 + j], hf);
#pragma unroll
                for (int t = 0; t < 8; ++t) acc[m] = fmaf(wf[t], hf[t], acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float s = acc[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
            if (a.bias) s += __ldg(a.bias + r0 + r);
            if (lane == 0) keys[m * kLhChunk + r] = rank_key(s, (uint32_t)(r0 + r));
        }
    }
    __syncthreads();
    // per hidden row: sort the chunk's keys and write its best kk
    for (int m = 0; m < M; ++m) {
        block_sort_desc<BlockBarrier>(keys + m * kLhChunk, (uint32_t)n);
        const int64_t base = (int64_t)m * a.cand_stride + c * a.kk;
        for (int j2 = tid; j2 < a.kk; j2 += kLhThreads) {
            if (j2 < n) {
                const uint64_t key = keys[m * kLhChunk + j2];
                a.cand_vals[base + j2] = rank_key_value(key);
                a.cand_idx[base + j2] = (int32_t)rank_key_index(key);
            } else {  // a short last chunk: filler below every score
                a.cand_vals[base + j2] = -INFINITY;
                a.cand_idx[base + j2] = -1;
            }
        }
    }
}

// Candidate positions to vocabulary indices.
__global__ void lm_head_gather_kernel(const int64_t *pos, const int32_t *cand_idx, int64_t cand_stride, int64_t M,
                                      int32_t k, int64_t *indices_out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= M * k) return;
    const int64_t m = i / k;
    indices_out[i] = cand_idx[m * cand_stride + pos[i]];
}

}  // namespace

size_t lm_head_smem_bytes(int64_t M, int64_t H) { return (size_t)M * kLhChunk * 8 + (size_t)M * H * 2; }

int64_t lm_head_chunks(int64_t V) { return (V + kLhChunk - 1) / kLhChunk; }

int32_t lm_head_kk(int32_t k) { return k < kLhChunk ? k : kLhChunk; }

int lm_head_pass1_launch(const LmHeadArgs &args, cudaStream_t st) {
    const void *fns[4] = {(const void *)lm_head_chunk_kernel<1>, (const void *)lm_head_chunk_kernel<2>,
                          (const void *)lm_head_chunk_kernel<3>, (const void *)lm_head_chunk_kernel<4>};
    const void *fn = fns[args.M - 1];
    const size_t smem = lm_head_smem_bytes(args.M, args.H);
    if (prepare_kernel(fn, smem, 1) != 0) return -1;
    LmHeadArgs a = args;
    void *params[] = {&a};
    return cudaLaunchKernel(fn, dim3((unsigned)args.nchunks), dim3(kLhThreads), params, smem, st) == cudaSuccess
               ? 0
               : -1;
}

int lm_head_gather_launch(const int64_t *pos, const int32_t *cand_idx, int64_t cand_stride, int64_t M, int32_t k,
                          int64_t *indices_out, cudaStream_t st) {
    const int64_t n = M * k;
    lm_head_gather_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(pos, cand_idx, cand_stride, M, k,
                                                                       indices_out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tsa
