// C-ABI entry points: argument validation, row split, launch, status.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/tsa.h"
#include "tsa_device.cuh"
#include "tsa_host.h"

namespace tsa {

namespace {
constexpr size_t kSliceMax = 200 * 1024;    // largest slice a CTA may hold
constexpr size_t kPipeSlice = 33280;        // double-buffered slice for 3 CTAs per SM
constexpr int kMaxSlices = 64;
constexpr int kMaxTopk = 2048;

struct Prepared {
    const void *fn;
    int device;
    size_t smem;
    int cluster16;
};
std::mutex g_mu;
Prepared g_prepared[64];
int g_nprepared = 0;

int esize_of(int dtype) { return dtype == TSA_F32 ? 4 : 2; }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

bool choose_split(int64_t V, int esize, size_t slice_target, size_t slice_max, int *cluster,
                  int64_t *max_vec) {
    const int64_t AE = 16 / esize;
    const int64_t nvec_max = V / AE + 1;
    for (int C = 1; C <= 16; C *= 2) {
        const int64_t mv = (nvec_max + C - 1) / C;
        if ((size_t)(mv + 2) * 16 <= slice_target) {
            *cluster = C;
            *max_vec = mv;
            return true;
        }
    }
    const int64_t mv = (nvec_max + 15) / 16;
    if ((size_t)(mv + 2) * 16 <= slice_max) {
        *cluster = 16;
        *max_vec = mv;
        return true;
    }
    return false;
}

bool choose_sample_split(int64_t V, int esize, int *slices, int64_t *max_vec, int *nbuf) {
    // Slices of <= kPipeSlice bytes, double-buffered, keep three CTAs per SM
    // with the next item's copy in flight; rows of more than kMaxSlices such
    // slices use kMaxSlices larger slices (double-buffered while they fit).
    const int64_t AE = 16 / esize;
    const int64_t nvec_max = V / AE + 1;
    const int64_t per = (int64_t)(kPipeSlice / 16) - 2;
    int64_t S = (nvec_max + per - 1) / per;
    if (S <= kMaxSlices) {
        *slices = (int)S;
        *max_vec = (nvec_max + S - 1) / S;
        *nbuf = 2;
        return true;
    }
    S = kMaxSlices;
    const int64_t mv = (nvec_max + S - 1) / S;
    *slices = (int)S;
    *max_vec = mv;
    *nbuf = (size_t)(mv + 2) * 16 * 2 <= kSliceMax ? 2 : 1;
    return (size_t)(mv + 2) * 16 <= kSliceMax;
}

int prepare_kernel(const void *fn, size_t smem, int cluster) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    std::lock_guard<std::mutex> lock(g_mu);
    Prepared *p = nullptr;
    for (int i = 0; i < g_nprepared; ++i)
        if (g_prepared[i].fn == fn && g_prepared[i].device == dev) p = &g_prepared[i];
    if (!p) {
        if (g_nprepared == 64) return -1;
        p = &g_prepared[g_nprepared++];
        p->fn = fn;
        p->device = dev;
        p->smem = 0;
        p->cluster16 = 0;
    }
    if (smem > p->smem) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        p->smem = smem;
    }
    if (cluster > 8 && !p->cluster16) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            return -1;
        p->cluster16 = 1;
    }
    return 0;
}

// A block that waits on an mbarrier nothing will complete, with a bounded wait.
__device__ unsigned int g_selftest_status;
__global__ void selftest_wait_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    mbar_wait_bounded(&bar, 0, &g_selftest_status, limit_ns);
}

int selftest_launch(uint32_t limit_us, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>((unsigned long long)limit_us * 1000ull);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tsa

using namespace tsa;

extern "C" {

int64_t tsa_max_vocab(tsa_dtype dtype) {
    const int es = (dtype == TSA_F32) ? 4 : 2;
    const int64_t AE = 16 / es;
    // 16 CTAs, each with at most kSliceMax bytes of vector slots (2 spare)
    return (int64_t)16 * ((int64_t)(kSliceMax / 16) - 2) * AE - AE;
}

const char *tsa_status_string(int status) {
    switch (status) {
    case TSA_OK: return "ok";
    case TSA_ERR_NULL: return "a required pointer is NULL";
    case TSA_ERR_SHAPE: return "invalid shape (B < 0, V < 1, V above the maximum, or row stride < V)";
    case TSA_ERR_DTYPE: return "unsupported dtype";
    case TSA_ERR_K_RANGE: return "k out of range (1 <= k <= min(2048, V))";
    case TSA_ERR_STRIDE: return "mask row stride < ceil(V / 32)";
    case TSA_ERR_WORKSPACE: return "workspace too small";
    case TSA_ERR_CUDA: return "CUDA runtime error";
    case TSA_ERR_DEVICE_TIMEOUT: return "a device-side bounded wait ran out";
    case TSA_ERR_ALIGN: return "pointer not aligned to its element size";
    default: return "unknown status";
    }
}

static int check_rows(const void *logits, int dtype, int64_t B, int64_t V, int64_t stride) {
    if (dtype != TSA_F32 && dtype != TSA_F16 && dtype != TSA_BF16) return TSA_ERR_DTYPE;
    if (B < 0 || V < 1 || stride < V) return TSA_ERR_SHAPE;
    if (V > tsa_max_vocab((tsa_dtype)dtype) || B > 0x7FFFFFFFll / 16) return TSA_ERR_SHAPE;
    if (!logits && B > 0) return TSA_ERR_NULL;
    if (!aligned(logits, esize_of(dtype))) return TSA_ERR_ALIGN;
    return TSA_OK;
}

}  // extern "C"

namespace tsa {
int sample_check_args(const void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                      int64_t mstride, const float *temperature, const int32_t *top_k, const float *top_p,
                      const float *min_p, const int64_t *tokens, const float *vstar) {
    int st = check_rows(logits, dtype, B, V, stride);
    if (st != TSA_OK) return st;
    if (!tokens && B > 0) return TSA_ERR_NULL;
    if (mask && mstride < (V + 31) / 32) return TSA_ERR_STRIDE;
    if (!aligned(mask, 4) || !aligned(tokens, 8) || !aligned(vstar, 4) || !aligned(temperature, 4) ||
        !aligned(top_k, 4) || !aligned(top_p, 4) || !aligned(min_p, 4))
        return TSA_ERR_ALIGN;
    return TSA_OK;
}
}  // namespace tsa

extern "C" {

int tsa_apply_token_bitmask(void *logits, tsa_dtype dtype, int64_t B, int64_t V, int64_t logits_row_stride,
                            const int32_t *bitmask, int64_t mask_row_stride, void *stream) {
    int st = check_rows(logits, dtype, B, V, logits_row_stride);
    if (st != TSA_OK) return st;
    if (!bitmask && B > 0) return TSA_ERR_NULL;
    if (mask_row_stride < (V + 31) / 32) return TSA_ERR_STRIDE;
    if (!aligned(bitmask, 4)) return TSA_ERR_ALIGN;
    if (B == 0) return TSA_OK;
    return mask_launch(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride,
                       (cudaStream_t)stream) == 0 ? TSA_OK : TSA_ERR_CUDA;
}

int tsa_selective_log_softmax(const void *logits, tsa_dtype dtype, int64_t B, int64_t V,
                              int64_t logits_row_stride, const int32_t *bitmask, int64_t mask_row_stride,
                              const float *temperature, float temperature_s, const int64_t *index, float *out,
                              void *stream) {
    int st = check_rows(logits, dtype, B, V, logits_row_stride);
    if (st != TSA_OK) return st;
    if ((!index || !out) && B > 0) return TSA_ERR_NULL;
    if (bitmask && mask_row_stride < (V + 31) / 32) return TSA_ERR_STRIDE;
    if (!aligned(bitmask, 4) || !aligned(temperature, 4) || !aligned(index, 8) || !aligned(out, 4))
        return TSA_ERR_ALIGN;
    if (B == 0) return TSA_OK;
    return logprob_launch(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride, temperature,
                          temperature_s, index, out, (cudaStream_t)stream) == 0
               ? TSA_OK
               : TSA_ERR_CUDA;
}

size_t tsa_sample_workspace_bytes(int64_t B, int64_t V, tsa_dtype dtype) {
    // one CTA per row (B >= kRowKernelMinB) keeps every step on chip
    if (B < 1 || B >= kRowKernelMinB || V < 1) return 0;
    int S = 1, nbuf = 1;
    int64_t mv = 0;
    if (!choose_sample_split(V, esize_of(dtype), &S, &mv, &nbuf)) return 0;
    size_t so = 0, co = 0;
    return sample_workspace_layout(B, S, &so, &co);
}
size_t tsa_topk_workspace_bytes(int64_t, int64_t, int32_t, tsa_dtype) { return 0; }

int tsa_sample(const void *logits, tsa_dtype dtype, int64_t B, int64_t V, int64_t logits_row_stride,
               const int32_t *bitmask, int64_t mask_row_stride, const float *temperature,
               float temperature_s, const int32_t *top_k, int32_t top_k_s, const float *top_p,
               float top_p_s, const float *min_p, float min_p_s, uint64_t seed, uint64_t offset,
               int64_t *tokens_out, float *min_kept_logit_out, void *workspace,
               size_t workspace_bytes, void *stream) {
    int st = sample_check_args(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride, temperature,
                               top_k, top_p, min_p, tokens_out, min_kept_logit_out);
    if (st != TSA_OK) return st;
    if (B == 0) return TSA_OK;
    int slices = 1, nbuf = 1;
    int64_t max_vec = 0;
    if (!choose_sample_split(V, esize_of(dtype), &slices, &max_vec, &nbuf)) return TSA_ERR_SHAPE;
    const size_t need = tsa_sample_workspace_bytes(B, V, dtype);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return TSA_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return TSA_ERR_ALIGN;
    }
    SampleArgs a = {};
    a.workspace = workspace;
    a.logits = logits;
    a.B = B;
    a.V = V;
    a.stride = logits_row_stride;
    a.mask = bitmask;
    a.mstride = mask_row_stride;
    a.temperature = temperature;
    a.temperature_s = temperature_s;
    a.top_k = top_k;
    a.top_k_s = top_k_s;
    a.top_p = top_p;
    a.top_p_s = top_p_s;
    a.min_p = min_p;
    a.min_p_s = min_p_s;
    a.seed = seed;
    a.offset = offset;
    a.tokens = tokens_out;
    a.vstar_out = min_kept_logit_out;
    return sample_launch(a, dtype, slices, max_vec, nbuf, (cudaStream_t)stream) == 0 ? TSA_OK : TSA_ERR_CUDA;
}

static size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

size_t tsa_sample_sequential_workspace_bytes(int64_t B, int64_t V, tsa_dtype dtype) {
    if (B < 1 || V < 1) return 0;
    const size_t words = (size_t)B * (size_t)((V + 31) / 32);
    return align256(words * 4) + align256((size_t)B * 4) + tsa_sample_workspace_bytes(B, V, dtype);
}

int tsa_sample_sequential(const void *logits, tsa_dtype dtype, int64_t B, int64_t V, int64_t logits_row_stride,
                          const int32_t *bitmask, int64_t mask_row_stride, const float *temperature,
                          float temperature_s, const int32_t *top_k, int32_t top_k_s, const float *top_p,
                          float top_p_s, const float *min_p, float min_p_s, uint64_t seed, uint64_t offset,
                          int64_t *tokens_out, float *min_kept_logit_out, void *workspace,
                          size_t workspace_bytes, void *stream) {
    int st = sample_check_args(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride, temperature,
                               top_k, top_p, min_p, tokens_out, min_kept_logit_out);
    if (st != TSA_OK) return st;
    if (B == 0) return TSA_OK;
    const size_t need = tsa_sample_sequential_workspace_bytes(B, V, dtype);
    if (!workspace || workspace_bytes < need) return TSA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return TSA_ERR_ALIGN;
    const int64_t W = (V + 31) / 32;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *survivors = reinterpret_cast<int32_t *>(ws);
    float *v_k = reinterpret_cast<float *>(ws + align256((size_t)B * (size_t)W * 4));
    uint8_t *ws_sample = ws + align256((size_t)B * (size_t)W * 4) + align256((size_t)B * 4);
    const size_t ws_sample_bytes = workspace_bytes - (size_t)(ws_sample - ws);
    void *ws_s = tsa_sample_workspace_bytes(B, V, dtype) > 0 ? ws_sample : nullptr;
    // 1. the top-k cut alone (v* with top-p and min-p off; the argmax value
    //    for greedy rows, -inf without top-k, NaN for an empty row)
    st = tsa_sample(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride, temperature, temperature_s,
                    top_k, top_k_s, nullptr, 1.0f, nullptr, 0.0f, seed, offset, tokens_out, v_k, ws_s,
                    ws_sample_bytes, stream);
    if (st != TSA_OK) return st;
    // 2. its survivors as a bitmask
    if (floor_mask_launch(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride, v_k, survivors,
                          (cudaStream_t)stream) != 0)
        return TSA_ERR_CUDA;
    // 3. top-p (renormalised over the survivors) and min-p; top-k again keeps
    //    every survivor and still sends top_k == 1 rows to the argmax
    return tsa_sample(logits, dtype, B, V, logits_row_stride, survivors, W, temperature, temperature_s, top_k,
                      top_k_s, top_p, top_p_s, min_p, min_p_s, seed, offset, tokens_out, min_kept_logit_out,
                      ws_s, ws_sample_bytes, stream);
}

size_t tsa_lm_head_topk_workspace_bytes(int64_t M, int64_t V, int32_t k) {
    if (M < 1 || M > 4 || V < 1 || k < 1) return 0;
    const size_t per_row = (size_t)lm_head_chunks(V) * (size_t)lm_head_kk(k);
    return 2 * align256((size_t)M * per_row * 4) + align256((size_t)M * (size_t)k * 8);
}

int tsa_lm_head_topk(const void *hidden, int64_t M, int64_t H, int64_t hidden_row_stride, const void *weight,
                     int64_t V, int64_t weight_row_stride, const float *bias, int32_t k, float *values_out,
                     int64_t *indices_out, void *workspace, size_t workspace_bytes, void *stream) {
    if (M < 0 || M > 4 || H < 8 || H > 8192 || H % 8 != 0 || V < 1 || hidden_row_stride < H ||
        weight_row_stride < H)
        return TSA_ERR_SHAPE;
    if (k < 1 || k > kMaxTopk || (int64_t)k > V) return TSA_ERR_K_RANGE;
    if (M == 0) return TSA_OK;
    if (!hidden || !weight || !values_out || !indices_out) return TSA_ERR_NULL;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || hidden_row_stride % 8 != 0 || weight_row_stride % 8 != 0 ||
        !aligned(bias, 4) || !aligned(values_out, 4) || !aligned(indices_out, 8))
        return TSA_ERR_ALIGN;
    const int64_t C = lm_head_chunks(V);
    const int32_t kk = lm_head_kk(k);
    const int64_t per_row = C * kk;
    if (per_row > tsa_max_vocab(TSA_F32)) return TSA_ERR_SHAPE;
    const size_t need = tsa_lm_head_topk_workspace_bytes(M, V, k);
    if (!workspace || workspace_bytes < need) return TSA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return TSA_ERR_ALIGN;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    LmHeadArgs la = {};
    la.hidden = static_cast<const uint16_t *>(hidden);
    la.M = M;
    la.H = H;
    la.hstride = hidden_row_stride;
    la.weight = static_cast<const uint16_t *>(weight);
    la.V = V;
    la.wstride = weight_row_stride;
    la.bias = bias;
    la.k = k;
    la.kk = kk;
    la.nchunks = C;
    la.cand_stride = per_row;
    la.cand_vals = reinterpret_cast<float *>(ws);
    la.cand_idx = reinterpret_cast<int32_t *>(ws + align256((size_t)M * per_row * 4));
    int64_t *pos = reinterpret_cast<int64_t *>(ws + 2 * align256((size_t)M * per_row * 4));
    cudaStream_t st = (cudaStream_t)stream;
    if (lm_head_pass1_launch(la, st) != 0) return TSA_ERR_CUDA;
    const int r = tsa_topk(la.cand_vals, TSA_F32, M, per_row, per_row, k, values_out, pos, nullptr, 0, stream);
    if (r != TSA_OK) return r;
    return lm_head_gather_launch(pos, la.cand_idx, per_row, M, k, indices_out, st) == 0 ? TSA_OK : TSA_ERR_CUDA;
}

int tsa_sample_icdf(const void *logits, tsa_dtype dtype, int64_t B, int64_t V, int64_t logits_row_stride,
                    const int32_t *bitmask, int64_t mask_row_stride, const float *temperature,
                    float temperature_s, const int32_t *top_k, int32_t top_k_s, const float *top_p,
                    float top_p_s, const float *min_p, float min_p_s, const float *uniform,
                    int64_t *tokens_out, float *min_kept_logit_out, void *workspace, size_t workspace_bytes,
                    void *stream) {
    int st = sample_check_args(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride, temperature,
                               top_k, top_p, min_p, tokens_out, min_kept_logit_out);
    if (st != TSA_OK) return st;
    if ((!uniform || !min_kept_logit_out) && B > 0) return TSA_ERR_NULL;
    if (!aligned(uniform, 4)) return TSA_ERR_ALIGN;
    if (B == 0) return TSA_OK;
    // the keep-threshold v* (and the argmax of greedy rows) from the sample
    // path; its Gumbel draw is then replaced row by row
    st = tsa_sample(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride, temperature, temperature_s,
                    top_k, top_k_s, top_p, top_p_s, min_p, min_p_s, 0, 0, tokens_out, min_kept_logit_out, workspace,
                    workspace_bytes, stream);
    if (st != TSA_OK) return st;
    IcdfArgs ia = {};
    ia.logits = logits;
    ia.B = B;
    ia.V = V;
    ia.stride = logits_row_stride;
    ia.mask = bitmask;
    ia.mstride = mask_row_stride;
    ia.temperature = temperature;
    ia.temperature_s = temperature_s;
    ia.top_k = top_k;
    ia.top_k_s = top_k_s;
    ia.uniform = uniform;
    ia.vstar = min_kept_logit_out;
    ia.tokens = tokens_out;
    return icdf_launch(ia, dtype, (cudaStream_t)stream) == 0 ? TSA_OK : TSA_ERR_CUDA;
}

int tsa_bitmask_from_allowed(const uint8_t *allowed, int64_t B, int64_t V, int64_t allowed_row_stride,
                             int32_t *bitmask_out, int64_t mask_row_stride, void *stream) {
    if (B < 0 || V < 1 || allowed_row_stride < V || B > 0x7FFFFFFFll) return TSA_ERR_SHAPE;
    if ((!allowed || !bitmask_out) && B > 0) return TSA_ERR_NULL;
    if (mask_row_stride < (V + 31) / 32) return TSA_ERR_STRIDE;
    if (!aligned(bitmask_out, 4)) return TSA_ERR_ALIGN;
    if (B == 0) return TSA_OK;
    return pack_launch(allowed, B, V, allowed_row_stride, bitmask_out, mask_row_stride, (cudaStream_t)stream) == 0
               ? TSA_OK
               : TSA_ERR_CUDA;
}

int tsa_topk(const void *logits, tsa_dtype dtype, int64_t B, int64_t V, int64_t logits_row_stride, int32_t k,
             float *values_out, int64_t *indices_out, void *workspace, size_t workspace_bytes,
             void *stream) {
    (void)workspace;
    (void)workspace_bytes;
    int st = check_rows(logits, dtype, B, V, logits_row_stride);
    if (st != TSA_OK) return st;
    if (k < 1 || k > kMaxTopk || (int64_t)k > V) return TSA_ERR_K_RANGE;
    if ((!values_out || !indices_out) && B > 0) return TSA_ERR_NULL;
    if (!aligned(values_out, 4) || !aligned(indices_out, 8)) return TSA_ERR_ALIGN;
    if (B == 0) return TSA_OK;
    int cluster = 1;
    int64_t max_vec = 0;
    if (!choose_split(V, esize_of(dtype), 64 * 1024, kSliceMax, &cluster, &max_vec)) return TSA_ERR_SHAPE;
    TopkArgs a = {};
    a.logits = logits;
    a.B = B;
    a.V = V;
    a.stride = logits_row_stride;
    a.k = k;
    a.values = values_out;
    a.indices = indices_out;
    return topk_launch(a, dtype, cluster, max_vec, (cudaStream_t)stream) == 0 ? TSA_OK : TSA_ERR_CUDA;
}

int tsa_device_status(int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return TSA_ERR_CUDA;
    unsigned int *ptrs[7] = {sample_status_ptr(),         sample_row_status_ptr(),
                             topk_status_ptr(),           nullptr,
                             sample_row_spec_status_ptr_f32(), sample_row_spec_status_ptr_f16(),
                             sample_row_spec_status_ptr_bf16()};
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_selftest_status) == cudaSuccess) ptrs[3] = (unsigned int *)p;
    unsigned int any = 0;
    for (int i = 0; i < 7; ++i) {
        if (!ptrs[i]) return TSA_ERR_CUDA;
        unsigned int v = 0;
        if (cudaMemcpy(&v, ptrs[i], sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return TSA_ERR_CUDA;
        any |= v;
        if (clear && v) {
            const unsigned int zero = 0;
            if (cudaMemcpy(ptrs[i], &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
                return TSA_ERR_CUDA;
        }
    }
    return (any & kStatusTimeout) ? TSA_ERR_DEVICE_TIMEOUT : TSA_OK;
}

int tsa_selftest_wait_timeout(uint32_t limit_us, void *stream) {
    if (limit_us == 0 || limit_us > 2000000u) return TSA_ERR_SHAPE;
    return selftest_launch(limit_us, (cudaStream_t)stream) == 0 ? TSA_OK : TSA_ERR_CUDA;
}

}  // extern "C"
