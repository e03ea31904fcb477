// Internal host-side interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tsa {

// Batches of at least this many rows run one CTA per row and need no
// workspace; smaller ones split rows into slices across the whole GPU.
constexpr int64_t kRowKernelMinB = 128;

struct SampleArgs {
    const void *logits;
    int64_t B, V, stride;
    const int32_t *mask;
    int64_t mstride;
    const float *temperature;
    float temperature_s;
    const int32_t *top_k;
    int32_t top_k_s;
    const float *top_p;
    float top_p_s;
    const float *min_p;
    float min_p_s;
    uint64_t seed, offset;
    int64_t *tokens;
    float *vstar_out;
    void *workspace;    // row counters (zero between calls), slice summaries, candidates
    int64_t max_vec;    // vector slots per slice buffer (set by the launcher)
    int64_t max_words;  // mask words per slice buffer (set by the launcher)
    int slices;         // slices per row
    size_t summ_off, cand_off;  // workspace offsets (set by the launcher)
};

struct TopkArgs {
    const void *logits;
    int64_t B, V, stride;
    int32_t k;
    float *values;
    int64_t *indices;
    int64_t max_vec;
};

// Row split: cluster size and vector slots per CTA for a row of V elements of
// `esize` bytes, keeping each CTA's slice within `slice_target` bytes where
// possible and never above `slice_max`.  Returns false if V does not fit.
bool choose_split(int64_t V, int esize, size_t slice_target, size_t slice_max, int *cluster,
                  int64_t *max_vec);

// Sets the kernel's dynamic shared-memory limit (and non-portable cluster
// sizes) once per device; returns 0 or -1.
int prepare_kernel(const void *fn, size_t smem, int cluster);

// The argument checks of tsa_sample (everything but the workspace); returns
// TSA_OK or the status tsa_sample would return.
int sample_check_args(const void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                      int64_t mstride, const float *temperature, const int32_t *top_k, const float *top_p,
                      const float *min_p, const int64_t *tokens, const float *vstar);

// Sample split: slices per row, vector slots per slice and slice buffers (1 or 2).
bool choose_sample_split(int64_t V, int esize, int *slices, int64_t *max_vec, int *nbuf);
size_t sample_workspace_layout(int64_t B, int S, size_t *summ_off, size_t *cand_off);
size_t sample_smem_bytes(int64_t max_vec, int64_t max_words, int nbuf);
int sample_launch(const SampleArgs &args, int dtype, int slices, int64_t max_vec, int nbuf, cudaStream_t st);
unsigned int *sample_status_ptr();
// One CTA per row (large batches); its own device status word.
int sample_row_launch(const SampleArgs &args, int dtype, cudaStream_t st);
unsigned int *sample_row_status_ptr();
// Specialised row kernels (nullptr for a specialisation not built) and their
// status words, one translation unit per element type.
const void *sample_row_spec_kernel_f32(int spec);
const void *sample_row_spec_kernel_f16(int spec);
const void *sample_row_spec_kernel_bf16(int spec);
unsigned int *sample_row_spec_status_ptr_f32();
unsigned int *sample_row_spec_status_ptr_f16();
unsigned int *sample_row_spec_status_ptr_bf16();
inline const void *sample_row_spec_kernel(int dtype, int spec) {
    return dtype == 0 ? sample_row_spec_kernel_f32(spec)
                      : (dtype == 1 ? sample_row_spec_kernel_f16(spec) : sample_row_spec_kernel_bf16(spec));
}

size_t topk_smem_bytes(int64_t max_vec);
int topk_launch(const TopkArgs &args, int dtype, int cluster, int64_t max_vec, cudaStream_t st);
unsigned int *topk_status_ptr();

// The dense lm-head projection fused with top-k: pass 1 (per 512-entry chunk
// of the vocabulary, its best min(k, 512) as candidates).
struct LmHeadArgs {
    const uint16_t *hidden;  // bf16 [M, hstride]
    int64_t M, H, hstride;
    const uint16_t *weight;  // bf16 [V, wstride]
    int64_t V, wstride;
    const float *bias;       // [V] or NULL
    int32_t k, kk;           // kk = min(k, chunk)
    int64_t nchunks, cand_stride;  // candidates per row = nchunks * kk
    float *cand_vals;
    int32_t *cand_idx;
};
size_t lm_head_smem_bytes(int64_t M, int64_t H);
int64_t lm_head_chunks(int64_t V);
int32_t lm_head_kk(int32_t k);
int lm_head_pass1_launch(const LmHeadArgs &args, cudaStream_t st);
int lm_head_gather_launch(const int64_t *pos, const int32_t *cand_idx, int64_t cand_stride, int64_t M, int32_t k,
                          int64_t *indices_out, cudaStream_t st);

// The inverse-CDF draw over the keep set of a sample call that ran before it
// (its v* per row), and the allow-set packer.
struct IcdfArgs {
    const void *logits;
    int64_t B, V, stride;
    const int32_t *mask;
    int64_t mstride;
    const float *temperature;
    float temperature_s;
    const int32_t *top_k;
    int32_t top_k_s;
    const float *uniform;
    const float *vstar;
    int64_t *tokens;
};
int icdf_launch(const IcdfArgs &args, int dtype, cudaStream_t st);
int pack_launch(const uint8_t *allowed, int64_t B, int64_t V, int64_t astride, int32_t *bits, int64_t wstride,
                cudaStream_t st);

int mask_launch(void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                int64_t mstride, cudaStream_t st);
// Bitmask (row stride ceil(V / 32)) of the tokens allowed by `mask` whose
// logit is >= floor[b].
int floor_mask_launch(const void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                      int64_t mstride, const float *floor, int32_t *out, cudaStream_t st);
int logprob_launch(const void *logits, int dtype, int64_t B, int64_t V, int64_t stride, const int32_t *mask,
                   int64_t mstride, const float *temperature, float temperature_s, const int64_t *index,
                   float *out, cudaStream_t st);
int selftest_launch(uint32_t limit_us, cudaStream_t st);

}  // namespace tsa
