/*
 * tsa.h -- per-row vocabulary selection on NVIDIA GB300 (sm_103a).
 *
 * The step between a model's logits and its next token: a packed grammar
 * mask, a fused temperature + top-k / top-p / min-p filter with a Gumbel-max
 * draw, and an exact sorted top-k.  Plain C ABI: device pointers, sizes and a
 * CUDA stream passed as void*; no framework types.
 *
 * Conventions shared by every call
 *   - Pointers named logits / bitmask / workspace / *_out and per-row
 *     parameter arrays are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory and keeps no state between calls.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.
 *   - Rows are row-major: element (b, i) of logits is at
 *     logits + (b * logits_row_stride + i) * element_size.  Row starts need
 *     only element alignment; 16-byte aligned rows take the fastest path.
 *   - Arguments are validated before anything is enqueued.  A negative
 *     return value means nothing was launched (TSA_ERR_CUDA: the launch itself
 *     failed).  B == 0 is a valid no-op.
 *   - The bitmask layout is [B, mask_row_stride] int32 with
 *     mask_row_stride >= ceil(V / 32); token i is allowed iff bit (i & 31) of
 *     word (i >> 5) is 1 (least significant bit first).  Bits at or beyond V
 *     are ignored.
 *   - Device-side faults of the library's own making (a bounded wait that ran
 *     out) never hang the GPU: the kernel records a flag, finishes, and
 *     tsa_device_status() reports it.
 */
#ifndef TSA_H
#define TSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { TSA_F32 = 0, TSA_F16 = 1, TSA_BF16 = 2 } tsa_dtype;

enum {
    TSA_OK = 0,
    TSA_ERR_NULL = -1,           /* a required pointer is NULL */
    TSA_ERR_SHAPE = -2,          /* B < 0, V < 1, V too large, or row stride < V */
    TSA_ERR_DTYPE = -3,          /* dtype not one of tsa_dtype */
    TSA_ERR_K_RANGE = -4,        /* topk: k < 1, k > 2048 or k > V */
    TSA_ERR_STRIDE = -5,         /* mask_row_stride < ceil(V / 32) */
    TSA_ERR_WORKSPACE = -6,      /* sample: workspace NULL or smaller than required */
    TSA_ERR_CUDA = -7,           /* a CUDA runtime call failed (launch / attribute) */
    TSA_ERR_DEVICE_TIMEOUT = -8, /* a kernel's bounded wait ran out (see tsa_device_status) */
    TSA_ERR_ALIGN = -9           /* a pointer is not aligned to its element size */
};

/* Largest vocabulary a row may have, per element type (elements). */
int64_t tsa_max_vocab(tsa_dtype dtype);

/*
 * apply_token_bitmask -- logits-processor, "API" (apply_token_bitmask) and
 * "Correctness": set to -inf, in place, exactly the logits whose mask bit is
 * 0; allowed logits are left bit-identical; V need not be a multiple of 32.
 *   logits   [B, logits_row_stride] of dtype, read and written in place
 *   bitmask  [B, mask_row_stride] int32, read only
 * Returns TSA_OK or a negative status.
 */
int tsa_apply_token_bitmask(void *logits, tsa_dtype dtype, int64_t B, int64_t V,
                            int64_t logits_row_stride, const int32_t *bitmask,
                            int64_t mask_row_stride, void *stream);

/*
 * sample -- logits-processor, "API" (sample) and "Method": one token per row.
 * Temperature scaling, then the intersection of the top-k, top-p and min-p
 * keep sets, which is one keep-threshold v* on the logit (the kept set is
 * every allowed token with logit >= v*), then a Gumbel-max draw over the kept
 * set: token = argmax_i (l_i / T + G_i), ties to the lower index, where G_i is
 * the standard Gumbel variate of the i-th token's Philox4x32-10 word under key
 * (seed lo, seed hi) and counter (i >> 2, row, offset lo, offset hi).
 * logits-mask-xpu, "Method": top_k == 1 returns the argmax.
 *   logits       [B, logits_row_stride] of dtype, read only
 *   bitmask      [B, mask_row_stride] int32 or NULL; a disallowed token is
 *                treated as -inf (the logits are not modified)
 *   temperature  [B] float or NULL to use temperature_s for every row;
 *                T <= 0 is greedy (argmax, lowest index on ties)
 *   top_k        [B] int32 or NULL (top_k_s); k <= 0 disables, k == 1 argmax,
 *                k >= number of allowed tokens keeps all; ties at the k-th
 *                value are all kept
 *   top_p        [B] float or NULL (top_p_s); p >= 1 disables; keeps every
 *                token whose probability mass strictly above it is < p; the
 *                argmax class is always kept
 *   min_p        [B] float or NULL (min_p_s); <= 0 disables; keeps tokens with
 *                probability >= min_p times the largest probability
 *   seed, offset the draw key; advance offset every decoding step
 *   tokens_out   [B] int64: the token, or -1 for a row with no allowed finite
 *                logit
 *   min_kept_logit_out  [B] float or NULL: v* (the argmax value for greedy
 *                rows, -inf when no filter is active, NaN for an empty row)
 *   workspace    device scratch of at least tsa_sample_workspace_bytes(B, V,
 *                dtype) bytes, 256-byte aligned, no initialisation needed, or
 *                NULL when that size is 0 (batches of 128 rows or more: one
 *                CTA holds each row's state on chip).  Smaller batches split
 *                rows across the GPU; the workspace then holds per-slice
 *                summaries and candidate lists, all written by the call before
 *                it reads them.  Calls that may run concurrently must use
 *                different workspaces.  TSA_ERR_WORKSPACE if a size > 0 is
 *                needed and the workspace is NULL or too small.
 * NaN logits are treated as -inf.  Rows with identical arguments give
 * bit-identical tokens on every call.
 */
int tsa_sample(const void *logits, tsa_dtype dtype, int64_t B, int64_t V,
               int64_t logits_row_stride, const int32_t *bitmask, int64_t mask_row_stride,
               const float *temperature, float temperature_s, const int32_t *top_k,
               int32_t top_k_s, const float *top_p, float top_p_s, const float *min_p,
               float min_p_s, uint64_t seed, uint64_t offset, int64_t *tokens_out,
               float *min_kept_logit_out, void *workspace, size_t workspace_bytes,
               void *stream);
/* Workspace bytes `sample` needs for B rows of V elements: 0 when B >= 128
 * (every row is resolved on chip by one CTA), and 0 for invalid sizes. */
size_t tsa_sample_workspace_bytes(int64_t B, int64_t V, tsa_dtype dtype);

/*
 * lm_head_topk -- lm-head-topk, "API", "Method" and "Correctness" (the dense
 * head): the exact top-k of scores = hidden . weight^T (+ bias) per hidden
 * row, without writing the [M, V] score matrix.  One CTA per 512-entry chunk
 * of the vocabulary computes its scores (fp32 accumulation of bf16 products)
 * and keeps its best min(k, 512); the exact top-k of those candidates follows
 * (tsa_topk), and their positions are mapped back to vocabulary indices.
 * Values are sorted descending, ties to the lower vocabulary index.  The
 * weight is read once per call; every hidden row is scored in that one read.
 *   hidden       bf16 [M, hidden_row_stride], 1 <= M <= 4 (M == 0: no-op)
 *   weight       bf16 [V, weight_row_stride]; H a multiple of 8, 8 <= H <=
 *                8192; both row strides multiples of 8 elements and both
 *                bases 16-byte aligned (TSA_ERR_ALIGN)
 *   bias         float [V] or NULL
 *   k            1 <= k <= min(2048, V) (TSA_ERR_K_RANGE)
 *   values_out   float [M, k]; indices_out int64 [M, k]
 *   workspace    at least tsa_lm_head_topk_workspace_bytes(M, V, k) bytes,
 *                256-byte aligned (the chunks' candidates)
 */
int tsa_lm_head_topk(const void *hidden, int64_t M, int64_t H, int64_t hidden_row_stride,
                     const void *weight, int64_t V, int64_t weight_row_stride, const float *bias,
                     int32_t k, float *values_out, int64_t *indices_out, void *workspace,
                     size_t workspace_bytes, void *stream);
size_t tsa_lm_head_topk_workspace_bytes(int64_t M, int64_t V, int32_t k);

/*
 * sample_sequential -- tsa_sample with top-p taken over the softmax
 * renormalised over the top-k survivors, the reading of the transformers
 * processor chain that logits-processor names as its reference (top-k, then
 * top-p, then min-p, each on what the one before kept), instead of the
 * intersection on the full softmax.  Without top-k (or top-p) the two
 * readings agree.  Three steps on `stream`: tsa_sample with top-p and min-p
 * off gives the top-k cut v_k per row; a bitmask of the tokens the caller's
 * mask allows with logit >= v_k; tsa_sample over that mask with every filter.
 * The draw is keyed as in tsa_sample (same seed and offset, same Philox word
 * per token), so a row whose keep set is the same gets the same token.
 *   arguments as tsa_sample, except
 *   workspace   at least tsa_sample_sequential_workspace_bytes(B, V, dtype)
 *               bytes, 256-byte aligned (never NULL for B >= 1: it holds the
 *               survivors' bitmask and v_k)
 */
int tsa_sample_sequential(const void *logits, tsa_dtype dtype, int64_t B, int64_t V,
                          int64_t logits_row_stride, const int32_t *bitmask,
                          int64_t mask_row_stride, const float *temperature, float temperature_s,
                          const int32_t *top_k, int32_t top_k_s, const float *top_p,
                          float top_p_s, const float *min_p, float min_p_s, uint64_t seed,
                          uint64_t offset, int64_t *tokens_out, float *min_kept_logit_out,
                          void *workspace, size_t workspace_bytes, void *stream);
/* Workspace bytes sample_sequential needs: B ceil(V / 32) words of bitmask and
 * B floats (each rounded up to 256 bytes) plus tsa_sample's workspace; 0 for
 * invalid sizes. */
size_t tsa_sample_sequential_workspace_bytes(int64_t B, int64_t V, tsa_dtype dtype);

/*
 * sample_icdf -- logits-mask-xpu, "Usage" (pass uniform [B] for deterministic
 * draws) and "Method" (the cooperative inverse-CDF draw).  The keep set is
 * tsa_sample's: every allowed finite logit >= v*.  With weights
 * w_i = exp((l_i - m) / T) over it, walked in token-index order with running
 * sums S_i, the token is the first kept one with S_i > u W, W the kept total
 * (the last kept token if rounding leaves u W unpassed).  Each row takes one
 * CTA: one read forms the masses of eight contiguous chunks, a scan over them
 * finds the chunk holding u W, and only that chunk is walked again.  Greedy
 * rows (T <= 0 or top_k == 1) give the argmax and empty rows -1, as
 * tsa_sample does.  The sums run in compensated fp32, so a token whose
 * boundary S_i lies within about 1e-6 W of u W may differ from an exact
 * (double precision) walk.
 *   uniform             [B] float in [0, 1), read only; u outside it gives
 *                       the first (u < 0) or last (u >= 1) kept token
 *   min_kept_logit_out  [B] float, REQUIRED here: v* per row, written by the
 *                       selection and read by the draw
 *   every other argument as tsa_sample (the same workspace size; no seed)
 * The call enqueues tsa_sample's kernels and then the draw's kernel.
 */
int tsa_sample_icdf(const void *logits, tsa_dtype dtype, int64_t B, int64_t V,
                    int64_t logits_row_stride, const int32_t *bitmask, int64_t mask_row_stride,
                    const float *temperature, float temperature_s, const int32_t *top_k,
                    int32_t top_k_s, const float *top_p, float top_p_s, const float *min_p,
                    float min_p_s, const float *uniform, int64_t *tokens_out,
                    float *min_kept_logit_out, void *workspace, size_t workspace_bytes,
                    void *stream);

/*
 * bitmask_from_allowed -- logits-mask-xpu, "Usage": pack a [B, V] bool
 * allow-set, one byte per token (nonzero = allowed), into the bitmask layout
 * every call here reads: token i is bit (i & 31) of word (i >> 5); the bits
 * of the last word past V are written 0.
 *   allowed      [B, allowed_row_stride] uint8, read only
 *   bitmask_out  [B, mask_row_stride] int32, words 0 .. ceil(V / 32) - 1 of
 *                each row written
 * Returns TSA_OK or a negative status (TSA_ERR_SHAPE, TSA_ERR_NULL,
 * TSA_ERR_STRIDE, TSA_ERR_ALIGN, TSA_ERR_CUDA).
 */
int tsa_bitmask_from_allowed(const uint8_t *allowed, int64_t B, int64_t V,
                             int64_t allowed_row_stride, int32_t *bitmask_out,
                             int64_t mask_row_stride, void *stream);

/*
 * sample_noalloc -- tsa_sample without a caller workspace.  The papers this
 * library follows have no counterpart: it exists for callers that cannot
 * allocate device memory when they sample (fixed, fully handed-out memory
 * pools; hosts that expose only the tensors they pass in; paths where an
 * allocation could synchronise the device or fail).  Arguments, results and
 * errors are those of tsa_sample, minus workspace / workspace_bytes.
 *   - Scratch is a fixed device array of TSA_SAMPLE_NOALLOC_SCRATCH_BYTES
 *     inside the library, held on every GPU where the library's module is
 *     loaded until the process exits.  The call itself allocates nothing.
 *   - The arguments are checked first, exactly as tsa_sample checks them.
 *     Then, when tsa_sample_workspace_bytes(B, V, dtype) exceeds
 *     TSA_SAMPLE_NOALLOC_SCRATCH_BYTES, the call returns TSA_ERR_WORKSPACE
 *     and launches nothing.  Only batches under 128 rows use the scratch;
 *     127 rows fit vocabularies up to about 265,000 fp32 or 530,000 bf16 /
 *     f16 entries, and 64 rows of an 800,000-entry fp32 vocabulary are
 *     refused.
 *   - A call on a stream that is not capturing looks up the array's device
 *     address on the current device (the first lookup may load the library's
 *     module there); a call on a capturing stream reuses the address that the
 *     last call outside capture found, so make the first call on each device
 *     outside any stream capture.
 *   - All calls on a device share the one array.  Calls that overlap on the
 *     GPU (different streams or threads without ordering between them) race
 *     and give wrong tokens; calls ordered on one stream are safe.  The array
 *     keeps the last call's contents, and nothing in it needs to start at
 *     zero.
 */
#define TSA_SAMPLE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int tsa_sample_noalloc(const void *logits, tsa_dtype dtype, int64_t B, int64_t V,
                       int64_t logits_row_stride, const int32_t *bitmask, int64_t mask_row_stride,
                       const float *temperature, float temperature_s, const int32_t *top_k,
                       int32_t top_k_s, const float *top_p, float top_p_s, const float *min_p,
                       float min_p_s, uint64_t seed, uint64_t offset, int64_t *tokens_out,
                       float *min_kept_logit_out, void *stream);

/*
 * topk -- lm-head-topk, "API" and "Method": the exact k largest logits of
 * every row, sorted by value descending with ties resolved to the lower
 * vocabulary index (the order of torch.topk on the materialised row).
 *   logits       [B, logits_row_stride] of dtype, read only
 *   k            1 <= k <= min(2048, V)
 *   values_out   [B, k] float: exact copies of the selected logits
 *   indices_out  [B, k] int64
 *   workspace    reserved; pass NULL / 0 (tsa_topk_workspace_bytes is 0)
 * -0.0 and +0.0 compare equal (the index decides); NaN ranks above +inf.
 */
int tsa_topk(const void *logits, tsa_dtype dtype, int64_t B, int64_t V,
             int64_t logits_row_stride, int32_t k, float *values_out, int64_t *indices_out,
             void *workspace, size_t workspace_bytes, void *stream);
size_t tsa_topk_workspace_bytes(int64_t B, int64_t V, int32_t k, tsa_dtype dtype);

/*
 * selective_log_softmax ("Selective Log Softmax": one log-probability per
 * row, the row's logit at a given index less the row's log-sum-exp), over the
 * allowed tokens of the temperature-scaled row:
 *   out[b] = (l[b, i_b] - m_b) / T_b - ln sum_{j allowed} exp((l[b, j] - m_b) / T_b),
 *   m_b the row's largest allowed logit.  Called with sample's tokens, it gives
 *   the log-probability of each sampled token before top-k / top-p / min-p.
 *   logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride,
 *   temperature, temperature_s: as for tsa_sample (device pointers; bitmask and
 *                temperature may be NULL); T <= 0 uses T = 1, the page's
 *                unscaled definition.
 *   index        [B] int64 device pointer, read only.
 *   out          [B] float device pointer: -inf for a disallowed index; NaN
 *                for an index outside [0, V) or a row with no allowed finite
 *                logit.  NaN logits count as -inf; +inf logits give NaN.
 * Reads each row once from HBM.  Errors as for tsa_apply_token_bitmask;
 * TSA_ERR_NULL when index or out is NULL (B > 0); TSA_ERR_ALIGN for a
 * misaligned index (8 bytes) or out / temperature (4 bytes).
 */
int tsa_selective_log_softmax(const void *logits, tsa_dtype dtype, int64_t B, int64_t V,
                              int64_t logits_row_stride, const int32_t *bitmask, int64_t mask_row_stride,
                              const float *temperature, float temperature_s, const int64_t *index,
                              float *out, void *stream);

/* Human-readable name of a status code. */
const char *tsa_status_string(int status);

/*
 * Device status: a bit set by any kernel of this library whose bounded wait
 * ran out on the current device.  Synchronises the device, returns TSA_OK or
 * TSA_ERR_DEVICE_TIMEOUT, and clears the flag when `clear` is non-zero.
 */
int tsa_device_status(int clear);

/*
 * Self-test of the bounded-wait path: launches one block that waits on a
 * barrier nothing will complete, with a wait limit of `limit_us`
 * microseconds; the kernel gives up, records the timeout flag and returns.
 * Used by the test-suite to check the failure path without hanging a GPU.
 */
int tsa_selftest_wait_timeout(uint32_t limit_us, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* TSA_H */
