// tsa_sample_noalloc: the sample call with library-owned scratch, for callers
// that cannot allocate device memory.
//
// Some callers have no way to reach an allocator at the moment they sample:
// code running inside a runtime whose memory pools are fixed and fully handed
// out before the first step, embedded or plugin hosts that expose only the
// tensors they pass in, and code paths where a cudaMalloc (or a framework's
// caching allocator) could synchronise the device or fail under memory
// pressure.  For them the scratch of the sample call lives in a fixed
// file-scope device array instead of a caller workspace.  The array is part of
// this library's device image, so every GPU on which the library's module is
// loaded holds its TSA_SAMPLE_NOALLOC_SCRATCH_BYTES until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/tsa.h"
#include "tsa_host.h"

namespace {

// The scratch shared by every tsa_sample_noalloc call on a device.  In host
// code this name is only a handle the runtime maps to the device copy; the
// device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TSA_SAMPLE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device.  Outside stream
// capture it is looked up on every call (the lookup loads the library's module
// on a device that has none, and follows a context that was reset and made
// again); a call on a capturing stream reuses the address found by the last
// call on that device outside capture.
int noalloc_scratch(cudaStream_t stream, void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TSA_ERR_CUDA;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (stream != nullptr && cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return TSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (cs == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return TSA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    if (!g_noalloc_ptr[dev]) return TSA_ERR_CUDA;  // first call on this device made inside a capture
    *out = g_noalloc_ptr[dev];
    return TSA_OK;
}

}  // namespace

extern "C" int tsa_sample_noalloc(const void *logits, tsa_dtype dtype, int64_t B, int64_t V,
                                  int64_t logits_row_stride, const int32_t *bitmask,
                                  int64_t mask_row_stride, const float *temperature, float temperature_s,
                                  const int32_t *top_k, int32_t top_k_s, const float *top_p,
                                  float top_p_s, const float *min_p, float min_p_s, uint64_t seed,
                                  uint64_t offset, int64_t *tokens_out, float *min_kept_logit_out,
                                  void *stream) {
    // the checks of tsa_sample come first, so an invalid call reports what
    // tsa_sample would report, whatever its size
    int st = tsa::sample_check_args(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride,
                                    temperature, top_k, top_p, min_p, tokens_out, min_kept_logit_out);
    if (st != TSA_OK) return st;
    const size_t need = tsa_sample_workspace_bytes(B, V, dtype);
    if (need > (size_t)TSA_SAMPLE_NOALLOC_SCRATCH_BYTES) return TSA_ERR_WORKSPACE;
    void *scratch = nullptr;
    size_t scratch_bytes = 0;
    // need == 0: an empty batch, a size tsa_sample rejects, or a batch whose
    // rows are each held on chip by one CTA; none of them touches the scratch
    if (need > 0) {
        st = noalloc_scratch((cudaStream_t)stream, &scratch);
        if (st != TSA_OK) return st;
        scratch_bytes = (size_t)TSA_SAMPLE_NOALLOC_SCRATCH_BYTES;
    }
    return tsa_sample(logits, dtype, B, V, logits_row_stride, bitmask, mask_row_stride, temperature,
                      temperature_s, top_k, top_k_s, top_p, top_p_s, min_p, min_p_s, seed, offset,
                      tokens_out, min_kept_logit_out, scratch, scratch_bytes, stream);
}
