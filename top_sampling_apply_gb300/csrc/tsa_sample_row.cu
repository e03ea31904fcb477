// sample, one CTA per row: the kernel itself is in tsa_sample_row.cuh.  This
// unit holds the generic kernels (mode and mask layout per row at run time)
// and the launcher, which takes a specialised kernel (tsa_sample_row_spec*.cu)
// when every row shares one filtered mode and a 16-byte aligned layout.
#include "tsa_sample_row.cuh"

namespace tsa {

unsigned int *sample_row_status_ptr() { return row_status_word(); }

size_t sample_row_smem_bytes() { return kRowSmemBytes; }

// The specialisation every row of the launch takes (4 mode + mask layout),
// or -1 when the rows may differ or take an unspecialised mode.  The same
// tests as row_params and the kernel's mode choice, on the scalar parameters.
static int row_spec(const SampleArgs &a, int dtype) {
    if (a.temperature || a.top_k || a.top_p || a.min_p) return -1;
    const float T = a.temperature_s, P = a.top_p_s, MP = a.min_p_s;
    const int32_t K = a.top_k_s;
    const bool greedy = !(T > 0.f) || K == 1;
    const bool k_on = !greedy && K > 1, p_on = !greedy && P < 1.f, m_on = !greedy && MP > 0.f;
    const bool filtered = k_on || p_on || m_on;
    const bool tau_on = k_on && (K + kCW - 1) / kCW <= kTauMaxR;
    if (greedy || !filtered || !(tau_on || m_on)) return -1;
    const int mode = p_on ? kFilterZ : kFilter;
    int mk = 0;
    if (a.mask) {
        const int esize = dtype == 0 ? 4 : 2;
        const bool aligned_rows =
            (reinterpret_cast<uintptr_t>(a.logits) % 16) == 0 && (a.stride * esize) % 16 == 0;
        if (!aligned_rows) return -1;
        mk = 1;
    }
    return mode * 4 + mk;
}

int sample_row_launch(const SampleArgs &args, int dtype, cudaStream_t st) {
    const void *fns[3] = {(const void *)sample_row_kernel<0, -1>, (const void *)sample_row_kernel<1, -1>,
                          (const void *)sample_row_kernel<2, -1>};
    const void *fn = fns[dtype];
    const int spec = row_spec(args, dtype);
    if (spec >= 0) {
        const void *sf = sample_row_spec_kernel(dtype, spec);
        if (sf) fn = sf;
    }
    const size_t smem = sample_row_smem_bytes();
    if (prepare_kernel(fn, smem, 1) != 0) return -1;
    SampleArgs a = args;
    void *params[] = {&a};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)args.B, 1, 1);
    cfg.blockDim = dim3(kRowThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, params) == cudaSuccess ? 0 : -1;
}

}  // namespace tsa
