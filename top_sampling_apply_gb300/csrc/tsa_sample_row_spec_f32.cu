// The one-CTA-per-row sample kernel specialised for f32 rows that all take
// one filtered mode (with or without top-p) and one 16-byte aligned mask
// layout (none, or aligned): only that mode's stream and end code are
// compiled in.  Its own translation unit, so that it compiles in parallel
// with the others.
#include "tsa_sample_row.cuh"

namespace tsa {

const void *sample_row_spec_kernel_f32(int spec) {
    switch (spec) {
        case kFilter * 4 + 0: return (const void *)sample_row_kernel<0, kFilter * 4 + 0>;
        case kFilter * 4 + 1: return (const void *)sample_row_kernel<0, kFilter * 4 + 1>;
        case kFilterZ * 4 + 0: return (const void *)sample_row_kernel<0, kFilterZ * 4 + 0>;
        case kFilterZ * 4 + 1: return (const void *)sample_row_kernel<0, kFilterZ * 4 + 1>;
        default: return nullptr;
    }
}

unsigned int *sample_row_spec_status_ptr_f32() { return row_status_word(); }

}  // namespace tsa
