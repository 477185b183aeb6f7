// dispatch.cu -- picks the partial kernel for a validated problem.
#include "sk_dispatch.h"

namespace sk {

// Tensor cores (tcgen05) for 16-bit storage with the library's M block (prefill and decode;
// launches of many short units in the persistent form, one CTA per SM);
// the streaming decode kernel for up to 16 queries per sequence where the tensor-core
// kernel does not apply (other M blocks, more than 65535 (sequence, split) units, tensors
// its TMA maps cannot describe); the register-tiled CUDA-core kernel for the rest (f32 storage,
// other M blocks, no keys).
const char *partial_kernel_name(const Problem &p, int dtype, const TensorView &q,
                                const TensorView &k, const TensorView &v) {
    (void)q; (void)k; (void)v;
    if (tc::partial_tc_supported(p, dtype)) return tc::persist_selected(p) ? "partial_tc_persist" : "partial_tc";
    if (dec::partial_decode_supported(p, dtype)) return "partial_decode";
    return "partial_fma";
}

cudaError_t run_partial(const Problem &p, int dtype, const TensorView &q, const TensorView &k,
                        const TensorView &v, float *o_part, float *lse_part, const TensorView *out,
                        float *lse_out, cudaStream_t st) {
    if (tc::partial_tc_supported(p, dtype)) {
        bool launched = false;
        cudaError_t e = tc::launch_partial_tc(p, dtype, q, k, v, o_part, lse_part, out, lse_out,
                                              nullptr, st, &launched);
        if (launched || e != cudaSuccess) return e;
    }
    if (dec::partial_decode_supported(p, dtype)) {
        bool launched = false;
        cudaError_t e = dec::launch_partial_decode(p, dtype, q, k, v, o_part, lse_part, out, lse_out,
                                                   st, &launched);
        if (launched || e != cudaSuccess) return e;
    }
    return launch_partial_fma(p, dtype, q, k, v, o_part, lse_part, out, lse_out, st);
}

cudaError_t run_partial_fused(const Problem &p, int dtype, const TensorView &q,
                              const TensorView &k, const TensorView &v, float *o_part,
                              float *lse_part, const TensorView &out, float *lse_out, int *tickets,
                              cudaStream_t st, bool *fused) {
    *fused = false;
    if (!tc::partial_tc_supported(p, dtype)) return cudaSuccess;
    return tc::launch_partial_tc(p, dtype, q, k, v, o_part, lse_part, &out, lse_out, tickets, st,
                                 fused);
}

}  // namespace sk
