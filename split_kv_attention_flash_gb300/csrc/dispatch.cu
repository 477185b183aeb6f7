// dispatch.cu -- picks the partial kernel for a validated problem.
#include "sk_dispatch.h"

namespace sk {

const char *partial_kernel_name(const Problem &p, int dtype, const TensorView &q,
                                const TensorView &k, const TensorView &v) {
    (void)p; (void)dtype; (void)q; (void)k; (void)v;
    return "partial_simt";
}

cudaError_t run_partial(const Problem &p, int dtype, const TensorView &q, const TensorView &k,
                        const TensorView &v, float *o_part, float *lse_part, const TensorView *out,
                        float *lse_out, cudaStream_t st) {
    return launch_partial_simt(p, dtype, q, k, v, o_part, lse_part, out, lse_out, st);
}

}  // namespace sk
