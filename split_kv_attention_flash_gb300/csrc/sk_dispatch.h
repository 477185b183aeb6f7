// sk_dispatch.h -- choice of the partial kernel for a validated problem.
#pragma once

#include "sk_common.cuh"

namespace sk {

// Launches the partial kernel that fits the problem. With `out` non-null (S == 1)
// the kernel writes the final output and LSE instead of the partial buffers.
cudaError_t run_partial(const Problem &p, int dtype, const TensorView &q, const TensorView &k,
                        const TensorView &v, float *o_part, float *lse_part, const TensorView *out,
                        float *lse_out, cudaStream_t st);

// Name of the kernel run_partial would launch.
const char *partial_kernel_name(const Problem &p, int dtype, const TensorView &q,
                                const TensorView &k, const TensorView &v);

}  // namespace sk
