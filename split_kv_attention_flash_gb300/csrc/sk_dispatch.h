// sk_dispatch.h -- choice of the partial kernel for a validated problem.
#pragma once

#include "sk_common.cuh"
#include "splitkv.h"

namespace sk {

// Launches the partial kernel that fits the problem. With `out` non-null (S == 1)
// the kernel writes the final output and LSE instead of the partial buffers.
cudaError_t run_partial(const Problem &p, int dtype, const TensorView &q, const TensorView &k,
                        const TensorView &v, float *o_part, float *lse_part, const TensorView *out,
                        float *lse_out, cudaStream_t st);

// The tensor-core partial kernel with the merge fused in: the last CTA of every
// (sequence, head, M block) merges its splits into out / lse_out. `tickets` (one int per
// (sequence, head, M block), zeroed beforehand) count the finished splits. Sets *fused
// when it launched; otherwise nothing ran and the caller takes the counts / partial /
// combine path.
cudaError_t run_partial_fused(const Problem &p, int dtype, const TensorView &q,
                              const TensorView &k, const TensorView &v, float *o_part,
                              float *lse_part, const TensorView &out, float *lse_out, int *tickets,
                              cudaStream_t st, bool *fused);

// Records `e` as the calling thread's last CUDA error (sk_last_cuda_error) and returns
// SK_ERR_CUDA, or SK_OK for cudaSuccess.
sk_status record_cuda_error(cudaError_t e);

// Name of the kernel run_partial would launch.
const char *partial_kernel_name(const Problem &p, int dtype, const TensorView &q,
                                const TensorView &k, const TensorView &v);

}  // namespace sk
