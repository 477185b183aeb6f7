// counts.cu -- per-row valid-split counts ([P1] Technical details, computeValidSplitKV).
#include "sk_common.cuh"

namespace sk {

// One thread per packed query row; blockIdx.y strides over sequences.
__global__ void __launch_bounds__(256) counts_kernel(Problem p, int32_t *counts) {
    for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
        SeqInfo si = seq_info(p, b);
        for (int pos = blockIdx.x * blockDim.x + threadIdx.x; pos < si.sq;
             pos += gridDim.x * blockDim.x)
            counts[si.q0 + pos] = valid_split_count(p, si.last_valid, pos);
    }
}

cudaError_t launch_counts(const Problem &p, int32_t *counts, cudaStream_t st) {
    if (p.total_q == 0 || p.max_sq == 0) return cudaSuccess;
    int bx = (p.max_sq + 255) / 256;
    if (bx > 1024) bx = 1024;
    int by = p.B < 65535 ? p.B : 65535;
    counts_kernel<<<dim3(bx, by), 256, 0, st>>>(p, counts);
    return cudaGetLastError();
}

}  // namespace sk
