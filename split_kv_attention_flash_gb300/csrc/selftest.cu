// selftest.cu -- a kernel that proves the bounded-wait path: it waits on an mbarrier
// that nothing ever arrives on, through the same helper every kernel of the library
// uses for its waits, so the wait runs out, records its code in the device error
// word and returns. No fault, trap or hang is involved.
#include "sk_common.cuh"
#include "sm100_ptx.cuh"

namespace sk {

constexpr int kSelftestCode = 0x401;

__global__ void __launch_bounds__(32) selftest_wait_kernel(int *err, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::fence_mbar_init();
        // phase 0 never completes: no thread arrives
        (void)ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0, &abort_flag, err, kSelftestCode, timeout_ns);
    }
}

cudaError_t launch_selftest_wait(int *err, unsigned long long timeout_ns, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace sk
