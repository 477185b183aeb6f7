// sk_static.cu -- sk_attn_fwd_static: the one-call forward pass for callers that
// cannot allocate device memory.
//
// sk_attn_fwd needs a caller-provided workspace for the split partials (and, for the
// merge fused into the tensor-core kernel, its per-M-block tickets) whenever it splits
// the keys. Some callers have no way to provide one at the moment they run attention:
// code whose device memory is planned once up front (a serving loop that must not
// allocate per request), or code running under a host framework that owns every
// allocation and exposes no allocator to plugins. For them this file keeps a fixed
// scratch array inside the library and passes it to the ordinary sk_attn_fwd path as
// its workspace.
#include <stdint.h>

#include <mutex>

#include <cuda_runtime.h>

#include "sk_dispatch.h"
#include "splitkv.h"

namespace {

// Scratch of sk_attn_fwd_static: the split partials O_s and L_s, and the tickets of the
// fused merge. It is a file-scope device array, so every GPU that loads the library
// holds these bytes until the process exits.
__device__ __align__(256) unsigned char g_static_scratch[SK_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device. In host code the array's
// name is only a host-side stand-in, not a device address, so the address is asked of
// the runtime with that device current. Only a successful lookup is kept: one that
// failed (a sticky error pending, a first call made during stream capture) is tried
// again by the next call, and its error is what sk_last_cuda_error reports.
sk_status scratch_for_current_device(void **addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return sk::record_cuda_error(e);
    }
    if (dev < 0 || dev >= kMaxDevices) return SK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            (void)cudaGetLastError();
            return sk::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        }
        g_scratch_addr[dev] = ptr;
    }
    *addr = g_scratch_addr[dev];
    return SK_OK;
}

}  // namespace

extern "C" sk_status sk_attn_fwd_static(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v,
                                        sk_tensor out, float *lse_out, sk_stream stream) {
    size_t need = 0;
    sk_status st = sk_workspace_bytes(p, &need);
    if (st != SK_OK) return st;
    if (need > (size_t)SK_STATIC_SCRATCH_BYTES) return SK_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0 && (st = scratch_for_current_device(&scratch)) != SK_OK) return st;
    return sk_attn_fwd(p, q, k, v, out, lse_out, scratch, need, stream);
}
