// sk_static.cu -- sk_attn_fwd_static: the one-call forward pass for callers that
// cannot allocate device memory.
//
// sk_attn_fwd needs a caller-provided workspace for the split counts and the split
// partials whenever it splits the keys. Some callers have no way to provide one at
// the moment they run attention: code whose device memory is planned once up front
// (a serving loop that must not allocate per request), or code running under a host
// framework that owns every allocation and exposes no allocator to plugins. For
// them this file keeps a fixed scratch array inside the library and passes it to
// the ordinary sk_attn_fwd path as its workspace.
#include <stdint.h>

#include <mutex>

#include <cuda_runtime.h>

#include "splitkv.h"

namespace {

// Scratch of sk_attn_fwd_static (split counts, partial outputs, partial LSEs). It is
// a file-scope device array, so every GPU that loads the library holds these bytes
// until the process exits.
__device__ __align__(256) unsigned char g_static_scratch[SK_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
cudaError_t g_scratch_status[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, not a device address, so the address
// is asked of the runtime once per device, with that device current, and kept.
sk_status scratch_for_current_device(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SK_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SK_ERR_UNSUPPORTED;
    std::call_once(g_scratch_once[dev], [dev] {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        g_scratch_status[dev] = e;
        g_scratch_addr[dev] = e == cudaSuccess ? ptr : nullptr;
        if (e != cudaSuccess) (void)cudaGetLastError();
    });
    if (g_scratch_status[dev] != cudaSuccess || g_scratch_addr[dev] == nullptr) return SK_ERR_CUDA;
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
