// sk_host.cu -- sk_attn_fwd_host: the one-call forward pass with Q, K, V and the output in
// host memory. The call copies the inputs into a caller-owned device buffer, runs the
// forward pass there and copies the output back, all enqueued on the caller's stream.
#include <stdint.h>

#include <cuda_runtime.h>

#include "sk_dispatch.h"
#include "splitkv.h"

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
int elem_size(sk_dtype t) { return t == SK_F32 ? 4 : 2; }

// Device buffer of sk_attn_fwd_host: Q | K | V | out | LSE | sk_attn_fwd's workspace.
struct HostLayout {
    size_t q, k, v, out, lse, ws, ws_bytes, total;
    size_t q_bytes, k_bytes, v_bytes, out_bytes, lse_bytes;
};

sk_status host_layout(const sk_params *p, sk_dtype dtype, bool with_lse, HostLayout *L) {
    if (!p || (dtype != SK_BF16 && dtype != SK_F16 && dtype != SK_F32)) return SK_ERR_INVALID_ARG;
    size_t ws = 0;
    const sk_status st = sk_workspace_bytes(p, &ws);  // validates p
    if (st != SK_OK) return st;
    const size_t es = (size_t)elem_size(dtype);
    L->q_bytes = (size_t)p->total_q * p->H * p->d_qk * es;
    L->k_bytes = (size_t)p->total_k * p->H * p->d_qk * es;
    L->v_bytes = (size_t)p->total_k * p->H * p->d_v * es;
    L->out_bytes = (size_t)p->total_q * p->H * p->d_v * es;
    L->lse_bytes = with_lse ? (size_t)p->H * p->total_q * 4 : 0;
    // every region at least 256 bytes, so that each device pointer is valid and distinct
    L->q = 0;
    L->k = L->q + align256(L->q_bytes > 0 ? L->q_bytes : 1);
    L->v = L->k + align256(L->k_bytes > 0 ? L->k_bytes : 1);
    L->out = L->v + align256(L->v_bytes > 0 ? L->v_bytes : 1);
    L->lse = L->out + align256(L->out_bytes > 0 ? L->out_bytes : 1);
    L->ws = L->lse + align256(L->lse_bytes);
    L->ws_bytes = ws;
    L->total = L->ws + align256(ws);
    return SK_OK;
}

// A host tensor must be one contiguous block: [rows][H][d] packed, or [B][seq][H][d] dense.
bool contiguous(const sk_params *p, const sk_tensor &t, int d, int seq) {
    if (t.stride_h != d || t.stride_row != (int64_t)p->H * d) return false;
    if (p->cu_seqlens_q == nullptr && t.stride_b != (int64_t)seq * p->H * d) return false;
    return true;
}

}  // namespace

extern "C" sk_status sk_host_buffer_bytes(const sk_params *p, sk_dtype dtype, int with_lse,
                                          size_t *bytes) {
    if (!bytes) return SK_ERR_INVALID_ARG;
    HostLayout L;
    const sk_status st = host_layout(p, dtype, with_lse != 0, &L);
    if (st != SK_OK) return st;
    *bytes = L.total;
    return SK_OK;
}

extern "C" sk_status sk_attn_fwd_host(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v,
                                      sk_tensor out, float *lse_out, void *device_buffer,
                                      size_t device_bytes, sk_stream stream) {
    if (!p || !q.ptr || !k.ptr || !v.ptr || !out.ptr) return SK_ERR_INVALID_ARG;
    if (q.dtype != k.dtype || q.dtype != v.dtype || q.dtype != out.dtype) return SK_ERR_UNSUPPORTED;
    HostLayout L;
    sk_status st = host_layout(p, q.dtype, lse_out != nullptr, &L);
    if (st != SK_OK) return st;
    if (!contiguous(p, q, p->d_qk, p->max_seqlen_q) || !contiguous(p, k, p->d_qk, p->max_seqlen_k) ||
        !contiguous(p, v, p->d_v, p->max_seqlen_k) || !contiguous(p, out, p->d_v, p->max_seqlen_q))
        return SK_ERR_UNSUPPORTED;
    if (!device_buffer || ((uintptr_t)device_buffer & 255u)) return SK_ERR_INVALID_ARG;
    if (device_bytes < L.total) return SK_ERR_WORKSPACE;

    char *base = (char *)device_buffer;
    cudaStream_t cs = (cudaStream_t)stream;
    const struct { size_t off, bytes; const void *src; } in[3] = {
        {L.q, L.q_bytes, q.ptr}, {L.k, L.k_bytes, k.ptr}, {L.v, L.v_bytes, v.ptr}};
    for (const auto &c : in) {
        if (c.bytes == 0) continue;
        const cudaError_t e = cudaMemcpyAsync(base + c.off, c.src, c.bytes, cudaMemcpyHostToDevice, cs);
        if (e != cudaSuccess) return sk::record_cuda_error(e);
    }
    sk_tensor qd = q, kd = k, vd = v, od = out;
    qd.ptr = base + L.q;
    kd.ptr = base + L.k;
    vd.ptr = base + L.v;
    od.ptr = base + L.out;
    float *lse_d = lse_out ? (float *)(base + L.lse) : nullptr;
    st = sk_attn_fwd(p, qd, kd, vd, od, lse_d, L.ws_bytes ? base + L.ws : nullptr, L.ws_bytes, stream);
    if (st != SK_OK) return st;
    if (L.out_bytes > 0) {
        const cudaError_t e = cudaMemcpyAsync(out.ptr, base + L.out, L.out_bytes, cudaMemcpyDeviceToHost, cs);
        if (e != cudaSuccess) return sk::record_cuda_error(e);
    }
    if (lse_out && L.lse_bytes > 0) {
        const cudaError_t e = cudaMemcpyAsync(lse_out, lse_d, L.lse_bytes, cudaMemcpyDeviceToHost, cs);
        if (e != cudaSuccess) return sk::record_cuda_error(e);
    }
    return SK_OK;
}
