// sk_api.cu -- the C ABI of include/splitkv.h: validation, split selection,
// workspace layout and dispatch to the kernels. No kernel lives here.
#include <math.h>
#include <string.h>

#include <mutex>

#include "sk_common.cuh"
#include "sk_dispatch.h"
#include "splitkv.h"

namespace {

// Device word that bounded device-side waits set when they give up.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
int *g_err_ptr[kMaxDevices];
std::mutex g_err_mutex;

// Device address of the error word on the current device. Only a successful lookup is
// kept, so a lookup that failed (a sticky error pending, a call made during stream
// capture) is tried again by the next call.
int *device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (!g_err_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_error) == cudaSuccess) g_err_ptr[dev] = (int *)ptr;
        else (void)cudaGetLastError();
    }
    return g_err_ptr[dev];
}

int elem_size(sk_dtype t) { return t == SK_F32 ? 4 : 2; }
bool dtype_ok(int t) { return t == SK_BF16 || t == SK_F16 || t == SK_F32; }

bool aligned16(const void *ptr) { return ((uintptr_t)ptr & 15u) == 0; }

sk_status check_params(const sk_params *p) {
    if (!p) return SK_ERR_INVALID_ARG;
    if (p->B < 1 || p->H < 1 || p->max_seqlen_q < 0 || p->max_seqlen_k < 0 || p->total_q < 0 ||
        p->total_k < 0)
        return SK_ERR_INVALID_ARG;
    if (p->H > 65535) return SK_ERR_UNSUPPORTED;
    if ((p->cu_seqlens_q == nullptr) != (p->cu_seqlens_k == nullptr)) return SK_ERR_INVALID_ARG;
    if (!p->cu_seqlens_q) {
        if ((long long)p->B * p->max_seqlen_q != p->total_q ||
            (long long)p->B * p->max_seqlen_k != p->total_k)
            return SK_ERR_INVALID_ARG;
    }
    if (p->mask != SK_MASK_NONE && p->mask != SK_MASK_CAUSAL && p->mask != SK_MASK_PREFIX_CAUSAL)
        return SK_ERR_INVALID_ARG;
    if (p->mask != SK_MASK_PREFIX_CAUSAL && p->prefix_offset != 0) return SK_ERR_INVALID_ARG;
    if (p->last_valid_kv_index < -1) return SK_ERR_INVALID_ARG;
    if (p->n_per_block < 1) return SK_ERR_INVALID_ARG;  // [P1] assert(nPerBlock > 0)
    if (p->split_kv < 0 || p->split_kv > SK_MAX_SPLIT_KV) return SK_ERR_INVALID_ARG;
    if (p->block_m < 0) return SK_ERR_INVALID_ARG;
    if (!(p->softmax_scale == p->softmax_scale) || isinf(p->softmax_scale))
        return SK_ERR_INVALID_ARG;
    if (p->fuse_combine != 0 && p->fuse_combine != 1) return SK_ERR_INVALID_ARG;
    if (p->window_left < -1 || (p->window_left >= 0 && p->mask == SK_MASK_NONE))
        return SK_ERR_INVALID_ARG;
    if (!sk_supported_head_dims(p->d_qk, p->d_v)) return SK_ERR_UNSUPPORTED;
    return SK_OK;
}

sk_status check_tensor(const sk_params *p, const sk_tensor &t, int rows_per_seq, bool dense) {
    (void)rows_per_seq;
    if (!t.ptr) return SK_ERR_INVALID_ARG;
    if (!dtype_ok(t.dtype)) return SK_ERR_INVALID_ARG;
    if (t.stride_row < 0 || t.stride_h < 0 || (dense && t.stride_b < 0)) return SK_ERR_INVALID_ARG;
    const int es = elem_size(t.dtype);
    if (!aligned16(t.ptr)) return SK_ERR_UNSUPPORTED;
    if ((t.stride_row * es) % 16 || (t.stride_h * es) % 16 || (dense && (t.stride_b * es) % 16))
        return SK_ERR_UNSUPPORTED;
    (void)p;
    return SK_OK;
}

sk_status check_qkv(const sk_params *p, const sk_tensor &q, const sk_tensor &k,
                    const sk_tensor &v) {
    const bool dense = p->cu_seqlens_q == nullptr;
    sk_status st;
    if ((st = check_tensor(p, q, p->max_seqlen_q, dense)) != SK_OK) return st;
    if ((st = check_tensor(p, k, p->max_seqlen_k, dense)) != SK_OK) return st;
    if ((st = check_tensor(p, v, p->max_seqlen_k, dense)) != SK_OK) return st;
    if (q.dtype != k.dtype || q.dtype != v.dtype) return SK_ERR_UNSUPPORTED;
    return SK_OK;
}

sk_status resolve_split(const sk_params *p, int *S) {
    if (p->split_kv > 0) { *S = p->split_kv; return SK_OK; }
    return sk_auto_split_kv(p, S);
}

sk::Problem make_problem(const sk_params *p, int S) {
    sk::Problem pr{};
    pr.B = p->B;
    pr.H = p->H;
    pr.max_sq = p->max_seqlen_q;
    pr.max_sk = p->max_seqlen_k;
    pr.total_q = p->total_q;
    pr.total_k = p->total_k;
    pr.d_qk = p->d_qk;
    pr.d_v = p->d_v;
    pr.cu_q = p->cu_seqlens_q;
    pr.cu_k = p->cu_seqlens_k;
    pr.causal = p->mask != SK_MASK_NONE;
    pr.prefix_offset = p->mask == SK_MASK_PREFIX_CAUSAL ? p->prefix_offset : 0;
    pr.last_valid_kv_index = p->last_valid_kv_index;
    pr.bn = p->n_per_block;
    pr.S = S;
    pr.bm = p->block_m > 0 ? p->block_m : sk_default_block_m(p->d_qk, p->d_v, SK_BF16);
    pr.scale = p->softmax_scale != 0.f ? p->softmax_scale : (float)(1.0 / sqrt((double)p->d_qk));
    pr.scale_log2 = (float)((double)pr.scale * 1.4426950408889634074);
    pr.err = device_error_word();
    pr.window_left = p->window_left;
    pr.seqused_k = p->seqused_k;
    return pr;
}

sk::TensorView view(const sk_tensor &t) {
    return sk::TensorView{(char *)t.ptr, t.stride_b, t.stride_row, t.stride_h};
}

thread_local int t_last_cuda_error = 0;

sk_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SK_OK;
    t_last_cuda_error = (int)e;
    return SK_ERR_CUDA;
}

}  // namespace

namespace sk {
sk_status record_cuda_error(cudaError_t e) { return cuda_status(e); }
}  // namespace sk

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WorkspaceLayout {
    size_t o_part, lse_part, tickets, ticket_bytes, total;
};

// O_part | L_part | tickets (one int per (sequence, head, 256-row M block), for the
// merge fused into the tensor-core kernel), each 256-byte aligned. The counts need no
// room: the combine evaluates their formula.
WorkspaceLayout layout_for(const sk_params *p, int S) {
    WorkspaceLayout w{};
    if (S <= 1) return w;
    const size_t rows = (size_t)p->total_q;
    w.o_part = 0;
    w.lse_part = w.o_part + align256((size_t)p->H * S * rows * p->d_v * 4);
    w.tickets = w.lse_part + align256((size_t)p->H * S * rows * 4);
    w.ticket_bytes = (size_t)p->B * p->H * (((size_t)p->max_seqlen_q + 255) / 256) * 4;
    w.total = w.tickets + align256(w.ticket_bytes);
    return w;
}

}  // namespace

extern "C" {

int sk_version(void) { return 100; }

int sk_last_cuda_error(const char **name) {
    if (name) *name = t_last_cuda_error ? cudaGetErrorName((cudaError_t)t_last_cuda_error) : "cudaSuccess";
    return t_last_cuda_error;
}

const char *sk_status_string(sk_status s) {
    switch (s) {
    case SK_OK: return "ok";
    case SK_ERR_INVALID_ARG: return "invalid argument";
    case SK_ERR_UNSUPPORTED: return "unsupported configuration";
    case SK_ERR_WORKSPACE: return "workspace too small";
    case SK_ERR_CUDA: return "CUDA error";
    case SK_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

int sk_supported_head_dims(int d_qk, int d_v) {
    return (d_qk == 64 && d_v == 64) || (d_qk == 128 && d_v == 128) || (d_qk == 192 && d_v == 128);
}

int sk_default_block_m(int d_qk, int d_v, sk_dtype dtype) {
    (void)d_qk; (void)d_v; (void)dtype;
    return 256;
}

sk_status sk_choose_split_kv(const sk_params *p, int sm_count, int *split_kv_out) {
    if (!p || !split_kv_out || sm_count < 1) return SK_ERR_INVALID_ARG;
    if (p->split_kv < 0 || p->split_kv > SK_MAX_SPLIT_KV) return SK_ERR_INVALID_ARG;
    if (p->split_kv > 0) { *split_kv_out = p->split_kv; return SK_OK; }
    int S = 1;
    if (p->max_seqlen_k > 0) {
        if (p->max_seqlen_q == 1) {
            // single-query problems: enough CTAs to cover every SM twice
            long long bh = (long long)p->B * p->H;
            while (S < SK_MAX_SPLIT_KV && bh * S < 2LL * sm_count) ++S;
        } else {
            // [P2] Technical details: split-3 when Sk >= 8192 and Q_tiles * heads <= 2 * CU
            const int bm = p->block_m > 0 ? p->block_m : sk_default_block_m(p->d_qk, p->d_v, SK_BF16);
            long long q_tiles = ((long long)p->max_seqlen_q + bm - 1) / bm;
            if (p->max_seqlen_k >= 8192 && q_tiles * p->H <= 2LL * sm_count) S = 3;
        }
        // The auto rule applies where the split kernel's contract matches ([P2] Technical
        // details). The partition starts its splits at key 0 and has no window term, so a
        // sliding window that hides the whole first split from the deepest query leaves
        // that split (and often more) with nothing to do: keep such problems unsplit.
        if (S > 1 && p->window_left >= 0 && p->mask != SK_MASK_NONE && p->n_per_block >= 1) {
            const long long off = p->mask == SK_MASK_PREFIX_CAUSAL ? p->prefix_offset : 0;
            const long long deepest = (long long)p->max_seqlen_q - 1 + off;
            long long last = deepest < p->max_seqlen_k - 1 ? deepest : p->max_seqlen_k - 1;
            if (p->last_valid_kv_index >= 0 && last > p->last_valid_kv_index)
                last = p->last_valid_kv_index;
            if (last >= 0) {
                const long long nb = p->n_per_block;
                const long long tiles = (last + nb) / nb;
                const long long first_split_keys = nb * ((tiles + S - 1) / S);
                if (deepest - p->window_left >= first_split_keys) S = 1;
            }
        }
    }
    *split_kv_out = S;
    return SK_OK;
}

sk_status sk_auto_split_kv(const sk_params *p, int *split_kv_out) {
    if (!p || !split_kv_out) return SK_ERR_INVALID_ARG;
    if (p->split_kv > 0) return sk_choose_split_kv(p, 1, split_kv_out);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return cuda_status(e);
    }
    return sk_choose_split_kv(p, sms, split_kv_out);
}

sk_status sk_workspace_bytes(const sk_params *p, size_t *bytes) {
    if (!bytes) return SK_ERR_INVALID_ARG;
    sk_status st = check_params(p);
    if (st != SK_OK) return st;
    int S = 0;
    if ((st = resolve_split(p, &S)) != SK_OK) return st;
    *bytes = layout_for(p, S).total;
    return SK_OK;
}

sk_status sk_valid_split_counts(const sk_params *p, int32_t *counts, sk_stream stream) {
    sk_status st = check_params(p);
    if (st != SK_OK) return st;
    if (!counts && p->total_q > 0) return SK_ERR_INVALID_ARG;
    int S = 0;
    if ((st = resolve_split(p, &S)) != SK_OK) return st;
    return cuda_status(sk::launch_counts(make_problem(p, S), counts, (cudaStream_t)stream));
}

const char *sk_partial_kernel_name(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v) {
    if (check_params(p) != SK_OK || check_qkv(p, q, k, v) != SK_OK) return nullptr;
    int S = 0;
    if (resolve_split(p, &S) != SK_OK) return nullptr;  // split_kv = 0: the automatic choice
    return sk::partial_kernel_name(make_problem(p, S), q.dtype, view(q), view(k), view(v));
}

sk_status sk_attn_partial_fwd(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v,
                              float *o_part, float *lse_part, sk_stream stream) {
    sk_status st = check_params(p);
    if (st != SK_OK) return st;
    if ((st = check_qkv(p, q, k, v)) != SK_OK) return st;
    if (p->total_q > 0 && (!o_part || !lse_part)) return SK_ERR_INVALID_ARG;
    if (!aligned16(o_part)) return SK_ERR_UNSUPPORTED;
    int S = 0;
    if ((st = resolve_split(p, &S)) != SK_OK) return st;
    return cuda_status(sk::run_partial(make_problem(p, S), q.dtype, view(q), view(k), view(v),
                                       o_part, lse_part, nullptr, nullptr,
                                       (cudaStream_t)stream));
}

sk_status sk_combine(const sk_params *p, const float *o_part, const float *lse_part,
                     const int32_t *counts, sk_tensor out, float *lse_out, sk_stream stream) {
    sk_status st = check_params(p);
    if (st != SK_OK) return st;
    if (p->total_q > 0 && (!o_part || !lse_part || !counts)) return SK_ERR_INVALID_ARG;
    if ((st = check_tensor(p, out, p->max_seqlen_q, p->cu_seqlens_q == nullptr)) != SK_OK)
        return st;
    if (!aligned16(o_part)) return SK_ERR_UNSUPPORTED;
    int S = 0;
    if ((st = resolve_split(p, &S)) != SK_OK) return st;
    return cuda_status(sk::launch_combine(make_problem(p, S), out.dtype, o_part, lse_part, counts,
                                          view(out), lse_out, (cudaStream_t)stream));
}

sk_status sk_attn_fwd(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v, sk_tensor out,
                      float *lse_out, void *workspace, size_t workspace_bytes, sk_stream stream) {
    sk_status st = check_params(p);
    if (st != SK_OK) return st;
    if ((st = check_qkv(p, q, k, v)) != SK_OK) return st;
    if ((st = check_tensor(p, out, p->max_seqlen_q, p->cu_seqlens_q == nullptr)) != SK_OK)
        return st;
    if (out.dtype != q.dtype) return SK_ERR_UNSUPPORTED;
    int S = 0;
    if ((st = resolve_split(p, &S)) != SK_OK) return st;
    const WorkspaceLayout w = layout_for(p, S);
    if (workspace_bytes < w.total) return SK_ERR_WORKSPACE;
    if (w.total > 0 && (!workspace || ((uintptr_t)workspace & 255u))) return SK_ERR_INVALID_ARG;
    const sk::Problem pr = make_problem(p, S);
    cudaStream_t cs = (cudaStream_t)stream;
    if (p->total_q == 0) return SK_OK;
    const sk::TensorView ov = view(out);
    if (S == 1)  // the partial kernel writes the final output and LSE directly
        return cuda_status(sk::run_partial(pr, q.dtype, view(q), view(k), view(v), nullptr,
                                           nullptr, &ov, lse_out, cs));
    char *ws = (char *)workspace;
    float *o_part = (float *)(ws + w.o_part);
    float *lse_part = (float *)(ws + w.lse_part);
    if (p->fuse_combine && pr.bm == 256) {
        // the tensor-core kernel merges in its last CTA per M block: zeroed tickets, one launch
        int *tickets = (int *)(ws + w.tickets);
        cudaError_t e = cudaMemsetAsync(tickets, 0, w.ticket_bytes, cs);
        bool fused = false;
        if (e == cudaSuccess)
            e = sk::run_partial_fused(pr, q.dtype, view(q), view(k), view(v), o_part, lse_part, ov,
                                      lse_out, tickets, cs, &fused);
        if (e != cudaSuccess || fused) return cuda_status(e);
    }
    sk::Problem pe = pr;
    pe.skip_empty = 1;     // splits without keys write nothing; the combine never reads them
    pe.counts_inline = 1;  // the combine evaluates the per-row count formula itself
    cudaError_t e = sk::run_partial(pe, q.dtype, view(q), view(k), view(v), o_part, lse_part,
                                    nullptr, nullptr, cs);
    if (e == cudaSuccess) e = sk::launch_combine(pe, out.dtype, o_part, lse_part, nullptr, ov, lse_out, cs);
    return cuda_status(e);
}

sk_status sk_selftest_bounded_wait(unsigned long long timeout_ns, sk_stream stream) {
    if (timeout_ns > 2000000000ull) return SK_ERR_INVALID_ARG;
    int *err = device_error_word();
    if (!err) return SK_ERR_CUDA;
    return cuda_status(sk::launch_selftest_wait(err, timeout_ns, (cudaStream_t)stream));
}

sk_status sk_read_device_error(int *code, int clear) {
    if (!code) return SK_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return SK_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return SK_ERR_CUDA;
    if (clear) {
        int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess)
            return SK_ERR_CUDA;
    }
    *code = v;
    return v ? SK_ERR_TIMEOUT : SK_OK;
}

}  // extern "C"
