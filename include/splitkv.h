/*
 * splitkv.h -- C ABI of a split-KV attention forward pass for NVIDIA GB300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *   [P1] "Recombine fully masked split-KV attention partials on the host"
 *        (ROCm/rocmlirTriton pull request 535)
 *   [P2] "[ASM] [HIP] [JIT] [gfx942] Optimize long-context FMHA with split-KV"
 *        (ROCm/aiter pull request 5592)
 *   [P3] "[HIP] MHA v4: check Q scale backing only on the sparse path"
 *        (ROCm/aiter pull request 7651) -- only its convention that an
 *        incompatible input gets a clear error rather than a fault.
 *
 * The method ([P1] Summary): each (batch-head, M block of queries) splits its keys
 * into split_kv chunks; one partial output O_s and one log-sum-exp L_s are written
 * per split (an empty split writes O_s = 0 and L_s = -inf); a combine stage merges
 * the partials with per-row valid-split counts, NaN-safely and in f32.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     never allocates, frees or synchronises (except sk_read_device_error, which
 *     says so). Every compute call only enqueues work on `stream` and returns.
 *   - Validation happens on the host before any launch. A rejected call returns
 *     SK_ERR_INVALID_ARG or SK_ERR_UNSUPPORTED and launches nothing ([P2] Technical
 *     details: incompatible requests raise; [P3] Summary: a clear error, not a fault).
 *     A launch failure returns SK_ERR_CUDA.
 *   - Device data (cu_seqlens) cannot be checked on the host without a sync. The
 *     kernels clamp every sequence to max_seqlen_{q,k} and to total_{q,k}, so bad
 *     cu_seqlens give wrong numbers but never an out-of-bounds access.
 *   - Packed row r of sequence b (varlen) is query/key position r - cu_seqlens[b].
 *     Without cu_seqlens (dense layout) sequence b has max_seqlen_{q,k} rows and
 *     packed row index b * max_seqlen + position.
 *   - Partial buffers: o_part f32 [H][S][total_q][d_v], lse_part f32 [H][S][total_q]
 *     (the split axis sits next to the batch-head axis, as in [P1] per-row mask
 *     layout). Final LSE: f32 [H][total_q]. Counts: int32 [total_q] (one count per
 *     packed row, the same for every head -- [P1] layout [batchHeads, 1, seq_len_q, 1]
 *     broadcast over heads).
 *   - Log-sum-exps are natural logs of the scaled scores softmax_scale * q.k.
 */
#ifndef SPLITKV_H
#define SPLITKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *sk_stream;

typedef enum {
    SK_OK = 0,
    SK_ERR_INVALID_ARG = 1,   /* a null pointer, a negative size, inconsistent fields */
    SK_ERR_UNSUPPORTED = 2,   /* valid but not implemented: head dims, dtype mix, alignment */
    SK_ERR_WORKSPACE = 3,     /* workspace_bytes smaller than sk_workspace_bytes() */
    SK_ERR_CUDA = 4,          /* a CUDA runtime call or a launch failed */
    SK_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up (sk_read_device_error) */
} sk_status;

typedef enum { SK_BF16 = 0, SK_F16 = 1, SK_F32 = 2 } sk_dtype;

/* [P1] Technical details: under causal and prefix-causal masking key j is visible to
 * query q when j <= q + prefix_offset (prefix_offset is 0 for plain causal);
 * under every mask j must also be <= lastValid. A sliding window (window_left >= 0)
 * also hides keys before q + prefix_offset - window_left; it changes neither the
 * per-row counts nor the partition (leading splits of a row then hold nothing). */
typedef enum { SK_MASK_NONE = 0, SK_MASK_CAUSAL = 1, SK_MASK_PREFIX_CAUSAL = 2 } sk_mask;

/* A [rows, heads, dim] (varlen) or [batch, rows, heads, dim] (dense) tensor with a
 * contiguous innermost dimension. Strides are in elements. The base pointer and
 * every stride times the element size must be multiples of 16 bytes. */
typedef struct {
    void *ptr;
    sk_dtype dtype;
    int64_t stride_b;     /* between sequences; dense layout only (ignored with cu_seqlens) */
    int64_t stride_row;   /* between consecutive rows (tokens) */
    int64_t stride_h;     /* between heads */
} sk_tensor;

typedef struct {
    int B;                       /* number of sequences (>= 1) */
    int H;                       /* heads (>= 1); K and V have H heads too */
    int max_seqlen_q;            /* >= every query length */
    int max_seqlen_k;            /* >= every key length; 0 is allowed ([P2] empty-K review) */
    int total_q;                 /* packed query rows (dense: B * max_seqlen_q) */
    int total_k;                 /* packed key rows (dense: B * max_seqlen_k) */
    int d_qk;                    /* head dim of Q and K ([P2] Motivation: 192) */
    int d_v;                     /* head dim of V and of the output ([P2]: 128) */
    const int32_t *cu_seqlens_q; /* device int32 [B+1], or NULL together with cu_seqlens_k */
    const int32_t *cu_seqlens_k; /* device int32 [B+1], or NULL (dense layout) */
    sk_mask mask;
    int prefix_offset;           /* must be 0 unless mask == SK_MASK_PREFIX_CAUSAL */
    int last_valid_kv_index;     /* -1: each sequence's last key; else min(this, Sk_b - 1) */
    int n_per_block;             /* the key tile nPerBlock of the partition (>= 1) */
    int split_kv;                /* 0: automatic (sk_auto_split_kv); else 1..32 */
    int block_m;                 /* query rows per M block of the partition; 0: default */
    float softmax_scale;         /* 0: 1/sqrt(d_qk) */
    int fuse_combine;            /* sk_attn_fwd only, 0 or 1: 1 lets the tensor-core partial
                                    kernel merge the splits itself (the last CTA of each M
                                    block), instead of the separate combine; 0 (default)
                                    keeps the combine kernel, which measured faster */
    int window_left;             /* -1: no sliding window; else (causal / prefix-causal masks
                                    only) key j is visible to query q only if
                                    j >= q + prefix_offset - window_left ([P2] Technical
                                    details: the forced split honours the caller's window) */
    const int32_t *seqused_k;    /* device int32 [B] or NULL: padded key slots -- sequence b
                                    uses only its first seqused_k[b] keys; the rest of its
                                    cu_seqlens / max_seqlen slot is padding ([P2] Technical
                                    details: padded cu_seqlens) */
} sk_params;

/* Largest split_kv accepted. */
#define SK_MAX_SPLIT_KV 32

/*
 * sk_valid_split_counts -- [P1] Technical details, per-row valid-split counts
 * (computeValidSplitKV). For packed query row r at position q of sequence b:
 *   rowLast      = clamp(q + prefix_offset, 0, lastValid)   (causal / prefix-causal)
 *                = lastValid                                 (no mask)
 *   keysPerSplit = n_per_block * ceil(ceil((rowLast + 1) / n_per_block) / S)
 *   counts[r]    = ceil((rowLast + 1) / keysPerSplit)
 * A sequence without keys gets count 1. S is split_kv after resolving 0 (auto).
 * counts: device int32 [total_q]. Exact integer arithmetic.
 */
sk_status sk_valid_split_counts(const sk_params *p, int32_t *counts, sk_stream stream);

/*
 * sk_attn_partial_fwd -- [P1] Summary and Technical details; [P2] Technical details.
 * For every (sequence, head, M block of block_m query rows, split s) the block's keys
 * 0..blockLast (blockLast = rowLast of the block's last row) are cut into key tiles of
 * n_per_block and dealt out in runs of itersPerBlock = ceil(tiles / S); split s gets
 * run s. Over the keys of its run that row q may see:
 *   O_s = sum_j softmax(scale * q.k_j) v_j        L_s = log sum_j exp(scale * q.k_j)
 * A row with no visible key in the split gets O_s = 0 and L_s = -inf ([P1]: the
 * kernel writes zero output and -inf LSE for empty splits).
 * q, k, v: storage bf16 / f16 / f32, all the same dtype.
 * o_part: device f32 [H][S][total_q][d_v]; lse_part: device f32 [H][S][total_q].
 */
sk_status sk_attn_partial_fwd(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v,
                              float *o_part, float *lse_part, sk_stream stream);

/*
 * sk_combine -- [P1] Technical details, NaN-safe merge (computeFinalAttentionStage)
 * and f32 merge for f16/bf16. Per (head, row), over the splits s < counts[row] that the
 * partition of the row's M block leaves non-empty (the others are never read: [P1]
 * review notes allow a split with nothing to do to write nothing; such a split would
 * contribute exactly 0):
 *   m = max(max_s L_s, lowest finite f32);  w_s = exp(L_s - m)
 *   O = sum_s w_s O_s / max(sum_s w_s, 1)   (in f32, then cast to out.dtype)
 *   lse_out = m + log(sum_s w_s), or -inf when that sum is 0
 * out: [rows, H, d_v] or dense, dtype = storage type; lse_out may be NULL ([P2]
 * review: return_lse=False passes a null LSE to the combine).
 */
sk_status sk_combine(const sk_params *p, const float *o_part, const float *lse_part,
                     const int32_t *counts, sk_tensor out, float *lse_out, sk_stream stream);

/*
 * sk_attn_fwd -- the whole forward pass in one call: partials, then the merge with
 * the per-row counts. With S == 1 the partial kernel writes `out` and `lse_out`
 * directly and no workspace is used. With S > 1, `workspace` (device, 256-byte
 * aligned, at least sk_workspace_bytes()) holds the split partials; the combine
 * evaluates the per-row count formula itself, and splits that hold no key of their
 * M block write nothing (a real early exit) and are not read. max_seqlen_k == 0 writes
 * O = 0 and LSE = -inf ([P2] review: forced split with empty K must not raise;
 * [P1]: an empty split's LSE is -inf). lse_out may be NULL.
 */
sk_status sk_attn_fwd(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v, sk_tensor out,
                      float *lse_out, void *workspace, size_t workspace_bytes, sk_stream stream);

/* Bytes of scratch that sk_attn_fwd_static keeps inside the library (32 MiB). */
#define SK_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * sk_attn_fwd_static -- sk_attn_fwd for callers that cannot allocate device memory.
 * The pages have no counterpart: this call exists for users of this library whose
 * device memory is planned once up front (a serving loop that must not allocate per
 * request) or whose host framework owns every allocation and gives a plugin no
 * allocator, so they cannot hand sk_attn_fwd a workspace. It computes exactly what
 * sk_attn_fwd computes, with the workspace taken from a file-scope device array of
 * SK_STATIC_SCRATCH_BYTES that every GPU loading the library holds until exit.
 *   - The caller still passes Q, K, V, out and (optionally) lse_out.
 *   - Problems whose sk_workspace_bytes() exceeds SK_STATIC_SCRATCH_BYTES are
 *     rejected with SK_ERR_WORKSPACE before anything is launched.
 *   - It calls no cudaMalloc / cudaFree and no allocating library routine.
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and keeps it; make that first call before any stream capture.
 *     A lookup that fails is not kept: the call returns SK_ERR_CUDA (the error is in
 *     sk_last_cuda_error) and the next call tries again.
 *   - The kept address belongs to the device's current context: do not call this
 *     entry point again after cudaDeviceReset (or anything else that destroys and
 *     recreates the context) in the same process.
 *   - Every call on a device shares the one array and leaves its contents behind;
 *     nothing in it has to start at zero (each call writes what it later reads).
 *     Calls that overlap on the GPU (other streams, other threads) race on it.
 */
sk_status sk_attn_fwd_static(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v,
                             sk_tensor out, float *lse_out, sk_stream stream);

/*
 * sk_attn_fwd_host -- sk_attn_fwd with Q, K, V and the output in HOST memory, for callers whose
 * data lives on the host (the one-call form of the pages' varlen API, with the copies inside).
 *   - q, k, v, out: host pointers to contiguous tensors, [total, H, d] packed (stride_row =
 *     H * d, stride_h = d) or [B, seq, H, d] dense (stride_b = seq * H * d); any other
 *     strides return SK_ERR_UNSUPPORTED. All four have the same storage type.
 *   - lse_out: host float [H][total_q], or NULL.
 *   - cu_seqlens_q / cu_seqlens_k / seqused_k in p stay DEVICE pointers, as in every call.
 *   - device_buffer: caller-owned device memory, 256-byte aligned, at least
 *     sk_host_buffer_bytes() (SK_ERR_WORKSPACE otherwise): it holds device copies of Q, K,
 *     V, the output and the LSE, then sk_attn_fwd's workspace.
 * Enqueued on `stream`, in order: the host-to-device copies of q, k, v, sk_attn_fwd on the
 * device copies, the device-to-host copies of out (and lse_out). The call returns without
 * waiting; the host output is complete once the stream has passed this point. With page-
 * locked (pinned) host memory every copy is asynchronous; pageable host memory works, but
 * its copies may return only once staged. Two calls on two streams with two device buffers
 * overlap one call's copies with the other's compute. Nothing is allocated.
 */
sk_status sk_attn_fwd_host(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v,
                           sk_tensor out, float *lse_out, void *device_buffer,
                           size_t device_bytes, sk_stream stream);

/* Bytes of device memory sk_attn_fwd_host needs for these parameters, storage type and
 * whether an LSE is returned (with_lse 0 or 1). */
sk_status sk_host_buffer_bytes(const sk_params *p, sk_dtype dtype, int with_lse, size_t *bytes);

/* Bytes of workspace sk_attn_fwd needs for these parameters (0 when S == 1).
 * Resolving split_kv = 0 reads the current device's SM count. */
sk_status sk_workspace_bytes(const sk_params *p, size_t *bytes);

/*
 * sk_auto_split_kv -- [P2] Technical details: num_splits 0 is auto, 1 keeps the
 * unsplit kernel, 2..8 (here 2..32) force that split. Auto uses 3 splits when
 * max_seqlen_k >= 8192 (an explicit boundary, as the review asks) and
 * ceil(max_seqlen_q / block_m) * H <= 2 * SM count; otherwise 1. For single-query
 * problems (max_seqlen_q == 1) it takes the smallest S <= 32 with B * H * S >= 2 * SM
 * count. Under a sliding window (causal / prefix-causal masks) the result is 1 when the
 * deepest query, max_seqlen_q - 1 + prefix_offset, sees no key of split 0 of that S: the
 * partition has no window term, so the leading splits would only write empty partials.
 * A non-zero split_kv is returned unchanged. Reads the current device.
 */
sk_status sk_auto_split_kv(const sk_params *p, int *split_kv_out);

/* Host-only form of sk_auto_split_kv with the SM count given. */
sk_status sk_choose_split_kv(const sk_params *p, int sm_count, int *split_kv_out);

/* The M block (block_m = 0) the library uses for these head dims and dtype: 256. */
int sk_default_block_m(int d_qk, int d_v, sk_dtype dtype);

/* Whether (d_qk, d_v) is one of the supported head-dimension pairs. */
int sk_supported_head_dims(int d_qk, int d_v);

/* Name of the kernel sk_attn_partial_fwd would launch for these parameters, for
 * logging and benchmarks: "partial_tc" (tensor cores, one unit per CTA),
 * "partial_tc_persist" (tensor cores, one CTA per SM taking many short units in turn),
 * "partial_decode" (CUDA cores, few queries per sequence) or "partial_fma" (CUDA cores,
 * f32 and the remaining cases); NULL when the call would be rejected. split_kv = 0 is
 * resolved as sk_auto_split_kv resolves it (reading the current device). The string is
 * static; the caller does not free it. */
const char *sk_partial_kernel_name(const sk_params *p, sk_tensor q, sk_tensor k, sk_tensor v);

/* Human-readable text of a status code. */
const char *sk_status_string(sk_status s);

/* The CUDA error (a cudaError_t value) behind the most recent SK_ERR_CUDA returned
 * on the calling thread, 0 if there was none; *name (optional) receives its name. */
int sk_last_cuda_error(const char **name);

/* Self-test of the give-up path of the kernels' bounded waits: launches one CTA that
 * waits, through the same helper, on a barrier nothing arrives on, with a limit of
 * timeout_ns (at most 2e9); the wait runs out, the CTA records code 0x401 in the device
 * error word and returns. Read it with sk_read_device_error (SK_ERR_TIMEOUT). Larger
 * limits return SK_ERR_INVALID_ARG without a launch. */
sk_status sk_selftest_bounded_wait(unsigned long long timeout_ns, sk_stream stream);

/* Debug: reads (and optionally clears) the device error word that bounded waits
 * set when they give up. SYNCHRONISES the current device. *code = 0: no error. */
sk_status sk_read_device_error(int *code, int clear);

/* Library version: major * 10000 + minor * 100 + patch. */
int sk_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPLITKV_H */
