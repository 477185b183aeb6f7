// sk_common.cuh -- problem description and index arithmetic shared by the kernels.
//
// Page tags used in comments across csrc/:
//   [P1] "Recombine fully masked split-KV attention partials on the host"
//   [P2] "[ASM] [HIP] [JIT] [gfx942] Optimize long-context FMHA with split-KV"
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sk {

// Storage types (same numbering as sk_dtype in include/splitkv.h).
enum : int { kBF16 = 0, kF16 = 1, kF32 = 2 };

// The validated problem, passed to every kernel by value.
struct Problem {
    int B, H, max_sq, max_sk, total_q, total_k, d_qk, d_v;
    const int32_t *cu_q, *cu_k;  // device; both null for the dense layout
    int causal;                  // 1 under causal or prefix-causal masking
    int prefix_offset;           // 0 for plain causal
    int last_valid_kv_index;     // -1: each sequence's last key
    int bn;                      // key tile n_per_block
    int S;                       // resolved split count
    int bm;                      // M block rows of the partition
    float scale;                 // softmax scale
    float scale_log2;            // scale * log2(e): scores are kept in base 2
    int *err;                    // device error word (bounded waits), may be null
    int skip_empty;              // 1: split CTAs with no key exit without writing (sk_attn_fwd)
    int counts_inline;           // 1: the combine evaluates the count formula itself (sk_attn_fwd)
    int window_left;             // -1: none; else keys before q + offset - window_left are hidden
    const int32_t *seqused_k;    // device; null, or keys used per sequence (padded slots)
};

// A [rows, heads, dim] view with element strides (dense layout adds stride_b).
struct TensorView {
    char *ptr;
    int64_t sb, sr, sh;  // element strides
};

// Where sequence b lives, clamped so that bad cu_seqlens cannot index outside
// [0, total) nor past max_seqlen.
struct SeqInfo {
    int q0, sq;        // first packed query row, query count
    int k0, sk;        // first packed key row, key count
    int last_valid;    // last key any query may see; -1 when there is none
};

__host__ __device__ inline int clamp_len(long long start, long long len, long long max_len,
                                         long long total) {
    if (len > max_len) len = max_len;
    if (start < 0 || start >= total) return 0;
    if (start + len > total) len = total - start;
    return len < 0 ? 0 : (int)len;
}

__device__ inline SeqInfo seq_info(const Problem &p, int b) {
    SeqInfo s;
    long long q0, q1, k0, k1;
    if (p.cu_q) {
        q0 = __ldg(p.cu_q + b); q1 = __ldg(p.cu_q + b + 1);
        k0 = __ldg(p.cu_k + b); k1 = __ldg(p.cu_k + b + 1);
    } else {
        q0 = (long long)b * p.max_sq; q1 = q0 + p.max_sq;
        k0 = (long long)b * p.max_sk; k1 = k0 + p.max_sk;
    }
    s.q0 = (int)q0;
    s.k0 = (int)k0;
    s.sq = clamp_len(q0, q1 - q0, p.max_sq, p.total_q);
    s.sk = clamp_len(k0, k1 - k0, p.max_sk, p.total_k);
    if (p.seqused_k) {  // padded slot: only the first seqused_k[b] keys belong to the sequence
        const int used = __ldg(p.seqused_k + b);
        if (used < s.sk) s.sk = used < 0 ? 0 : used;
    }
    int last = s.sk - 1;
    if (p.last_valid_kv_index >= 0 && p.last_valid_kv_index < last) last = p.last_valid_kv_index;
    s.last_valid = last;
    return s;
}

// Element offset of row `pos` of sequence b in a tensor view.
__device__ inline int64_t row_offset(const Problem &p, const TensorView &t, int b, int start,
                                     int pos) {
    return p.cu_q ? (int64_t)(start + pos) * t.sr : (int64_t)b * t.sb + (int64_t)pos * t.sr;
}

// Last key the partition must cover for `row` ([P1] Technical details):
// clamp(row + prefix_offset, 0, lastValid) under causal masks, lastValid otherwise;
// -1 when the sequence has no key.
__host__ __device__ inline long long covered_last(const Problem &p, int last_valid, long long row) {
    if (last_valid < 0) return -1;
    if (!p.causal) return last_valid;
    long long x = row + p.prefix_offset;
    if (x < 0) x = 0;
    if (x > last_valid) x = last_valid;
    return x;
}

// [P1] per-row valid-split count (computeValidSplitKV).
// ceil(a / b) for b >= 1 in 32-bit unsigned arithmetic (a - 1 avoids the overflow of
// a + b - 1); the quantities below stay under 2^32: n <= 2^31 and bn * tiles < n + bn.
__host__ __device__ inline uint32_t ceil_div_u32(uint32_t a, uint32_t b) {
    return a == 0 ? 0u : (a - 1u) / b + 1u;
}
__host__ __device__ inline int valid_split_count(const Problem &p, int last_valid, int pos) {
    long long rl = covered_last(p, last_valid, pos);
    if (rl < 0) return 1;
    const uint32_t n = (uint32_t)rl + 1u;
    const uint32_t tiles = ceil_div_u32(n, (uint32_t)p.bn);
    const uint32_t kps = (uint32_t)p.bn * ceil_div_u32(tiles, (uint32_t)p.S);
    return (int)ceil_div_u32(n, kps);
}

// Keys [kb, ke) of split s for the M block that holds query `pos` ([P1]: the kernel
// partitions each M block's keys by the block's last row, in runs of
// itersPerBlock = ceil(tiles / S) key tiles).
__host__ __device__ inline void split_key_range(const Problem &p, int sq, int last_valid, int pos,
                                                int s, int &kb, int &ke) {
    long long first = (long long)(pos / p.bm) * p.bm;
    long long last_row = first + p.bm - 1;
    if (last_row > sq - 1) last_row = sq - 1;
    long long bl = covered_last(p, last_valid, last_row);
    kb = ke = 0;
    if (bl < 0) return;
    const long long nt = (uint32_t)bl / (uint32_t)p.bn + 1u;
    const long long it = ceil_div_u32((uint32_t)nt, (uint32_t)p.S);
    long long t0 = (long long)s * it, t1 = t0 + it;
    if (t1 > nt) t1 = nt;
    if (t0 >= t1) return;
    kb = (int)(t0 * p.bn);
    long long e = t1 * p.bn;
    ke = (int)(e < bl + 1 ? e : bl + 1);
}

// Longest-first launch order. The CTAs of a (sequence, split) unit all stream that
// split's keys; with sequences of very different lengths, launching the units in
// index order can leave the longest ones for the last wave. lpt_unit returns the unit
// of rank r when the n units are sorted by their key count, largest first (ties by
// index), so that a CTA's rank in the hardware's launch order picks its unit. Every
// thread of the CTA calls it; `keys` is shared memory for n ints, `found` one int.
constexpr int kLptMaxUnits = 256;
__device__ inline int unit_keys(const Problem &p, int u) {
    const int b = u / p.S, s = u % p.S;
    const SeqInfo si = seq_info(p, b);
    if (si.sq <= 0) return -1;
    int kb, ke;
    split_key_range(p, si.sq, si.last_valid, ((si.sq - 1) / p.bm) * p.bm, s, kb, ke);
    return ke > kb ? ke - kb : 0;
}
__device__ inline int lpt_unit(const Problem &p, int r, int n, int *keys, int *found) {
    for (int u = threadIdx.x; u < n; u += blockDim.x) keys[u] = unit_keys(p, u);
    __syncthreads();
    for (int u = threadIdx.x; u < n; u += blockDim.x) {
        const int ku = keys[u];
        int rank = 0;
        for (int v = 0; v < n; ++v) {
            const int kv = keys[v];
            rank += (kv > ku) | ((kv == ku) & (v < u));
        }
        if (rank == r) *found = u;
    }
    __syncthreads();
    const int u = *found;
    __syncthreads();  // the scratch may be reused from here on
    return u;
}

// Splits that the partition of the M block holding query `pos` leaves non-empty: the
// first ceil(tiles / itersPerBlock) of them. The merge never reads the others ([P1]
// review notes on a real early exit: a split with nothing to do may write nothing,
// so the merge must not assume its memory was written).
__host__ __device__ inline int nonempty_splits(const Problem &p, int sq, int last_valid, int pos) {
    long long first = (long long)(pos / p.bm) * p.bm;
    long long last_row = first + p.bm - 1;
    if (last_row > sq - 1) last_row = sq - 1;
    long long bl = covered_last(p, last_valid, last_row);
    if (bl < 0) return 0;
    const uint32_t nt = (uint32_t)bl / (uint32_t)p.bn + 1u;
    const uint32_t it = ceil_div_u32(nt, (uint32_t)p.S);
    return (int)ceil_div_u32(nt, it);
}

// Splits the merge reads for query `pos`: min(count, non-empty splits of its block).
__device__ inline int merged_splits(const Problem &p, int sq, int last_valid, int pos, int count) {
    int c = count < 1 ? 1 : (count > p.S ? p.S : count);
    const int ne = nonempty_splits(p, sq, last_valid, pos);
    return c < ne ? c : ne;
}

// The count of packed row q0 + pos: the caller's array, or the formula itself.
__device__ inline int row_count(const Problem &p, const SeqInfo &si, const int32_t *counts, int pos) {
    return p.counts_inline ? valid_split_count(p, si.last_valid, pos) : __ldg(counts + si.q0 + pos);
}

// Last key query `pos` may see, ignoring the split: lastValid, and q + offset
// under a causal mask. Negative when the row sees nothing.
__device__ inline long long row_limit(const Problem &p, int last_valid, int pos) {
    long long lim = last_valid;
    if (p.causal) {
        long long c = (long long)pos + p.prefix_offset;
        if (c < lim) lim = c;
    }
    return lim;
}

// First key query `pos` may see under a sliding window (0 without one).
__device__ inline long long row_start(const Problem &p, int pos) {
    if (!p.causal || p.window_left < 0) return 0;
    const long long x = (long long)pos + p.prefix_offset - p.window_left;
    return x < 0 ? 0 : x;
}

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) {
    return __float2half_rn(x);
}

// Warp reductions over groups of W consecutive lanes (W a power of two <= 32).
template <int W> __device__ __forceinline__ float group_max(float x) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
template <int W> __device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace sk

// Launchers implemented in the .cu files (host side).
namespace sk {
cudaError_t launch_counts(const Problem &p, int32_t *counts, cudaStream_t st);
cudaError_t launch_partial_fma(const Problem &p, int dtype, const TensorView &q,
                               const TensorView &k, const TensorView &v, float *o_part,
                               float *lse_part, const TensorView *out, float *lse_out,
                               cudaStream_t st);
namespace tc {
bool partial_tc_supported(const Problem &p, int dtype);
cudaError_t launch_partial_tc(const Problem &p, int dtype, const TensorView &q, const TensorView &k,
                              const TensorView &v, float *o_part, float *lse_part,
                              const TensorView *out, float *lse_out, int *tickets, cudaStream_t st,
                              bool *launched);
// The persistent form (partial_tc_persist.cu): whether it takes the launch, and the launch
// with the tensor maps already made (out: split 1, the output written directly).
bool persist_fits(const Problem &p, int sm_count);
bool persist_selected(const Problem &p);  // persist_fits with the current device's SM count
cudaError_t launch_partial_tc_persist(const Problem &p, int dtype, const CUtensorMap &mq,
                                      const CUtensorMap &mk, const CUtensorMap &mv, float *o_part,
                                      float *lse_part, const TensorView *out, float *lse_out,
                                      int sm_count, cudaStream_t st);
// TMA map of a [rows, H, D] (varlen) or [B][rows][H][D] (dense) 16-bit tensor: boxes of
// 64 elements x box_rows rows, 128-byte swizzle. False when TMA cannot describe it.
bool make_map(CUtensorMap *m, const TensorView &t, int dtype, int D, long long rows, int H, int B,
              bool dense, unsigned box_rows);
}  // namespace tc
namespace dec {
bool partial_decode_supported(const Problem &p, int dtype);
cudaError_t launch_partial_decode(const Problem &p, int dtype, const TensorView &q,
                                  const TensorView &k, const TensorView &v, float *o_part,
                                  float *lse_part, const TensorView *out, float *lse_out,
                                  cudaStream_t st, bool *launched);
}  // namespace dec
cudaError_t launch_selftest_wait(int *err, unsigned long long timeout_ns, cudaStream_t st);
cudaError_t launch_combine(const Problem &p, int dtype, const float *o_part,
                           const float *lse_part, const int32_t *counts, const TensorView &out,
                           float *lse_out, cudaStream_t st);
}  // namespace sk
