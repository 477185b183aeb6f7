// combine.cu -- NaN-safe f32 merge of split partials ([P1] Technical details:
// NaN-safe merge (computeFinalAttentionStage), f32 merge for f16/bf16).
//
// One warp merges one (head, query row). Lane s < count holds L_s; a warp max and
// sum give m and sum_s w_s; then every partial row O_s (d_v f32, contiguous) is read
// once with 16-byte loads, weighted and summed. Splits s >= count are never read.
// The pass is HBM-bound: it reads count * (4 d_v + 4) bytes and writes d_v
// storage-type elements (+ 4 bytes of LSE) per (head, row).
#include <float.h>

#include "sk_common.cuh"

namespace sk {

constexpr int kCombineWarps = 8;

template <typename TO, int DV>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(Problem p, const float *__restrict__ o_part, const float *__restrict__ lse_part,
                   const int32_t *__restrict__ counts, TensorView out, float *__restrict__ lse_out,
                   int row_blocks) {
    static_assert(DV % 4 == 0 && DV / 4 <= 32, "one float4 per lane");
    constexpr int kLanes = DV / 4;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int h = blockIdx.y;
    const int b = blockIdx.x / row_blocks;
    const int pos = (blockIdx.x % row_blocks) * kCombineWarps + warp;
    const SeqInfo si = seq_info(p, b);
    if (pos >= si.sq) return;
    const int row = si.q0 + pos;
    const int S = p.S;

    int count = __ldg(counts + row);
    count = count < 1 ? 1 : (count > S ? S : count);

    // m = max(max_s L_s, lowest finite); w_s = exp(L_s - m)
    const float *lrow = lse_part + (int64_t)h * S * p.total_q + row;
    float l = lane < count ? __ldg(lrow + (int64_t)lane * p.total_q) : -INFINITY;
    float m = fmaxf(group_max<32>(l), -FLT_MAX);
    float w = lane < count ? expf(l - m) : 0.f;
    float wsum = group_sum<32>(w);

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float *orow = o_part + ((int64_t)h * S * p.total_q + row) * DV + lane * 4;
    const int64_t split_stride = (int64_t)p.total_q * DV;
    int s = 0;
    for (; s + 4 <= count; s += 4) {  // four independent 16-byte loads in flight
        float4 o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            o[u] = lane < kLanes ? __ldg((const float4 *)(orow + (s + u) * split_stride))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float ws = __shfl_sync(0xffffffffu, w, s + u);
            acc.x = fmaf(ws, o[u].x, acc.x);
            acc.y = fmaf(ws, o[u].y, acc.y);
            acc.z = fmaf(ws, o[u].z, acc.z);
            acc.w = fmaf(ws, o[u].w, acc.w);
        }
    }
    for (; s < count; ++s) {
        float4 o = lane < kLanes ? __ldg((const float4 *)(orow + s * split_stride))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        float ws = __shfl_sync(0xffffffffu, w, s);
        acc.x = fmaf(ws, o.x, acc.x);
        acc.y = fmaf(ws, o.y, acc.y);
        acc.z = fmaf(ws, o.z, acc.z);
        acc.w = fmaf(ws, o.w, acc.w);
    }
    const float denom = fmaxf(wsum, 1.f);  // only binds when every split is empty

    if (lane < kLanes) {
        TO *dst = (TO *)out.ptr + row_offset(p, out, b, si.q0, pos) + (int64_t)h * out.sh + lane * 4;
        if constexpr (sizeof(TO) == 4) {
            *(float4 *)dst = make_float4(acc.x / denom, acc.y / denom, acc.z / denom, acc.w / denom);
        } else {
            TO v[4] = {from_f32<TO>(acc.x / denom), from_f32<TO>(acc.y / denom),
                       from_f32<TO>(acc.z / denom), from_f32<TO>(acc.w / denom)};
            *(uint2 *)dst = *(const uint2 *)v;
        }
    }
    if (lse_out && lane == 0)
        lse_out[(int64_t)h * p.total_q + row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

template <typename TO>
static cudaError_t launch_dv(const Problem &p, const float *o_part, const float *lse_part,
                             const int32_t *counts, const TensorView &out, float *lse_out,
                             cudaStream_t st) {
    const int row_blocks = (p.max_sq + kCombineWarps - 1) / kCombineWarps;
    dim3 grid((unsigned)((long long)row_blocks * p.B), (unsigned)p.H);
    if (p.d_v == 128)
        combine_kernel<TO, 128><<<grid, kCombineWarps * 32, 0, st>>>(p, o_part, lse_part, counts,
                                                                      out, lse_out, row_blocks);
    else if (p.d_v == 64)
        combine_kernel<TO, 64><<<grid, kCombineWarps * 32, 0, st>>>(p, o_part, lse_part, counts,
                                                                     out, lse_out, row_blocks);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_combine(const Problem &p, int dtype, const float *o_part,
                           const float *lse_part, const int32_t *counts, const TensorView &out,
                           float *lse_out, cudaStream_t st) {
    if (p.total_q == 0 || p.max_sq == 0) return cudaSuccess;
    switch (dtype) {
    case kBF16: return launch_dv<__nv_bfloat16>(p, o_part, lse_part, counts, out, lse_out, st);
    case kF16: return launch_dv<__half>(p, o_part, lse_part, counts, out, lse_out, st);
    default: return launch_dv<float>(p, o_part, lse_part, counts, out, lse_out, st);
    }
}

}  // namespace sk
