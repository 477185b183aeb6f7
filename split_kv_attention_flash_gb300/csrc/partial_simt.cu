// partial_simt.cu -- split partials on the CUDA cores (f32 storage, and any case the
// tensor-core kernel does not take).
//
// [P1] Summary / Technical details: for each (sequence, head, M block, split) the
// kernel computes, over the keys of the split's run that the row may see,
//   O_s = sum_j softmax(scale q.k_j) v_j,   L_s = log sum_j exp(scale q.k_j),
// and an empty split writes O_s = 0, L_s = -inf. Scores are kept in base 2
// (scale * log2 e folded into the dot product) and the online softmax keeps a
// running max m, a running sum l and an unnormalised accumulator.
//
// Layout of a CTA (128 threads): 16 query rows of one (sequence, head, split),
// 8 threads per row. A tile of 16 keys (K and V, widened to f32) is staged in shared
// memory; thread c of row r scores keys c and c+8, and accumulates output columns
// c, c+8, c+16, ... Rows of the CTA may belong to different M blocks, so each row
// keeps its own key range and the CTA walks the union of them.
#include <climits>
#include <float.h>

#include "sk_common.cuh"
#include "sm100_ptx.cuh"

namespace sk {

namespace {
constexpr int kRows = 16;      // query rows per CTA
constexpr int kTpr = 8;        // threads per row
constexpr int kKT = 16;        // keys per tile
constexpr int kThreads = kRows * kTpr;
}  // namespace

template <typename T, int DQK, int DV, bool DIRECT>
__global__ void __launch_bounds__(kThreads)
    partial_simt_kernel(Problem p, TensorView q, TensorView k, TensorView v, float *o_part,
                        float *lse_part, TensorView out, float *lse_out, int row_blocks) {
    __shared__ float sQ[kRows][DQK + 1];
    __shared__ float sK[kKT][DQK + 1];
    __shared__ float sV[kKT][DV];
    __shared__ float sP[kRows][kKT + 1];
    __shared__ int sRange[2];
    ptx::launch_dependents();  // the combine may be scheduled onto SMs this grid leaves idle

    const int tid = threadIdx.x;
    const int r = tid / kTpr, c = tid % kTpr;
    const int h = blockIdx.y;
    const int rb = blockIdx.x % row_blocks;
    const int bs = blockIdx.x / row_blocks;
    const int s = bs % p.S, b = bs / p.S;
    const SeqInfo si = seq_info(p, b);
    const int pos0 = rb * kRows;
    if (pos0 >= si.sq) return;  // whole CTA past the sequence end
    const int pos = pos0 + r;
    const bool row_ok = pos < si.sq;

    // this row's keys: [kb, min(ke, lim + 1))
    int kb = 0, ke = 0;
    if (row_ok) {
        split_key_range(p, si.sq, si.last_valid, pos, s, kb, ke);
        long long lim = row_limit(p, si.last_valid, pos);
        if (lim + 1 < ke) ke = (int)(lim + 1 > kb ? lim + 1 : kb);
        const long long first = row_start(p, pos);  // sliding window
        if (first > kb) kb = (int)(first < ke ? first : ke);
    }
    if (tid == 0) { sRange[0] = INT_MAX; sRange[1] = 0; }
    // stage Q (widened) while the range is being reduced
    for (int e = tid; e < kRows * DQK; e += kThreads) {
        int rr = e / DQK, d = e % DQK;
        float x = 0.f;
        if (pos0 + rr < si.sq)
            x = to_f32(((const T *)q.ptr)[row_offset(p, q, b, si.q0, pos0 + rr) + (int64_t)h * q.sh + d]);
        sQ[rr][d] = x;
    }
    __syncthreads();
    if (c == 0 && ke > kb) {
        atomicMin(&sRange[0], kb);
        atomicMax(&sRange[1], ke);
    }
    __syncthreads();
    const int t_begin = sRange[0], t_end = sRange[1];
    // real early exit: no row of this CTA has a key in the split (the merge never reads it)
    if (!DIRECT && p.skip_empty && t_begin >= t_end) {
        bool all_empty = true;
        for (int rr = 0; rr < kRows && all_empty; ++rr) {
            if (pos0 + rr >= si.sq) break;
            int rkb, rke;
            split_key_range(p, si.sq, si.last_valid, pos0 + rr, s, rkb, rke);
            all_empty = rke <= rkb;
        }
        if (all_empty) return;
    }

    float m = -INFINITY;    // running max, base-2 scaled scores
    float l = 0.f;          // this thread's share of the running sum
    float acc[DV / kTpr];
#pragma unroll
    for (int i = 0; i < DV / kTpr; ++i) acc[i] = 0.f;

    for (int t0 = t_begin; t0 < t_end; t0 += kKT) {
        __syncthreads();  // previous tile fully consumed
        for (int e = tid; e < kKT * DQK; e += kThreads) {
            int kk = e / DQK, d = e % DQK, j = t0 + kk;
            float x = 0.f;
            if (j < si.sk)
                x = to_f32(((const T *)k.ptr)[row_offset(p, k, b, si.k0, j) + (int64_t)h * k.sh + d]);
            sK[kk][d] = x;
        }
        for (int e = tid; e < kKT * DV; e += kThreads) {
            int kk = e / DV, d = e % DV, j = t0 + kk;
            float x = 0.f;
            if (j < si.sk)
                x = to_f32(((const T *)v.ptr)[row_offset(p, v, b, si.k0, j) + (int64_t)h * v.sh + d]);
            sV[kk][d] = x;
        }
        __syncthreads();

        float sc[kKT / kTpr];
        float tmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < kKT / kTpr; ++u) {
            const int kk = c + u * kTpr, j = t0 + kk;
            float dot = 0.f;
#pragma unroll 8
            for (int d = 0; d < DQK; ++d) dot = fmaf(sQ[r][d], sK[kk][d], dot);
            sc[u] = (j >= kb && j < ke) ? dot * p.scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, sc[u]);
        }
        tmax = group_max<kTpr>(tmax);
        const float m_new = fmaxf(m, tmax);
        // rows that have seen no key yet keep m = -inf and p = 0
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = exp2f(m - m_use);
        m = m_new;
        l *= alpha;
#pragma unroll
        for (int i = 0; i < DV / kTpr; ++i) acc[i] *= alpha;
#pragma unroll
        for (int u = 0; u < kKT / kTpr; ++u) {
            float pr = exp2f(sc[u] - m_use);
            l += pr;
            sP[r][c + u * kTpr] = pr;
        }
        __syncwarp();
#pragma unroll 4
        for (int kk = 0; kk < kKT; ++kk) {
            const float pr = sP[r][kk];
#pragma unroll
            for (int i = 0; i < DV / kTpr; ++i) acc[i] = fmaf(pr, sV[kk][c + i * kTpr], acc[i]);
        }
    }

    l = group_sum<kTpr>(l);
    if (!row_ok) return;
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
    const float lse = empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
    const int row = si.q0 + pos;
    if constexpr (DIRECT) {
        T *dst = (T *)out.ptr + row_offset(p, out, b, si.q0, pos) + (int64_t)h * out.sh;
#pragma unroll
        for (int i = 0; i < DV / kTpr; ++i) dst[c + i * kTpr] = from_f32<T>(acc[i] * inv);
        if (lse_out && c == 0) lse_out[(int64_t)h * p.total_q + row] = lse;
    } else {
        const int64_t slot = ((int64_t)h * p.S + s) * p.total_q + row;
        float *dst = o_part + slot * DV;
#pragma unroll
        for (int i = 0; i < DV / kTpr; ++i) dst[c + i * kTpr] = acc[i] * inv;
        if (c == 0) lse_part[slot] = lse;
    }
}

template <typename T, int DQK, int DV>
static cudaError_t launch_t(const Problem &p, const TensorView &q, const TensorView &k,
                            const TensorView &v, float *o_part, float *lse_part,
                            const TensorView *out, float *lse_out, cudaStream_t st) {
    const int row_blocks = (p.max_sq + kRows - 1) / kRows;
    const long long nx = (long long)row_blocks * p.B * p.S;
    if (nx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)nx, (unsigned)p.H);
    TensorView o = out ? *out : TensorView{nullptr, 0, 0, 0};
    if (out)
        partial_simt_kernel<T, DQK, DV, true><<<grid, kThreads, 0, st>>>(p, q, k, v, o_part, lse_part,
                                                                        o, lse_out, row_blocks);
    else
        partial_simt_kernel<T, DQK, DV, false><<<grid, kThreads, 0, st>>>(p, q, k, v, o_part, lse_part,
                                                                         o, lse_out, row_blocks);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_dims(const Problem &p, const TensorView &q, const TensorView &k,
                               const TensorView &v, float *o_part, float *lse_part,
                               const TensorView *out, float *lse_out, cudaStream_t st) {
    if (p.d_qk == 64 && p.d_v == 64)
        return launch_t<T, 64, 64>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    if (p.d_qk == 128 && p.d_v == 128)
        return launch_t<T, 128, 128>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    if (p.d_qk == 192 && p.d_v == 128)
        return launch_t<T, 192, 128>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_partial_simt(const Problem &p, int dtype, const TensorView &q,
                                const TensorView &k, const TensorView &v, float *o_part,
                                float *lse_part, const TensorView *out, float *lse_out,
                                cudaStream_t st) {
    if (p.total_q == 0 || p.max_sq == 0) return cudaSuccess;
    switch (dtype) {
    case kBF16: return launch_dims<__nv_bfloat16>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    case kF16: return launch_dims<__half>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    default: return launch_dims<float>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    }
}

}  // namespace sk
