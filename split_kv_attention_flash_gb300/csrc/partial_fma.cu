// partial_fma.cu -- split partials on the CUDA cores: f32 storage (tf32 tensor-core MMAs
// cannot meet its 1e-5 bound), and every case the tensor-core kernels do not take.
//
// [P1] Summary / Technical details: for each (sequence, head, M block, split) the kernel
// computes, over the keys of the split's run that the row may see,
//   O_s = sum_j softmax(scale q.k_j) v_j,   L_s = log sum_j exp(scale q.k_j),
// and an empty split writes O_s = 0, L_s = -inf. Scores are kept in base 2 (scale * log2 e
// folded in); the online softmax keeps a running max m, a running sum l and an
// unnormalised accumulator, all in f32.
//
// Layout of a CTA (512 threads): 128 query rows of one (sequence, head, split); keys in tiles
// of 64. Thread (ty, tx) of the 32 x 16 grid owns rows 4 ty .. 4 ty + 3, and
//   * scores of keys 4 tx .. 4 tx + 3 (a 4 x 4 block of S = Q K^T),
//   * output columns 4 tx + 64 c .. + 3 (c < D_V / 64) of its rows.
// Q and each K tile sit in shared memory transposed ([d][row], [d][key]) and P transposed
// ([key][row]), so that every operand of the inner loops is one 16-byte load: 16 FMAs per
// two loads for S, 4 * D_V / 16 FMAs per 1 + D_V / 64 loads for P V. A row's max and sum are
// reduced over the 16 threads that share it (one half-warp).
#include <climits>
#include <float.h>

#include <mutex>

#include "sk_common.cuh"
#include "sm100_ptx.cuh"

namespace sk {
namespace fma {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 64;           // keys per tile
constexpr int kThreads = 512;     // 32 (rows / 4) x 16 (keys / 4)
constexpr int kPad = 4;           // floats of padding per transposed row

template <int DQK, int DV> struct FCfg {
    static constexpr int kQS = kBM + kPad;  // sQt[d][kQS]
    static constexpr int kKS = kBN + kPad;  // sKt[d][kKS]
    static constexpr int kPS = kBM + kPad;  // sPt[key][kPS]
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + DQK * kQS;
    static constexpr int kVOff = kKOff + DQK * kKS;  // sV[key][DV]
    static constexpr int kPOff = kVOff + kBN * DV;
    static constexpr size_t kSmemBytes = (size_t)(kPOff + kBN * kPS) * 4;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(DV % 64 == 0 && DQK % 8 == 0, "head dims");
};

// Loads `rows` rows x D elements of a [row][d] tensor slice (rows at `base`, `sr` elements
// apart) as f32; element (r, d) goes to dst[d * ld + r] (transposed) or dst[r * ld + d].
// Rows at or past `valid` read as zero. 16 bytes per load.
template <typename T, int D, bool TRANSPOSE>
__device__ __forceinline__ void load_tile(float *dst, int ld, const T *base, int64_t sr, int rows,
                                          int valid) {
    constexpr int kVec = 16 / (int)sizeof(T);
    constexpr int kChunks = D / kVec;
    for (int e = threadIdx.x; e < rows * kChunks; e += kThreads) {
        int r, c;
        if constexpr (TRANSPOSE) {  // a warp covers consecutive rows: conflict-free stores
            r = e % rows;
            c = e / rows;
        } else {                    // a warp covers consecutive chunks of a row: coalesced loads
            r = e / kChunks;
            c = e % kChunks;
        }
        float x[kVec];
        if (r < valid) {
            const uint4 raw = *(const uint4 *)(base + (int64_t)r * sr + c * kVec);
            const T *t = (const T *)&raw;
#pragma unroll
            for (int i = 0; i < kVec; ++i) x[i] = to_f32(t[i]);
        } else {
#pragma unroll
            for (int i = 0; i < kVec; ++i) x[i] = 0.f;
        }
        if constexpr (TRANSPOSE) {
#pragma unroll
            for (int i = 0; i < kVec; ++i) dst[(c * kVec + i) * ld + r] = x[i];
        } else {
#pragma unroll
            for (int i = 0; i < kVec; i += 4)
                *(float4 *)&dst[r * ld + c * kVec + i] = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
        }
    }
}

template <typename T, int DQK, int DV, bool DIRECT>
__global__ void __launch_bounds__(kThreads, 1)
    partial_fma_kernel(Problem p, TensorView q, TensorView k, TensorView v, float *o_part,
                       float *lse_part, TensorView out, float *lse_out, int row_blocks) {
    using C = FCfg<DQK, DV>;
    constexpr int kCols = DV / 64;  // float4 column groups per thread
    extern __shared__ __align__(16) float smem[];
    float *sQt = smem + C::kQOff, *sKt = smem + C::kKOff, *sV = smem + C::kVOff, *sPt = smem + C::kPOff;
    __shared__ int sRange[2];
    __shared__ int sAnyKeys;
    ptx::launch_dependents();  // the combine may be scheduled onto SMs this grid leaves idle

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int h = blockIdx.y;
    const int rb = blockIdx.x % row_blocks;
    const int bs = blockIdx.x / row_blocks;
    const int s = bs % p.S, b = bs / p.S;
    const SeqInfo si = seq_info(p, b);
    const int pos0 = rb * kBM;
    if (pos0 >= si.sq) return;  // whole CTA past the sequence end

    // the keys [kb, ke) each of this thread's four rows may see in the split
    int kb[4], ke[4];
    bool any_keys = false;  // the partition gives some row of this thread keys in the split
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int pos = pos0 + 4 * ty + i;
        kb[i] = ke[i] = 0;
        if (pos < si.sq) {
            split_key_range(p, si.sq, si.last_valid, pos, s, kb[i], ke[i]);
            any_keys |= ke[i] > kb[i];
            const long long lim = row_limit(p, si.last_valid, pos);
            if (lim + 1 < ke[i]) ke[i] = (int)(lim + 1 > kb[i] ? lim + 1 : kb[i]);
            const long long first = row_start(p, pos);  // sliding window
            if (first > kb[i]) kb[i] = (int)(first < ke[i] ? first : ke[i]);
        }
    }
    if (tid == 0) {
        sRange[0] = INT_MAX;
        sRange[1] = 0;
        sAnyKeys = 0;
    }
    // Q, widened and transposed, while the range is being reduced
    const T *qbase = (const T *)q.ptr + row_offset(p, q, b, si.q0, pos0) + (int64_t)h * q.sh;
    load_tile<T, DQK, true>(sQt, C::kQS, qbase, q.sr, kBM, si.sq - pos0);
    __syncthreads();
    if (tx == 0) {
        int lo = INT_MAX, hi = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (ke[i] > kb[i]) {
                lo = min(lo, kb[i]);
                hi = max(hi, ke[i]);
            }
        if (hi > lo) {
            atomicMin(&sRange[0], lo);
            atomicMax(&sRange[1], hi);
        }
        if (any_keys) sAnyKeys = 1;
    }
    __syncthreads();
    const int t_begin = sRange[0], t_end = sRange[1];
    // real early exit: the partition gives no row of this CTA a key in the split, so the
    // merge never reads it (rows whose keys are all masked still write 0 / -inf)
    if (!DIRECT && p.skip_empty && !sAnyKeys) return;

    float m[4], l[4], acc[4][4 * kCols];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < 4 * kCols; ++c) acc[i][c] = 0.f;
    }
    const T *kbase = (const T *)k.ptr + row_offset(p, k, b, si.k0, 0) + (int64_t)h * k.sh;
    const T *vbase = (const T *)v.ptr + row_offset(p, v, b, si.k0, 0) + (int64_t)h * v.sh;
    const int key_end = min(t_end, si.sk);  // keys at or past it read as zero

    for (int t0 = t_begin; t0 < t_end; t0 += kBN) {
        __syncthreads();  // the previous tile's K, V and P are fully consumed
        load_tile<T, DQK, true>(sKt, C::kKS, kbase + (int64_t)t0 * k.sr, k.sr, kBN, key_end - t0);
        load_tile<T, DV, false>(sV, DV, vbase + (int64_t)t0 * v.sr, v.sr, kBN, key_end - t0);
        __syncthreads();

        // S: a 4 x 4 block per thread
        float sc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) sc[i][j] = 0.f;
#pragma unroll 8
        for (int d = 0; d < DQK; ++d) {
            const float4 a = *(const float4 *)&sQt[d * C::kQS + 4 * ty];
            const float4 kk = *(const float4 *)&sKt[d * C::kKS + 4 * tx];
            const float av[4] = {a.x, a.y, a.z, a.w}, kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) sc[i][j] = fmaf(av[i], kv[j], sc[i][j]);
        }
        // masks, online softmax (rows that have seen no key yet keep m = -inf and p = 0)
        float pr[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int key = t0 + 4 * tx + j;
                sc[i][j] = (key >= kb[i] && key < ke[i]) ? sc[i][j] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, sc[i][j]);
            }
            mx = group_max<16>(mx);
            const float m_new = fmaxf(m[i], mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = exp2f(m[i] - m_use);
            m[i] = m_new;
            l[i] *= alpha;
#pragma unroll
            for (int c = 0; c < 4 * kCols; ++c) acc[i][c] *= alpha;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pr[i][j] = exp2f(sc[i][j] - m_use);
                l[i] += pr[i][j];
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *(float4 *)&sPt[(4 * tx + j) * C::kPS + 4 * ty] = make_float4(pr[0][j], pr[1][j], pr[2][j], pr[3][j]);
        __syncthreads();

        // O += P V
#pragma unroll 4
        for (int kk = 0; kk < kBN; ++kk) {
            const float4 pv = *(const float4 *)&sPt[kk * C::kPS + 4 * ty];
            const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                const float4 vv = *(const float4 *)&sV[kk * DV + 4 * tx + 64 * c];
                const float va[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) acc[i][4 * c + jj] = fmaf(pa[i], va[jj], acc[i][4 * c + jj]);
            }
        }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lsum = group_sum<16>(l[i]);
        const int pos = pos0 + 4 * ty + i;
        if (pos >= si.sq) continue;
        const bool empty = !(lsum > 0.f);
        const float inv = empty ? 0.f : 1.f / lsum;
        const float lse = empty ? -INFINITY : (m[i] + log2f(lsum)) * 0.69314718055994530942f;
        const int row = si.q0 + pos;
        if constexpr (DIRECT) {
            T *dst = (T *)out.ptr + row_offset(p, out, b, si.q0, pos) + (int64_t)h * out.sh;
#pragma unroll
            for (int c = 0; c < kCols; ++c) {
                T w[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) w[jj] = from_f32<T>(acc[i][4 * c + jj] * inv);
                if constexpr (sizeof(T) == 4) *(float4 *)&dst[4 * tx + 64 * c] = *(const float4 *)w;
                else *(uint2 *)&dst[4 * tx + 64 * c] = *(const uint2 *)w;
            }
            if (lse_out && tx == 0) lse_out[(int64_t)h * p.total_q + row] = lse;
        } else {
            const int64_t slot = ((int64_t)h * p.S + s) * p.total_q + row;
            float *dst = o_part + slot * DV;
#pragma unroll
            for (int c = 0; c < kCols; ++c)
                *(float4 *)&dst[4 * tx + 64 * c] = make_float4(acc[i][4 * c] * inv, acc[i][4 * c + 1] * inv,
                                                               acc[i][4 * c + 2] * inv, acc[i][4 * c + 3] * inv);
            if (tx == 0) lse_part[slot] = lse;
        }
    }
}

template <typename T, int DQK, int DV, bool DIRECT>
static cudaError_t launch_cfg(const Problem &p, const TensorView &q, const TensorView &k,
                              const TensorView &v, float *o_part, float *lse_part,
                              const TensorView &out, float *lse_out, dim3 grid, int row_blocks,
                              cudaStream_t st) {
    using C = FCfg<DQK, DV>;
    auto kern = partial_fma_kernel<T, DQK, DV, DIRECT>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmemBytes);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    kern<<<grid, kThreads, C::kSmemBytes, st>>>(p, q, k, v, o_part, lse_part, out, lse_out, row_blocks);
    return cudaGetLastError();
}

template <typename T, int DQK, int DV>
static cudaError_t launch_t(const Problem &p, const TensorView &q, const TensorView &k,
                            const TensorView &v, float *o_part, float *lse_part,
                            const TensorView *out, float *lse_out, cudaStream_t st) {
    const int row_blocks = (p.max_sq + kBM - 1) / kBM;
    const long long nx = (long long)row_blocks * p.B * p.S;
    if (nx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)nx, (unsigned)p.H);
    if (out)
        return launch_cfg<T, DQK, DV, true>(p, q, k, v, o_part, lse_part, *out, lse_out, grid, row_blocks, st);
    return launch_cfg<T, DQK, DV, false>(p, q, k, v, o_part, lse_part, TensorView{nullptr, 0, 0, 0},
                                         nullptr, grid, row_blocks, st);
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

}  // namespace fma

cudaError_t launch_partial_fma(const Problem &p, int dtype, const TensorView &q,
                               const TensorView &k, const TensorView &v, float *o_part,
                               float *lse_part, const TensorView *out, float *lse_out,
                               cudaStream_t st) {
    if (p.total_q == 0 || p.max_sq == 0) return cudaSuccess;
    switch (dtype) {
    case kBF16: return fma::launch_dims<__nv_bfloat16>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    case kF16: return fma::launch_dims<__half>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    default: return fma::launch_dims<float>(p, q, k, v, o_part, lse_part, out, lse_out, st);
    }
}

}  // namespace sk
