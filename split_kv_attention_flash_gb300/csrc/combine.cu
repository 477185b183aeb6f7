// combine.cu -- NaN-safe f32 merge of split partials ([P1] Technical details:
// NaN-safe merge (computeFinalAttentionStage), f32 merge for f16/bf16).
//
// Per (head, row), over the splits s < count that the row's block partition leaves
// non-empty (the others are never read; an empty split contributes exactly 0):
//   m = max(max_s L_s, lowest finite);  w_s = exp(L_s - m)
//   O = sum_s w_s O_s / max(sum_s w_s, 1);   LSE = m + log(sum_s w_s)  (or -inf)
//
// The pass is HBM-bound: it reads count * (4 d_v + 4) bytes and writes d_v
// storage-type elements (+ 4 bytes of LSE) per (head, row).
//
// combine_bulk_kernel: a CTA merges ROWS consecutive packed rows of one head, whichever
// sequences they belong to: 16 rows for up to 8 splits, 8 for up to 16, 4 for up to 32, so
// that the staged partials take at most 64 KB of shared memory. For a (head, split) plane
// those rows are one contiguous chunk of ROWS * d_v floats, so one thread first issues one
// bulk asynchronous copy per split into shared memory, before any load the copies would
// depend on; warp 0 loads each row's log-sum-exps and finds its sequence, count and weights
// while they land; then every warp merges its rows out of shared memory.
#include <float.h>

#include <mutex>

#include "sk_common.cuh"
#include "sm100_ptx.cuh"

namespace sk {

// Launch with programmatic stream serialization: the combine's CTAs may be scheduled while
// the partial kernel before it in the stream is finishing (it issues launch_dependents at
// its start), and every combine kernel waits in wait_prior_grid before reading a partial.
template <typename... Params, typename... Args>
static cudaError_t launch_after_prior(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

namespace {
constexpr int kBulkThreads = 128;
// Up to 8 splits: 16 packed rows per CTA (measured: 8 rows / 64 threads and 32 rows / 256
// threads no faster, 32 rows / 128 threads slower); more splits take fewer rows, so that the
// staged partials stay within 64 KB.
constexpr uint64_t kBulkTimeoutNs = 1000000000ull;
}  // namespace

// Sequence holding packed query row `row`: the last b with cu_q[b] <= row (binary search;
// bad cu_seqlens give a wrong b in [0, B), never an index outside cu_q), or row / max_sq in
// the dense layout. Sets *pos to the row's position in that sequence.
__device__ inline int seq_of_row(const Problem &p, int row, int *pos) {
    if (!p.cu_q) {
        const int b = row / p.max_sq;
        *pos = row - b * p.max_sq;
        return b;
    }
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.cu_q + mid) <= row) lo = mid;
        else hi = mid - 1;
    }
    *pos = row - __ldg(p.cu_q + lo);
    return lo;
}

// A CTA merges 16 consecutive packed rows of one head, whichever sequences they belong
// to. The rows of a (head, split) plane are contiguous, so the first thread issues the S
// bulk copies before anything else is known; meanwhile warp 0 (one lane per row) loads
// the row's S log-sum-exps, finds its sequence, count and weights. Splits that the
// partition leaves empty are copied but never read (their memory may be unwritten).
template <typename TO, int DV, int kBulkRows, int kBulkMaxSplits>
__global__ void __launch_bounds__(kBulkThreads)
    combine_bulk_kernel(Problem p, const float *__restrict__ o_part,
                        const float *__restrict__ lse_part, const int32_t *__restrict__ counts,
                        TensorView out, float *__restrict__ lse_out) {
    static_assert(DV % 4 == 0 && DV / 4 <= 32, "one float4 per lane");
    constexpr int kLanes = DV / 4;
    constexpr int kRowsPerWarp = kBulkRows / (kBulkThreads / 32);
    static_assert(kBulkRows % (kBulkThreads / 32) == 0 && kBulkRows <= 32, "rows per CTA");
    extern __shared__ __align__(128) uint8_t sO_raw[];   // [split][kBulkRows rows][DV] f32
    __shared__ __align__(8) uint64_t sBar;
    __shared__ float sW[kBulkMaxSplits][kBulkRows];
    __shared__ float sInv[kBulkRows];
    __shared__ int sCnt[kBulkRows];
    __shared__ long long sOff[kBulkRows];   // element offset of the row in `out`; -1: none
    __shared__ volatile int sAbort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.y;
    const int r0 = blockIdx.x * kBulkRows;
    const int nrows = min(kBulkRows, p.total_q - r0);
    const int S = p.S;
    const int64_t plane = p.total_q;
    const uint32_t bar = ptx::smem_u32(&sBar);
    const float *sO = (const float *)sO_raw;
    if (tid == 0) {
        sAbort = 0;
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    ptx::wait_prior_grid();  // launched early (programmatic serialization): partials complete

    if (tid == 0) {
        const uint32_t chunk = (uint32_t)nrows * DV * 4;
        ptx::mbar_arrive_expect_tx(bar, chunk * (uint32_t)S);
        for (int sp = 0; sp < S; ++sp)
            ptx::bulk_load(ptx::smem_u32(sO_raw) + (uint32_t)sp * kBulkRows * DV * 4,
                           o_part + (((int64_t)h * S + sp) * plane + r0) * DV, chunk, bar);
    }
    if (warp == 0 && lane < kBulkRows) {
        const int r = lane;
        const bool row_in = r < nrows;
        // the row's L_s first (in bounds for every s < S; only s < count are used)
        const float *lrow = lse_part + (int64_t)h * S * plane + r0 + r;
        float l[kBulkMaxSplits];
#pragma unroll
        for (int sp = 0; sp < kBulkMaxSplits; ++sp)
            l[sp] = (row_in && sp < S) ? __ldg(lrow + sp * plane) : -INFINITY;
        int c = 0;
        long long off = -1;
        if (row_in) {
            int pos = 0;
            const int b = seq_of_row(p, r0 + r, &pos);
            const SeqInfo si = seq_info(p, b);
            if (pos >= 0 && pos < si.sq) {  // else a row outside every sequence: not written
                c = merged_splits(p, si.sq, si.last_valid, pos, row_count(p, si, counts, pos));
                off = row_offset(p, out, b, si.q0, pos);
            }
        }
        sCnt[r] = c;
        sOff[r] = off;
        // m = max(max_s L_s, lowest finite), w_s = exp(L_s - m) over s < count
        float m = -FLT_MAX;
#pragma unroll
        for (int sp = 0; sp < kBulkMaxSplits; ++sp)
            if (sp < c) m = fmaxf(m, l[sp]);
        float wsum = 0.f;
#pragma unroll
        for (int sp = 0; sp < kBulkMaxSplits; ++sp) {
            const float w = sp < c ? expf(l[sp] - m) : 0.f;
            sW[sp][r] = w;
            wsum += w;
        }
        sInv[r] = 1.f / fmaxf(wsum, 1.f);  // the max only binds when every split is empty
        if (lse_out && off >= 0)
            lse_out[(int64_t)h * plane + r0 + r] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
    }
    __syncthreads();
    if (!ptx::mbar_wait_bounded(bar, 0, &sAbort, p.err, 0x301, kBulkTimeoutNs)) return;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int r = warp * kRowsPerWarp + i;
        if (r >= nrows) break;  // warp-uniform
        const long long off = sOff[r];
        if (off < 0) continue;  // warp-uniform
        const int c = sCnt[r];
        if (lane < kLanes) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sp = 0; sp < c; ++sp) {
                const float4 o = *(const float4 *)(sO + ((size_t)sp * kBulkRows + r) * DV + lane * 4);
                const float w = sW[sp][r];
                acc.x = fmaf(w, o.x, acc.x);
                acc.y = fmaf(w, o.y, acc.y);
                acc.z = fmaf(w, o.z, acc.z);
                acc.w = fmaf(w, o.w, acc.w);
            }
            const float inv = sInv[r];
            TO *dst = (TO *)out.ptr + off + (int64_t)h * out.sh + lane * 4;
            if constexpr (sizeof(TO) == 4) {
                *(float4 *)dst = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            } else {
                TO v[4] = {from_f32<TO>(acc.x * inv), from_f32<TO>(acc.y * inv),
                           from_f32<TO>(acc.z * inv), from_f32<TO>(acc.w * inv)};
                *(uint2 *)dst = *(const uint2 *)v;
            }
        }
    }
}

template <typename TO, int DV, int ROWS, int MAXS>
static cudaError_t launch_bulk(const Problem &p, const float *o_part, const float *lse_part,
                               const int32_t *counts, const TensorView &out, float *lse_out,
                               cudaStream_t st) {
    auto kern = combine_bulk_kernel<TO, DV, ROWS, MAXS>;
    constexpr int kMaxSmem = MAXS * ROWS * DV * 4;
    static_assert(kMaxSmem <= 64 * 1024, "staged partials");
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    const int row_blocks = (p.total_q + ROWS - 1) / ROWS;
    const int smem = p.S * ROWS * DV * 4;
    return launch_after_prior(kern, dim3((unsigned)row_blocks, (unsigned)p.H), dim3(kBulkThreads),
                              (size_t)smem, st, p, o_part, lse_part, counts, out, lse_out);
}

template <typename TO, int DV>
static cudaError_t launch_splits(const Problem &p, const float *o_part, const float *lse_part,
                                 const int32_t *counts, const TensorView &out, float *lse_out,
                                 cudaStream_t st) {
    if (p.S <= 8) return launch_bulk<TO, DV, 16, 8>(p, o_part, lse_part, counts, out, lse_out, st);
    if (p.S <= 16) return launch_bulk<TO, DV, 8, 16>(p, o_part, lse_part, counts, out, lse_out, st);
    if (p.S <= 32) return launch_bulk<TO, DV, 4, 32>(p, o_part, lse_part, counts, out, lse_out, st);
    return cudaErrorInvalidValue;
}

template <typename TO>
static cudaError_t launch_dv(const Problem &p, const float *o_part, const float *lse_part,
                             const int32_t *counts, const TensorView &out, float *lse_out,
                             cudaStream_t st) {
    if (p.d_v == 128) return launch_splits<TO, 128>(p, o_part, lse_part, counts, out, lse_out, st);
    if (p.d_v == 64) return launch_splits<TO, 64>(p, o_part, lse_part, counts, out, lse_out, st);
    return cudaErrorInvalidValue;
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
