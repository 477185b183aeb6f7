// partial_decode.cu -- split partials for sequences of up to 16 queries (decode) where the
// tensor-core kernel does not apply: an M block other than its 256 rows, more than 65535
// (sequence, split) units, or tensors its TMA maps cannot describe; bf16 / f16 storage.
//
// [P1] Summary / Technical details: O_s and L_s of one (sequence, head, split) over
// the split's key run, empty splits giving O_s = 0 and L_s = -inf. With a handful
// of queries per sequence the work is a stream over K and V (2 (D_QK + D_V) bytes
// per key for up to 16 dot products each), bound by HBM bandwidth, so it runs on
// the CUDA cores:
//   * warp 8 streams 64-key tiles of K and V into a 3-stage shared-memory ring
//     with TMA (128-byte swizzle, so per-key reads below are bank-conflict free);
//   * warps 0-7 own 8 keys of every tile each: four lanes split a key's dot
//     product over D_QK, each warp keeps its own running max / sum / accumulator
//     per query (lane l owns output columns l*DV/32 ..), and the eight partial
//     states are merged through shared memory at the end.
// Scores are kept in base 2 (q pre-multiplied by scale * log2 e).
#include <float.h>

#include <mutex>
#include <type_traits>

#include "sk_common.cuh"
#include "sm100_ptx.cuh"

namespace sk {
namespace dec {

constexpr int kKT = 64;            // keys per tile
constexpr int kStages = 3;
constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kMaxRows = 16;
constexpr uint64_t kTimeoutNs = 1000000000ull;
enum ErrCode : int { kErrProducer = 0x201, kErrConsumer = 0x202 };

template <int DQK, int DV> struct Cfg {
    static constexpr int kKBytes = kKT * DQK * 2;
    static constexpr int kVBytes = kKT * DV * 2;
    static constexpr int kStageBytes = kKBytes + kVBytes;
    static constexpr int kQFloats = kMaxRows * DQK;
    static constexpr int kMergeFloats = kComputeWarps * kMaxRows * (DV + 2);
    static_assert(kStages * kStageBytes >= kMergeFloats * 4, "merge area fits in the ring");
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kQFloats * 4 + 2 * kStages * 8 + 16;
    static constexpr int kDPer = DQK / 4;   // dot-product elements per lane
    static constexpr int kVPer = DV / 32;   // output columns per lane
};

// Element (row, col) of a tile stored as 64-column panels of `rows` rows, each row
// 128 bytes with 16-byte chunks swizzled by row % 8 (the TMA 128-byte pattern).
__device__ __forceinline__ uint32_t swz(int row, int col, int rows) {
    const int panel = col >> 6, c = col & 63;
    return (uint32_t)(panel * rows * 128 + row * 128 + ((((c >> 3) ^ (row & 7)) << 4) | ((c & 7) << 1)));
}

template <typename T>
__device__ __forceinline__ void widen8(uint4 u, float (&f)[8]) {
    const T *h = reinterpret_cast<const T *>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = to_f32(h[i]);
}

// Up to 4 query rows the kernel fits two CTAs per SM (registers <= 112).
template <typename T, int DQK, int DV, bool DIRECT, int NR>
__global__ void __launch_bounds__(kThreads, NR <= 4 ? 2 : 1)
    partial_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          Problem p, TensorView q, float *o_part, float *lse_part, TensorView out,
                          float *lse_out) {
    using C = Cfg<DQK, DV>;
    extern __shared__ uint8_t smem_raw[];
    ptx::launch_dependents();  // the combine may be scheduled onto SMs this grid leaves idle
    // CTA i of the launch order (x fastest) takes head i % H of the unit of rank i / H
    // in longest-first order (the ring's memory serves as scratch before any load)
    int h = blockIdx.y, unit = blockIdx.x;
    if (gridDim.x > 1 && gridDim.x <= kLptMaxUnits) {
        const int i = blockIdx.x + blockIdx.y * gridDim.x;
        h = i % p.H;
        int *scratch = (int *)smem_raw;
        unit = lpt_unit(p, i / p.H, gridDim.x, scratch, scratch + kLptMaxUnits);
    }
    const int s = unit % p.S, b = unit / p.S;
    const SeqInfo si = seq_info(p, b);
    // NR (a power of two >= every sequence's query count) rows are computed; rows at or
    // past this sequence's count are masked out and never stored
    const int R = si.sq < NR ? si.sq : NR;
    if (R <= 0) return;
    int kb, ke;
    split_key_range(p, si.sq, si.last_valid, 0, s, kb, ke);
    int n_tiles = ke > kb ? (ke - kb + kKT - 1) / kKT : 0;
    if (!DIRECT && n_tiles == 0 && p.skip_empty) return;  // real early exit: nothing is read
    {
        // sliding window: skip key tiles before row 0's window (the earliest of all rows)
        const long long first = row_start(p, 0);
        if (first > kb) {
            int skip = (int)((first - kb) / kKT);
            if (skip > n_tiles) skip = n_tiles;
            kb += skip * kKT;
            n_tiles -= skip;
        }
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    const uint32_t ring = (raw_u32 + 1023u) & ~1023u;
    uint8_t *const gring = smem_raw + (ring - raw_u32);
    float *const sq = (float *)(gring + kStages * C::kStageBytes);
    const uint32_t bar0 = ring + kStages * C::kStageBytes + C::kQFloats * 4;
    volatile int *const abort_flag = (volatile int *)(gring + (bar0 - ring) + 2 * kStages * 8);
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kStages + i); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(full(i), 1);
            ptx::mbar_init(empty(i), kComputeWarps);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    // queries, widened and pre-scaled into base-2 score units
    for (int e = threadIdx.x; e < NR * DQK; e += kThreads) {
        const int r = e / DQK, d = e % DQK;
        float x = 0.f;
        if (r < R)
            x = to_f32(((const T *)q.ptr)[row_offset(p, q, b, si.q0, r) + (int64_t)h * q.sh + d]);
        sq[r * DQK + d] = x * p.scale_log2;
    }
    __syncthreads();

    const bool dense = p.cu_q == nullptr;
    const int cb = dense ? b : 0;
    if (warp == kComputeWarps) {
        // --------------------------------------------------------------- producer
        if (lane == 0) {
            const int krow = (dense ? 0 : si.k0) + kb;
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % kStages;
                ok = ptx::mbar_wait_bounded(empty(st), ((j / kStages) & 1) ^ 1, abort_flag, p.err,
                                            kErrProducer, kTimeoutNs);
                if (!ok) break;
                const uint32_t dst = ring + st * C::kStageBytes;
                ptx::mbar_arrive_expect_tx(full(st), C::kStageBytes);
                for (int c = 0; c < DQK / 64; ++c)
                    ptx::tma_load_4d(dst + c * kKT * 128, &tmK, full(st), c * 64, krow + j * kKT, h, cb);
                for (int c = 0; c < DV / 64; ++c)
                    ptx::tma_load_4d(dst + C::kKBytes + c * kKT * 128, &tmV, full(st), c * 64,
                                     krow + j * kKT, h, cb);
                issued = j + 1;
            }
            if (!ok) {
                int quiet = 0;
                for (int i = 0; i < kStages && i < issued; ++i) {
                    const int last = i + ((issued - 1 - i) / kStages) * kStages;
                    ptx::mbar_wait_bounded(full(i), (last / kStages) & 1, (volatile int *)&quiet,
                                           nullptr, 0, kTimeoutNs);
                }
            }
        }
        __syncthreads();  // merge area is reused below: wait until compute warps are done
        __syncthreads();
        return;
    }

    // ------------------------------------------------------------------ compute
    const int kl = lane >> 2;          // key of the warp's 8 in this tile
    const int dq = lane & 3;           // quarter of the dot product
    int kend[NR];
    long long kfirst[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) kfirst[r] = row_start(p, r);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        int e = kb;  // rows past the sequence see nothing
        if (r < R) {
            e = ke;
            const long long lim = row_limit(p, si.last_valid, r);
            if (lim + 1 < e) e = (int)(lim + 1 > kb ? lim + 1 : kb);
        }
        kend[r] = e;
    }
    float m[NR], l[NR], acc[NR][C::kVPer];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int i = 0; i < C::kVPer; ++i) acc[r][i] = 0.f;
    }

    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
        const int st = j % kStages;
        // whole-warp bounded wait
        uint64_t t0 = 0;
        for (uint32_t it = 0;; ++it) {
            bool done = ptx::mbar_try_wait(full(st), (j / kStages) & 1);
            if (__all_sync(0xffffffffu, done)) break;
            if ((it & 63u) == 63u) {
                int give = 0;
                if (lane == 0) {
                    if (t0 == 0) t0 = ptx::globaltimer();
                    if (*abort_flag) give = 1;
                    else if (ptx::globaltimer() - t0 > kTimeoutNs) {
                        *abort_flag = 1;
                        if (p.err) atomicCAS(p.err, 0, kErrConsumer);
                        give = 1;
                    }
                }
                if (__shfl_sync(0xffffffffu, give, 0)) { ok = false; break; }
            }
        }
        if (!ok) break;
        const uint8_t *kt = gring + st * C::kStageBytes;
        const uint8_t *vt = kt + C::kKBytes;
        const int key = warp * 8 + kl;                // row of the tile
        const int kidx = kb + j * kKT + key;           // key index in the sequence

        // scores of this lane's key for every query (quarter dot + 2 shuffles)
        float sc[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) sc[r] = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < C::kDPer / 8; ++c8) {
            const int d0 = dq * C::kDPer + c8 * 8;
            float kf[8];
            widen8<T>(*(const uint4 *)(kt + swz(key, d0, kKT)), kf);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float4 qa = *(const float4 *)(sq + r * DQK + d0);
                const float4 qb = *(const float4 *)(sq + r * DQK + d0 + 4);
                sc[r] = fmaf(qa.x, kf[0], sc[r]); sc[r] = fmaf(qa.y, kf[1], sc[r]);
                sc[r] = fmaf(qa.z, kf[2], sc[r]); sc[r] = fmaf(qa.w, kf[3], sc[r]);
                sc[r] = fmaf(qb.x, kf[4], sc[r]); sc[r] = fmaf(qb.y, kf[5], sc[r]);
                sc[r] = fmaf(qb.z, kf[6], sc[r]); sc[r] = fmaf(qb.w, kf[7], sc[r]);
            }
        }
        float pr[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float x = sc[r];
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            x = (kidx < kend[r] && kidx >= kfirst[r]) ? x : -INFINITY;
            float tmax = x;
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
            const float m_new = fmaxf(m[r], tmax);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = ptx::ex2(m[r] - m_use);
            m[r] = m_new;
            const float pv = ptx::ex2(x - m_use);
            float ps = pv;
            ps += __shfl_xor_sync(0xffffffffu, ps, 4);
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            l[r] = l[r] * alpha + ps;
#pragma unroll
            for (int i = 0; i < C::kVPer; ++i) acc[r][i] *= alpha;
            pr[r] = pv;
        }
        // P V: lane owns columns lane*kVPer .. ; p of key k lives in lane 4k
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
            const int vrow = warp * 8 + k8;
            float vf[C::kVPer];
            const int col = lane * C::kVPer;
            if constexpr (C::kVPer == 4) {
                const uint2 u = *(const uint2 *)(vt + swz(vrow, col, kKT));
                const T *hh = reinterpret_cast<const T *>(&u);
#pragma unroll
                for (int i = 0; i < 4; ++i) vf[i] = to_f32(hh[i]);
            } else {
                const uint32_t u = *(const uint32_t *)(vt + swz(vrow, col, kKT));
                const T *hh = reinterpret_cast<const T *>(&u);
#pragma unroll
                for (int i = 0; i < C::kVPer; ++i) vf[i] = to_f32(hh[i]);
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float pk = __shfl_sync(0xffffffffu, pr[r], 4 * k8);
#pragma unroll
                for (int i = 0; i < C::kVPer; ++i) acc[r][i] = fmaf(pk, vf[i], acc[r][i]);
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty(st));
    }

    // ------------------------------------------------------- merge of the 8 warps
    __syncthreads();  // (1) every warp left the loop; the ring is free
    float *mm = (float *)gring;                  // [8][NR] max
    float *ll = mm + kComputeWarps * NR;         // [8][NR] sum
    float *aa = ll + kComputeWarps * NR;         // [8][NR][DV]
    if (ok) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            if (r >= R) continue;
            if (lane == 0) {
                mm[warp * NR + r] = m[r];
                ll[warp * NR + r] = l[r];
            }
#pragma unroll
            for (int i = 0; i < C::kVPer; ++i)
                aa[(warp * NR + r) * DV + lane * C::kVPer + i] = acc[r][i];
        }
    }
    __syncthreads();  // (2)
    if (!ok || *abort_flag) return;
    for (int e = threadIdx.x; e < R * DV; e += kComputeWarps * 32) {
        const int r = e / DV, d = e % DV;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, mm[w * NR + r]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) {
            const float f = ptx::ex2(mm[w * NR + r] - Mu);
            L = fmaf(ll[w * NR + r], f, L);
            O = fmaf(aa[(w * NR + r) * DV + d], f, O);
        }
        const bool emp = !(L > 0.f);
        const float o = emp ? 0.f : O / L;
        const float lse = emp ? -INFINITY : (M + log2f(L)) * 0.69314718055994530942f;
        const int row = si.q0 + r;
        if constexpr (DIRECT) {
            T *dst = (T *)out.ptr + row_offset(p, out, b, si.q0, r) + (int64_t)h * out.sh + d;
            *dst = from_f32<T>(o);
            if (d == 0 && lse_out) lse_out[(int64_t)h * p.total_q + row] = lse;
        } else {
            const int64_t slot = ((int64_t)h * p.S + s) * p.total_q + row;
            o_part[slot * DV + d] = o;
            if (d == 0) lse_part[slot] = lse;
        }
    }
}

// ------------------------------------------------------------------------ host
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)f;
        else
            (void)cudaGetLastError();
    });
    return fn;
}

static bool make_map(CUtensorMap *m, const TensorView &t, int dtype, int D, long long rows, int H,
                     int B, bool dense) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows <= 0 || t.sr <= 0 || t.sh <= 0 || (dense && t.sb <= 0)) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)(dense ? B : 1)};
    cuuint64_t strides[3] = {(cuuint64_t)t.sr * 2, (cuuint64_t)t.sh * 2,
                             (cuuint64_t)(dense ? t.sb : rows * t.sr) * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)kKT, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
               t.ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int DQK, int DV, bool DIRECT, int NR>
static cudaError_t launch_rows(const Problem &p, const CUtensorMap &mk, const CUtensorMap &mv,
                               const TensorView &q, float *o_part, float *lse_part,
                               const TensorView &out, float *lse_out, cudaStream_t st) {
    using C = Cfg<DQK, DV>;
    auto kern = partial_decode_kernel<T, DQK, DV, DIRECT, NR>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    dim3 grid((unsigned)(p.B * p.S), (unsigned)p.H);
    kern<<<grid, kThreads, C::kSmemBytes, st>>>(mk, mv, p, q, o_part, lse_part, out, lse_out);
    return cudaGetLastError();
}

template <typename T, int DQK, int DV, bool DIRECT>
static cudaError_t launch_cfg(const Problem &p, const CUtensorMap &mk, const CUtensorMap &mv,
                              const TensorView &q, float *o_part, float *lse_part,
                              const TensorView &out, float *lse_out, cudaStream_t st) {
    if (p.max_sq <= 1) return launch_rows<T, DQK, DV, DIRECT, 1>(p, mk, mv, q, o_part, lse_part, out, lse_out, st);
    if (p.max_sq <= 2) return launch_rows<T, DQK, DV, DIRECT, 2>(p, mk, mv, q, o_part, lse_part, out, lse_out, st);
    if (p.max_sq <= 4) return launch_rows<T, DQK, DV, DIRECT, 4>(p, mk, mv, q, o_part, lse_part, out, lse_out, st);
    if (p.max_sq <= 8) return launch_rows<T, DQK, DV, DIRECT, 8>(p, mk, mv, q, o_part, lse_part, out, lse_out, st);
    return launch_rows<T, DQK, DV, DIRECT, 16>(p, mk, mv, q, o_part, lse_part, out, lse_out, st);
}

template <typename T, int DQK, int DV>
static cudaError_t launch_dims(const Problem &p, const CUtensorMap &mk, const CUtensorMap &mv,
                               const TensorView &q, float *o_part, float *lse_part,
                               const TensorView *out, float *lse_out, cudaStream_t st) {
    if (out) return launch_cfg<T, DQK, DV, true>(p, mk, mv, q, o_part, lse_part, *out, lse_out, st);
    return launch_cfg<T, DQK, DV, false>(p, mk, mv, q, o_part, lse_part, TensorView{}, nullptr, st);
}

bool partial_decode_supported(const Problem &p, int dtype) {
    if (dtype != kBF16 && dtype != kF16) return false;
    if (!((p.d_qk == 64 && p.d_v == 64) || (p.d_qk == 128 && p.d_v == 128) ||
          (p.d_qk == 192 && p.d_v == 128)))
        return false;
    if (p.max_sq > kMaxRows || p.max_sq < 1 || p.bm < p.max_sq) return false;
    if (p.total_k <= 0 || p.max_sk <= 0 || p.total_q <= 0) return false;
    if ((long long)p.B * p.S > 0x7fffffffLL || p.H > 65535) return false;
    return encode_fn() != nullptr;
}

cudaError_t launch_partial_decode(const Problem &p, int dtype, const TensorView &q,
                                  const TensorView &k, const TensorView &v, float *o_part,
                                  float *lse_part, const TensorView *out, float *lse_out,
                                  cudaStream_t st, bool *launched) {
    *launched = false;
    const bool dense = p.cu_q == nullptr;
    CUtensorMap mk, mv;
    const long long krows = dense ? p.max_sk : p.total_k;
    if (!make_map(&mk, k, dtype, p.d_qk, krows, p.H, p.B, dense) ||
        !make_map(&mv, v, dtype, p.d_v, krows, p.H, p.B, dense))
        return cudaSuccess;
    *launched = true;
#define SK_DEC_DIMS(T)                                                                                \
    if (p.d_qk == 192) return launch_dims<T, 192, 128>(p, mk, mv, q, o_part, lse_part, out, lse_out, st); \
    if (p.d_qk == 128) return launch_dims<T, 128, 128>(p, mk, mv, q, o_part, lse_part, out, lse_out, st); \
    return launch_dims<T, 64, 64>(p, mk, mv, q, o_part, lse_part, out, lse_out, st);
    if (dtype == kBF16) { SK_DEC_DIMS(__nv_bfloat16) }
    SK_DEC_DIMS(__half)
#undef SK_DEC_DIMS
}

}  // namespace dec
}  // namespace sk
