// tc_softmax.cuh -- pieces of the tcgen05 partial kernel: tile sizes, the bounded
// warp wait, and the online softmax that the softmax warpgroups run over TMEM.
//
// [P1] Technical details: per-split partials O_s = sum_j softmax(scale q.k_j) v_j and
// L_s = log sum_j exp(scale q.k_j) under the per-row masks; a row without a visible
// key writes O_s = 0 and L_s = -inf.
#pragma once

#include <float.h>

#include <type_traits>

#include "sk_common.cuh"
#include "sm100_ptx.cuh"

namespace sk {
namespace tc {

constexpr int kBM = 256;         // query rows per CTA (the partition's M block)
constexpr int kTileM = 128;      // rows per MMA tile (one TMEM lane per row)
constexpr int kBN = 128;         // keys per MMA tile
constexpr int kChunkBytes = 128 * 128;  // one 64-column (128-byte) swizzled panel of 128 rows
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.f;  // log2 units: rescale O only when m grows by > 2^8

enum ErrCode : int { kErrProducer = 0x101, kErrMma = 0x102, kErrSoftmax = 0x103 };

// Wait of a whole warp: every lane polls, the warp leaves together.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int *err, int code) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        bool ok = ptx::mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((i & 63u) == 63u) {
            int give_up = 0;
            if (lane == 0) {
                if (t0 == 0) t0 = ptx::globaltimer();
                if (*abort) give_up = 1;
                else if (ptx::globaltimer() - t0 > kTimeoutNs) {
                    *abort = 1;
                    if (err) atomicCAS(err, 0, code);
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
}

// The barriers one softmax warpgroup (tile t) works with (every thread arrives on
// p_ready).
struct SoftmaxBars {
    uint32_t s_full;   // S_t(j) is in TMEM (one phase per key tile)
    uint32_t p_ready;  // P_t(j) written
    uint32_t o_done;   // every MMA of the CTA finished (one phase)
};

// Online softmax of one query row per thread over the key tiles [kb, kb + n_tiles * kBN)
// of the (sequence, head, split), then the epilogue: O_s / l (or the final output when
// DIRECT) and L_s in natural log. Warp `wq` of the warpgroup owns TMEM lanes
// 32 wq .. 32 wq + 31; S_t / P_t live in TMEM columns [128 t, 128 t + 128), O_t in
// [256 + 128 t, 256 + 128 t + DV). Per key tile:
//   * load the S row, mask keys past the row's limit (and before its window start),
//   * running max m (base 2, scale * log2 e folded in) and sum l; when m grows by more
//     than 2^8 the row's O accumulator is rescaled (warp-uniform: TMEM accesses are
//     warp-collective; S_t(j) completing implies PV_t(j - 1) did, so O_t is stable),
//   * p = 2^(s * scale * log2 e - m) written back as 16-bit pairs over S's first
//     64 columns, then P_t(j) is reported.
// KVI (M blocks of at most 128 rows): both warpgroups own the same 128 rows, and tile t
// takes the key tiles 2 i + t; the loop then hands back its m and l (base 2) instead of
// writing anything, and kvi_epilogue merges the two halves.
// A CTA that runs several units in turn (the persistent form) passes the number of S_t
// phases its earlier units used (step0) and the parity of this unit's O-done phase.
// Returns false when a wait gave up (the CTA's abort flag is then raised).
template <typename T, int DV, bool DIRECT, bool KVI = false>
__device__ __forceinline__ bool softmax_rows(const Problem &p, const SeqInfo &si, int b, int h, int s,
                                             int pos0, int t, uint32_t tmem, int kb, int ke,
                                             int n_tiles, const SoftmaxBars &bars,
                                             volatile int *abort_flag, float *o_part,
                                             float *lse_part, const TensorView &out, float *lse_out,
                                             float4 *stage, float *m_out = nullptr,
                                             float *l_out = nullptr, uint32_t step0 = 0,
                                             uint32_t o_phase = 0) {
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wq = warp & 3;
    const int pos = pos0 + (KVI ? 0 : t * kTileM) + wq * 32 + lane;
    const bool row_ok = pos < si.sq;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)t * 128u;
    const uint32_t tO = tmem + lane_off + 256u + (uint32_t)t * 128u;
    const long long lim = row_limit(p, si.last_valid, pos);
    const int kend = lim + 1 < ke ? (int)(lim + 1 > kb ? lim + 1 : kb) : ke;
    // sliding window: the row's first visible key (0 without one), at most ke
    const long long kfirst_ll = row_start(p, pos);
    const int kfirst = kfirst_ll < ke ? (int)kfirst_ll : ke;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    const int n_mine = KVI ? (n_tiles + 1 - t) / 2 : n_tiles;  // KVI: t = 0 even, t = 1 odd tiles
    for (int j = 0; j < n_mine; ++j) {
        ok = warp_wait(bars.s_full, (step0 + j) & 1, abort_flag, p.err, kErrSoftmax);
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t r[128];
        ptx::tmem_ld_x128(tS, r);
        const int kt = KVI ? 2 * j + t : j;  // the key tile
        const int nvalid = kend - (kb + kt * kBN);
        const int nlow = kfirst - (kb + kt * kBN);
        if (nvalid < kBN || nlow > 0) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
                if (c >= nvalid || c < nlow) r[c] = __float_as_uint(-INFINITY);
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 128; c += 4) {
#pragma unroll
            for (int u = 0; u < 4; ++u) mx[u] = fmaxf(mx[u], __uint_as_float(r[c + u]));
        }
        const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        const float m_new = fmaxf(m, tmax * sl2);
        const bool grow = m_new > m + kRescaleThreshold;  // also true for the first finite max
        const bool any_grow = __any_sync(0xffffffffu, grow);
        const float alpha = grow ? ptx::ex2(m - m_new) : 1.f;  // 0 while m is -inf
        if (grow) m = m_new;
        l *= alpha;
        const float mneg = m == -INFINITY ? 0.f : -m;
        // p = 2^(s * scale * log2 e - m), two columns per packed FMA
        const uint64_t sc2 = ptx::f2pack(sl2, sl2), mn2 = ptx::f2pack(mneg, mneg);
        uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            float a, bq;
            ptx::f2unpack(ptx::ffma2(ptx::f2pack(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])),
                                     sc2, mn2),
                          a, bq);
            a = ptx::ex2(a);
            bq = ptx::ex2(bq);
            sum2[c & 1] = ptx::fadd2(sum2[c & 1], ptx::f2pack(a, bq));
            r[c] = ptx::pack2(a, bq, kBF16);
        }
        {
            float s0, s1, s2, s3;
            ptx::f2unpack(sum2[0], s0, s1);
            ptx::f2unpack(sum2[1], s2, s3);
            l += (s0 + s1) + (s2 + s3);
        }
        if (any_grow && j > 0) {
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 32) {
                uint32_t o[32];
                ptx::tmem_ld_x32(tO + c0, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                ptx::tmem_st_x32(tO + c0, o);
            }
        }
        __syncwarp();
        ptx::tmem_st_x64(tS, *reinterpret_cast<uint32_t(*)[64]>(r));
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bars.p_ready);
    }
    if (ok && n_tiles > 0) ok = warp_wait(bars.o_done, o_phase, abort_flag, p.err, kErrSoftmax);
    if constexpr (KVI) {
        *m_out = m;
        *l_out = l;
        return ok;
    }
    if (!ok) return false;
    ptx::tc_fence_after();
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
    const float lse = empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
    const int row = si.q0 + pos;
    // The warp's rows leave through its shared-memory slice (32 rows x 128 bytes), so that
    // each store covers four whole 128-byte row segments instead of 16 bytes of 32 rows.
    // Slot k (16 bytes) of row r sits at r * 8 + (k ^ (r & 7)): conflict-free both when a
    // thread writes its own row and when eight lanes read one row.
    const int row_w = pos0 + t * kTileM + wq * 32;  // the warp's first row
    const int k_rd = lane & 7;
    if constexpr (DIRECT) {
        // 64 output columns (128 bytes of bf16 / f16) per pass
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += 64) {
            uint32_t pk[32];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t o[32];
                if (n_tiles > 0) ptx::tmem_ld_x32(tO + c0 + 32 * hf, o);
                else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[16 * hf + i] = ptx::pack2(__uint_as_float(o[2 * i]) * inv,
                                                 __uint_as_float(o[2 * i + 1]) * inv, kBF16);
            }
            uint4 *st = reinterpret_cast<uint4 *>(stage);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                st[lane * 8 + (k ^ (lane & 7))] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + (lane >> 3);
                if (row_w + r < si.sq) {
                    T *dst = (T *)out.ptr + row_offset(p, out, b, si.q0, row_w + r) + (int64_t)h * out.sh +
                             c0 + 8 * k_rd;
                    *(uint4 *)dst = st[r * 8 + (k_rd ^ (r & 7))];
                }
            }
            __syncwarp();
        }
    } else {
        // 32 f32 partial columns (128 bytes) per pass
#pragma unroll
        for (int c0 = 0; c0 < DV; c0 += 32) {
            uint32_t o[32];
            if (n_tiles > 0) ptx::tmem_ld_x32(tO + c0, o);
            else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0u;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
                stage[lane * 8 + (k ^ (lane & 7))] =
                    make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + (lane >> 3);
                if (row_w + r < si.sq) {
                    float *dst = o_part + (((int64_t)h * p.S + s) * p.total_q + si.q0 + row_w + r) * DV +
                                 c0 + 4 * k_rd;
                    *(float4 *)dst = stage[r * 8 + (k_rd ^ (r & 7))];
                }
            }
            __syncwarp();
        }
    }
    if (row_ok) {
        if constexpr (DIRECT) {
            if (lse_out) lse_out[(int64_t)h * p.total_q + row] = lse;
        } else {
            lse_part[((int64_t)h * p.S + s) * p.total_q + row] = lse;
        }
    }
    return true;
}

// The KVI merge of the two halves of a 128-row M block. Warpgroup t held
// (m_t, l_t, O_t) over the key tiles 2 i + t (O_t in TMEM columns 256 + 128 t, scaled by
// 2^-m_t); with M = max(m_0, m_1) and a_t = 2^(m_t - M) (0 where l_t = 0):
//   O = (a_0 O_0 + a_1 O_1) / (a_0 l_0 + a_1 l_1),  L = ln 2 * (M + log2(a_0 l_0 + a_1 l_1))
// -- the merge of two splits, inside the CTA. The warpgroups swap m and l through shared
// memory (`xchg`, 2 KB that no load or MMA touches any more); then each warpgroup writes
// its share of the columns (the f32 partial O_s, or with DIRECT the output itself)
// through its warps' staging slices, 128 bytes of a row per pass, and warpgroup 0 the
// LSE. Every softmax thread reaches the barrier, also after an abort.
template <typename T, int DV, bool DIRECT>
__device__ __forceinline__ void kvi_epilogue(const Problem &p, const SeqInfo &si, int b, int h, int s,
                                             int pos0, int t, uint32_t tmem, int n_tiles, float m,
                                             float l, bool ok, float *xchg, float4 *stage,
                                             float *o_part, float *lse_part, const TensorView &out,
                                             float *lse_out) {
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kPassCols = DIRECT ? 64 : 32;                        // 128 bytes of a row
    constexpr int kMyCols = DV / 2 >= kPassCols ? DV / 2 : kPassCols;  // columns per warpgroup
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wq = warp & 3;
    const int i = wq * 32 + lane;
    if (ok) {
        xchg[(2 * t) * kTileM + i] = m;
        xchg[(2 * t + 1) * kTileM + i] = l;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (!ok) return;  // warp-uniform
    const float mo = xchg[(2 * (1 - t)) * kTileM + i], lo = xchg[(2 * (1 - t) + 1) * kTileM + i];
    const float m0 = t == 0 ? m : mo, l0 = t == 0 ? l : lo;
    const float m1 = t == 0 ? mo : m, l1 = t == 0 ? lo : l;
    const float mx = fmaxf(m0, m1);
    const float a0 = l0 > 0.f ? ptx::ex2(m0 - mx) : 0.f;
    const float a1 = l1 > 0.f ? ptx::ex2(m1 - mx) : 0.f;
    const float sum = a0 * l0 + a1 * l1;
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    const float w0 = a0 * inv, w1 = a1 * inv;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int row_w = pos0 + wq * 32;  // the warp's first row
    const int k_rd = lane & 7;
    // 32 merged columns c0 .. c0 + 31 of this thread's row
    auto merged = [&](int c0, float (&v)[32]) {
        uint32_t o0[32], o1[32];
        if (n_tiles > 0) ptx::tmem_ld_x32(tmem + lane_off + 256u + c0, o0);
        else {
#pragma unroll
            for (int c = 0; c < 32; ++c) o0[c] = 0u;
        }
        if (n_tiles > 1) ptx::tmem_ld_x32(tmem + lane_off + 384u + c0, o1);
        else {
#pragma unroll
            for (int c = 0; c < 32; ++c) o1[c] = 0u;
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = w0 * __uint_as_float(o0[c]) + w1 * __uint_as_float(o1[c]);
    };
#pragma unroll
    for (int c0 = t * kMyCols; c0 < DV && c0 < (t + 1) * kMyCols; c0 += kPassCols) {
        // slot k (16 bytes) of row r at r * 8 + (k ^ (r & 7)), as in softmax_rows
        if constexpr (DIRECT) {
            uint4 *st = reinterpret_cast<uint4 *>(stage);
            uint32_t pk[32];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float v[32];
                merged(c0 + 32 * hf, v);
#pragma unroll
                for (int c = 0; c < 16; ++c) pk[16 * hf + c] = ptx::pack2(v[2 * c], v[2 * c + 1], kBF16);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)
                st[lane * 8 + (k ^ (lane & 7))] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + (lane >> 3);
                if (row_w + r < si.sq) {
                    T *dst = (T *)out.ptr + row_offset(p, out, b, si.q0, row_w + r) + (int64_t)h * out.sh +
                             c0 + 8 * k_rd;
                    *(uint4 *)dst = st[r * 8 + (k_rd ^ (r & 7))];
                }
            }
        } else {
            float v[32];
            merged(c0, v);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                stage[lane * 8 + (k ^ (lane & 7))] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int r = it * 4 + (lane >> 3);
                if (row_w + r < si.sq) {
                    float *dst = o_part + (((int64_t)h * p.S + s) * p.total_q + si.q0 + row_w + r) * DV +
                                 c0 + 4 * k_rd;
                    *(float4 *)dst = stage[r * 8 + (k_rd ^ (r & 7))];
                }
            }
        }
        __syncwarp();
    }
    if (t == 0 && pos0 + i < si.sq) {
        const float lse = sum > 0.f ? (mx + log2f(sum)) * 0.69314718055994530942f : -INFINITY;
        if constexpr (DIRECT) {
            if (lse_out) lse_out[(int64_t)h * p.total_q + si.q0 + pos0 + i] = lse;
        } else {
            lse_part[((int64_t)h * p.S + s) * p.total_q + si.q0 + pos0 + i] = lse;
        }
    }
}

}  // namespace tc
}  // namespace sk
