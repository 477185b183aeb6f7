// partial_tc.cu -- split partials on the tcgen05 tensor cores (bf16 / f16 storage).
//
// [P1] Summary / Technical details; [P2] Technical details (split kernel plus a
// separate LSE combine). One CTA owns one (sequence, head, split, M block of 256
// query rows) and computes, over the keys of the split's run,
//   O_s = sum_j softmax(scale q.k_j) v_j,  L_s = log sum_j exp(scale q.k_j)
// with the causal / last-valid masks applied per row; rows without a visible key
// write O_s = 0 and L_s = -inf.
//
// Design (GB300, one CTA per SM):
//   * The M block is two 128-row MMA tiles Q0, Q1, kept in shared memory for the
//     whole CTA (TMA, 128-byte swizzle). Keys stream through in tiles of 128.
//   * Warps 8 and 10 (one lane each) are the TMA producers -- Q once and K(j);
//     V(j) -- into rings of shared-memory stages guarded by full / empty mbarriers,
//     so that a K stage is refilled as soon as it is free. With a single
//     V stage (D_QK = 192, where Q takes 96 KB) the stage is two 64-key halves with
//     their own barriers: PV1(j) frees the first half after its first four MMAs, so
//     V(j+1) starts arriving before PV1(j) has finished.
//   * Warp 9 (one lane) issues the tcgen05 MMAs: S_t = Q_t K(j)^T into TMEM
//     (128 f32 columns per tile), then O_t += P_t V(j) with P_t read from TMEM and
//     V(j) from shared memory (MN-major operand). The order
//       S0(0) S1(0) | PV0(0) S0(1) | PV1(0) S1(1) | PV0(1) S0(2) | ...
//     keeps the tensor core busy on one tile while the other tile's softmax runs.
//   * Warps 0-3 (tile 0) and 4-7 (tile 1) run the online softmax, one query row
//     per thread (TMEM lane = row): load the S row, mask, update the running max
//     m and sum l, write P (16-bit) over the first half of the S columns. When the
//     max grows by more than 2^8 the row's O accumulator in TMEM is rescaled first
//     (TMEM columns 256.. / 384..). Scores are kept in base 2 (scale * log2 e).
//   * TMEM: S0/P0 cols [0,128), S1/P1 [128,256), O0 [256,256+DV), O1 [384,384+DV).
//   * The epilogue writes each warp's 32 rows through a swizzled 4 KB slice of the (by
//     then idle) K stages, so that every global store covers whole 128-byte row segments.
//   * Single-block form (KVI, launches whose M blocks hold at most 128 queries: decode
//     with one or a few queries per sequence): tile 1 would hold only padding, so both
//     halves work on Q0's rows -- tile t takes the key tiles 2i + t into its own S / P /
//     O -- and the two halves are merged like two splits before anything is written.
//     One Q tile leaves room for one more V stage.
//   * Every mbarrier wait is bounded (1 s); a timeout records an error code in the
//     library's device error word, raises a CTA-wide abort flag, drains in-flight
//     TMA loads and MMAs, frees TMEM and returns.
#include <float.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "sk_common.cuh"
#include "sm100_ptx.cuh"
#include "sk_dispatch.h"
#include "tc_softmax.cuh"

namespace sk {
namespace tc {

constexpr int kThreads = 384;    // softmax warpgroups 0, 1; warpgroup 2: producers, MMA, 1 idle
constexpr int kProducerWarp = 8;   // Q and K
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10; // V
// Every warp keeps the 168 registers a thread of a 12-warp CTA starts with. Moving some
// of them from the control warps to the softmax warps made the MMA-issuing and producer
// code spill while the softmax fits in 168; every long workload ran slower that way.
constexpr int kLaunchRegs = 168;
// Launches whose M blocks hold at most 128 queries split each block's key tiles between
// the two halves (KVI), taking their (sequence, split) units longest first when there are
// at most kLptMaxUnits of them and in index order otherwise. One query per sequence comes
// here too: B32 H32 D128 decode takes 5.2 ms (7.4 TB/s of K and V) against 6.5 ms on the
// CUDA-core streaming decode kernel, 5.3-5.4 ms against 6.7-6.8 ms with 512-1024 units.

// KVI: M blocks of at most 128 rows. Tile 1 then holds no query of its own; instead it
// takes the odd key tiles of tile 0's rows (tile 0 the even ones), into its own S / P / O
// in TMEM, and the two halves are merged at the end. Only one Q tile is stored, which
// leaves room for one more V stage at D_QK = 192 and 128.
template <int DQK, int DV, bool KVI = false> struct Cfg {
    static constexpr int kQTiles = KVI ? 1 : 2;
    static constexpr int kQBytes = kTileM * DQK * 2;
    static constexpr int kKBytes = kBN * DQK * 2;
    static constexpr int kVBytes = kBN * DV * 2;
    static constexpr int kKStages = DQK == 192 ? 2 : (DQK == 128 ? 3 : 4);
    static constexpr int kVStages = DQK == 192 ? (KVI ? 2 : 1) : (DQK == 128 ? (KVI ? 3 : 2) : 4);
    // barriers: Q, K full/empty, V full/empty, S full x2, P full x2, O done x2, drain
    static constexpr int kBarQ = 0;
    static constexpr int kBarKF = 1;
    static constexpr int kBarKE = kBarKF + kKStages;
    static constexpr bool kSplitV = DQK == 192;             // V stages in two 64-key halves
    static constexpr int kVParts = kSplitV ? 2 : 1;
    static constexpr int kVPartBytes = kVBytes / kVParts;
    static constexpr int kVPanelBytes = kVPartBytes / (DV / 64);  // one 64-column panel of a part
    static constexpr int kBarVF = kBarKE + kKStages;       // [stage][part]
    static constexpr int kBarVE = kBarVF + kVParts * kVStages;
    static constexpr int kBarS = kBarVE + kVParts * kVStages;
    static constexpr int kBarP = kBarS + 2;
    static constexpr int kBarO = kBarP + 2;
    static constexpr int kBarDrain = kBarO + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kTileBytes = kQTiles * kQBytes + kKStages * kKBytes + kVStages * kVBytes;
    static constexpr int kSmemBytes = 1024 + kTileBytes + kNumBars * 8 + 16;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(DQK % 64 == 0 && DV % 64 == 0 && DV <= 128, "head dims");
    static_assert(kSplitV == (DQK == 192), "the V tensor map's box rows follow this rule");
};

constexpr int kMaxFusedSplits = 8;
constexpr int kMergeBatch = 8;  // rows a warp loads at once
constexpr int kMergePre = 3;    // splits per row among those loads (more are read afterwards)

// Merge of one M block's splits, run by the 256 softmax threads of the CTA that finished
// that (sequence, head, M block) last ([P1] NaN-safe merge over s < count, the count
// being the per-row formula of the count kernel):
//   1. thread i forms the weights of row pos0 + i: m = max(max_s L_s, lowest finite),
//      w_s = exp(L_s - m), 1 / max(sum_s w_s, 1), and writes the row's LSE;
//   2. warp w merges rows pos0 + 32 w .. + 31, eight rows at a time: every lane first
//      issues the 16-byte loads of eight rows x three splits (partials written by this
//      kernel, read through L2), then weights, sums and stores.
template <typename T, int DV>
__device__ __forceinline__ void merge_block(const Problem &p, const SeqInfo &si, int b, int h,
                                            int pos0, const float *o_part, const float *lse_part,
                                            const TensorView &out, float *lse_out, float *sW,
                                            float *sInv, int *sCnt) {
    constexpr int kLanes = DV / 4;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.S;
    const int64_t plane = p.total_q;
    {
        const int own = pos0 + tid;
        int c = 0;
        if (own < si.sq) c = merged_splits(p, si.sq, si.last_valid, own, valid_split_count(p, si.last_valid, own));
        const float *lrow = lse_part + (int64_t)h * S * plane + si.q0 + own;
        float l[kMaxFusedSplits];
        float m = -FLT_MAX;
#pragma unroll
        for (int sp = 0; sp < kMaxFusedSplits; ++sp) {
            l[sp] = sp < c ? __ldcg(lrow + sp * plane) : -INFINITY;
            m = fmaxf(m, l[sp]);
        }
        float wsum = 0.f;
#pragma unroll
        for (int sp = 0; sp < kMaxFusedSplits; ++sp) {
            const float w = sp < c ? expf(l[sp] - m) : 0.f;
            sW[sp * 256 + tid] = w;
            wsum += w;
        }
        sInv[tid] = 1.f / fmaxf(wsum, 1.f);
        sCnt[tid] = c;
        if (own < si.sq && lse_out)
            lse_out[(int64_t)h * plane + si.q0 + own] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const float *obase = o_part + ((int64_t)h * S * plane + si.q0 + pos0) * DV + lane * 4;
    for (int r0 = 0; r0 < 32; r0 += kMergeBatch) {
        const int rb = warp * 32 + r0;
        if (pos0 + rb >= si.sq) break;  // warp-uniform
        float4 o[kMergeBatch][kMergePre];
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
            const int ci = sCnt[rb + i];
#pragma unroll
            for (int sp = 0; sp < kMergePre; ++sp)
                o[i][sp] = (sp < ci && lane < kLanes)
                               ? __ldcg((const float4 *)(obase + ((int64_t)sp * plane + rb + i) * DV))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
            const int rl = rb + i;
            if (pos0 + rl >= si.sq) break;  // warp-uniform
            const int ci = sCnt[rl];
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int sp = 0; sp < kMergePre; ++sp) {
                const float w = sp < ci ? sW[sp * 256 + rl] : 0.f;
                acc.x = fmaf(w, o[i][sp].x, acc.x);
                acc.y = fmaf(w, o[i][sp].y, acc.y);
                acc.z = fmaf(w, o[i][sp].z, acc.z);
                acc.w = fmaf(w, o[i][sp].w, acc.w);
            }
            for (int sp = kMergePre; sp < ci; ++sp) {
                const float4 v = lane < kLanes
                                     ? __ldcg((const float4 *)(obase + ((int64_t)sp * plane + rl) * DV))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                const float w = sW[sp * 256 + rl];
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
            const float inv = sInv[rl];
            if (lane < kLanes) {
                T *dst = (T *)out.ptr + row_offset(p, out, b, si.q0, pos0 + rl) + (int64_t)h * out.sh +
                         lane * 4;
                uint2 v;
                v.x = ptx::pack2(acc.x * inv, acc.y * inv, kBF16);
                v.y = ptx::pack2(acc.z * inv, acc.w * inv, kBF16);
                *(uint2 *)dst = v;
            }
        }
    }
}

// LPT: the (sequence, split) units -- the slowest launch dimension -- are taken longest
// first (lpt_unit), for launches of at most kLptMaxUnits units where ragged sequence
// lengths would otherwise leave the longest sequences for the last wave: single-M-block
// launches (decode-like shapes with a few queries per sequence) and partials of several
// sequences over more than one wave of CTAs (packed varlen prefill). Other launches keep
// the unit from blockIdx.
// KVI: the single-block form (see Cfg); DIRECT: split 1, the output written directly.
template <typename T, int DQK, int DV, bool DIRECT, bool LPT = false, bool KVI = false>
__global__ void __launch_bounds__(kThreads, 1)
    partial_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, Problem p, float *o_part,
                      float *lse_part, TensorView out, float *lse_out, int *tickets) {
    using C = Cfg<DQK, DV, KVI>;
    constexpr bool kBF16 = sizeof(T) == 2 && std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    ptx::launch_dependents();  // the combine may be scheduled onto SMs this grid leaves idle

    // under causal masks the last M blocks of a sequence see the most keys: they go first,
    // so that the short ones fill the last wave (single-block launches have one M block)
    const int mb = (!KVI && p.causal) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    const int h = blockIdx.y;
    int s, b;
    if constexpr (LPT) {
        __shared__ int lpt_found;
        const int unit = lpt_unit(p, blockIdx.z, gridDim.z, (int *)smem_raw, &lpt_found);
        s = unit % p.S;
        b = unit / p.S;
    } else {
        // straight from the block index, which the compiler may re-read instead of keeping
        s = blockIdx.z % p.S;
        b = blockIdx.z / p.S;
    }
    const SeqInfo si = seq_info(p, b);
    const int pos0 = mb * kBM;
    if (pos0 >= si.sq) return;  // uniform: the M block lies past this sequence
    int kb, ke;
    split_key_range(p, si.sq, si.last_valid, pos0, s, kb, ke);
    int n_tiles = ke > kb ? (ke - kb + kBN - 1) / kBN : 0;
    // real early exit: a split without keys writes nothing (the merge never reads it)
    if (!DIRECT && n_tiles == 0 && p.skip_empty && tickets == nullptr) return;
    {
        // sliding window: key tiles before the first key any row of the block may see
        // (row pos0 has the earliest window) are skipped by every role
        const long long first = row_start(p, pos0);
        if (first > kb) {
            int skip = (int)((first - kb) / kBN);
            if (skip > n_tiles) skip = n_tiles;
            kb += skip * kBN;
            n_tiles -= skip;
        }
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    const uint32_t sQ = (raw_u32 + 1023u) & ~1023u;
    const uint32_t sK = sQ + C::kQTiles * C::kQBytes;
    const uint32_t sV = sK + C::kKStages * C::kKBytes;
    const uint32_t bar0 = sV + C::kVStages * C::kVBytes;
    uint8_t *const gen_base = smem_raw + (sQ - raw_u32);
    uint32_t *const tmem_holder = (uint32_t *)(gen_base + (bar0 - sQ) + C::kNumBars * 8);
    volatile int *const abort_flag = (volatile int *)(tmem_holder + 1);
    volatile int *const fused_last = (volatile int *)(tmem_holder + 2);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(C::kBarQ), 1);
        for (int i = 0; i < C::kKStages; ++i) {
            ptx::mbar_init(bar(C::kBarKF + i), 1);
            ptx::mbar_init(bar(C::kBarKE + i), 1);
        }
        for (int i = 0; i < C::kVParts * C::kVStages; ++i) {
            ptx::mbar_init(bar(C::kBarVF + i), 1);
            ptx::mbar_init(bar(C::kBarVE + i), 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bar(C::kBarS + t), 1);
            ptx::mbar_init(bar(C::kBarP + t), kTileM);
            ptx::mbar_init(bar(C::kBarO + t), 1);
        }
        ptx::mbar_init(bar(C::kBarDrain), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    const bool dense = p.cu_q == nullptr;
    const int cb = dense ? b : 0;

    if (warp >= 8) {
    if (warp == kProducerWarp || warp == kVProducerWarp) {
        // ---------------------------------------------------------- TMA producers
        // Two threads: K (with Q) and V, so that K(j + 1) is requested as soon as its
        // stage is free rather than after V(j), whose single stage frees late.
        if (lane == 0 && n_tiles > 0) {
            const int krow = (dense ? 0 : si.k0) + kb;
            int quiet = 0;
            volatile int *no_abort = (volatile int *)&quiet;
            bool ok = true;
            if (warp == kProducerWarp) {
                ptx::prefetch_tensormap(&tmQ);
                ptx::prefetch_tensormap(&tmK);
                const int qrow = dense ? pos0 : si.q0 + pos0;
                ptx::mbar_arrive_expect_tx(bar(C::kBarQ), C::kQTiles * C::kQBytes);
                for (int t = 0; t < C::kQTiles; ++t)
                    for (int c = 0; c < DQK / 64; ++c)
                        ptx::tma_load_4d(sQ + t * C::kQBytes + c * kChunkBytes, &tmQ, bar(C::kBarQ),
                                         c * 64, qrow + t * kTileM, h, cb);
                int issued_k = 0;
                for (int j = 0; j < n_tiles; ++j) {
                    const int ks = j % C::kKStages;
                    ok = ptx::mbar_wait_bounded(bar(C::kBarKE + ks), ((j / C::kKStages) & 1) ^ 1,
                                                abort_flag, p.err, kErrProducer, kTimeoutNs);
                    if (!ok) break;
                    ptx::mbar_arrive_expect_tx(bar(C::kBarKF + ks), C::kKBytes);
                    for (int c = 0; c < DQK / 64; ++c)
                        ptx::tma_load_4d(sK + ks * C::kKBytes + c * kChunkBytes, &tmK,
                                         bar(C::kBarKF + ks), c * 64, krow + j * kBN, h, cb);
                    issued_k = j + 1;
                }
                if (!ok) {
                    // drain: every load already issued must land before the CTA exits
                    ptx::mbar_wait_bounded(bar(C::kBarQ), 0, no_abort, nullptr, 0, kTimeoutNs);
                    for (int i = 0; i < C::kKStages && i < issued_k; ++i) {
                        const int last = i + ((issued_k - 1 - i) / C::kKStages) * C::kKStages;
                        ptx::mbar_wait_bounded(bar(C::kBarKF + i), (last / C::kKStages) & 1, no_abort,
                                               nullptr, 0, kTimeoutNs);
                    }
                }
            } else {
                ptx::prefetch_tensormap(&tmV);
                int issued_v = 0;
                for (int j = 0; j < n_tiles && ok; ++j) {
                    const int vs = j % C::kVStages;
                    for (int hf = 0; hf < C::kVParts; ++hf) {
                        const int vb = C::kVParts * vs + hf;
                        ok = ptx::mbar_wait_bounded(bar(C::kBarVE + vb), ((j / C::kVStages) & 1) ^ 1,
                                                    abort_flag, p.err, kErrProducer, kTimeoutNs);
                        if (!ok) break;
                        ptx::mbar_arrive_expect_tx(bar(C::kBarVF + vb), C::kVPartBytes);
                        for (int c = 0; c < DV / 64; ++c)
                            ptx::tma_load_4d(sV + vs * C::kVBytes + hf * C::kVPartBytes + c * C::kVPanelBytes,
                                             &tmV, bar(C::kBarVF + vb), c * 64,
                                             krow + j * kBN + hf * (kBN / C::kVParts), h, cb);
                        issued_v = C::kVParts * j + hf + 1;
                    }
                }
                if (!ok) {
                    // V parts are issued in the order P j, P j + 1, ... (P = kVParts) into
                    // barrier (j % kVStages) * P + part
                    constexpr int kVB = C::kVParts * C::kVStages;
                    for (int i = 0; i < kVB && i < issued_v; ++i) {
                        const int last = i + ((issued_v - 1 - i) / kVB) * kVB;
                        ptx::mbar_wait_bounded(bar(C::kBarVF + i), ((last / C::kVParts) / C::kVStages) & 1,
                                               no_abort, nullptr, 0, kTimeoutNs);
                    }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------------- MMA issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t kIdescQK = ptx::idesc_f16(kBF16, false, false, kTileM, kBN);
            constexpr uint32_t kIdescPV = ptx::idesc_f16(kBF16, false, true, kTileM, DV);
            const uint32_t tS[2] = {tmem, tmem + 128u};
            const uint32_t tO[2] = {tmem + 256u, tmem + 384u};
            auto issue_qk = [&](int t, int j) {
                const uint64_t kd = ptx::smem_desc_sw128(sK + (j % C::kKStages) * C::kKBytes, 16, 1024);
                const uint64_t qd = ptx::smem_desc_sw128(sQ + t * C::kQBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < DQK / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    ptx::mma_ss(tS[t], ptx::desc_advance(qd, off), ptx::desc_advance(kd, off), kIdescQK, kk > 0);
                }
                ptx::tc_commit(bar(C::kBarS + t));
            };
            // O_t (+)= P_t V(j) over one V part (all 128 keys, or one 64-key half); N = DV
            // spans the part's 64-column panels, kVPanelBytes apart
            auto issue_pv_part = [&](int t, int j, int hf) {
                constexpr int kSteps = kBN / 16 / C::kVParts;
                const uint64_t vd = ptx::smem_desc_sw128(sV + (j % C::kVStages) * C::kVBytes + hf * C::kVPartBytes,
                                                         C::kVPanelBytes, 1024);
#pragma unroll
                for (int k4 = 0; k4 < kSteps; ++k4) {
                    const int kk = hf * kSteps + k4;
                    ptx::mma_ts(tO[t], tS[t] + kk * 8, ptx::desc_advance(vd, k4 * 2048), kIdescPV,
                                (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            if constexpr (KVI) {
                // tile t takes the key tiles k = 2 i + t: S_t(i) = Q0 K(k)^T, then
                // O_t (+)= P_t(i) V(k); the order S0 S1 | PV0 S0 | PV1 S1 | ... is kept
                auto wait_k = [&](int k) {
                    return ptx::mbar_wait_bounded(bar(C::kBarKF + k % C::kKStages), (k / C::kKStages) & 1,
                                                  abort_flag, p.err, kErrMma, kTimeoutNs);
                };
                auto issue_qk_k = [&](int t, int k) {
                    const uint64_t kd = ptx::smem_desc_sw128(sK + (k % C::kKStages) * C::kKBytes, 16, 1024);
                    const uint64_t qd = ptx::smem_desc_sw128(sQ, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < DQK / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                        ptx::mma_ss(tS[t], ptx::desc_advance(qd, off), ptx::desc_advance(kd, off), kIdescQK, kk > 0);
                    }
                    ptx::tc_commit(bar(C::kBarS + t));
                    ptx::tc_commit(bar(C::kBarKE + k % C::kKStages));  // only S_t(i) reads K(k)
                };
                // V(k) part by part, each part freed once its MMAs are done
                auto issue_pv_k = [&](int t, int k, int i) {
                    constexpr int kSteps = kBN / 16 / C::kVParts;
                    const int vs = k % C::kVStages;
                    const uint32_t vpar = (k / C::kVStages) & 1;
                    for (int hf = 0; hf < C::kVParts; ++hf) {
                        if (!ptx::mbar_wait_bounded(bar(C::kBarVF + C::kVParts * vs + hf), vpar, abort_flag,
                                                    p.err, kErrMma, kTimeoutNs))
                            return false;
                        ptx::tc_fence_after();
                        const uint64_t vd = ptx::smem_desc_sw128(sV + vs * C::kVBytes + hf * C::kVPartBytes,
                                                                 C::kVPanelBytes, 1024);
#pragma unroll
                        for (int k4 = 0; k4 < kSteps; ++k4) {
                            const int kk = hf * kSteps + k4;
                            ptx::mma_ts(tO[t], tS[t] + kk * 8, ptx::desc_advance(vd, k4 * 2048), kIdescPV,
                                        (i > 0 || kk > 0) ? 1u : 0u);
                        }
                        ptx::tc_commit(bar(C::kBarVE + C::kVParts * vs + hf));
                    }
                    return true;
                };
                bool ok = ptx::mbar_wait_bounded(bar(C::kBarQ), 0, abort_flag, p.err, kErrMma, kTimeoutNs) &&
                          wait_k(0);
                if (ok) {
                    ptx::tc_fence_after();
                    issue_qk_k(0, 0);
                }
                if (ok && n_tiles > 1) {
                    ok = wait_k(1);
                    if (ok) {
                        ptx::tc_fence_after();
                        issue_qk_k(1, 1);
                    }
                }
                for (int i = 0; 2 * i < n_tiles && ok; ++i) {
                    for (int t = 0; t < 2 && ok; ++t) {
                        const int k = 2 * i + t;
                        if (k >= n_tiles) break;
                        ok = ptx::mbar_wait_bounded(bar(C::kBarP + t), i & 1, abort_flag, p.err, kErrMma,
                                                    kTimeoutNs) &&
                             issue_pv_k(t, k, i);
                        if (ok && k + 2 < n_tiles) {
                            ok = wait_k(k + 2);
                            if (ok) {
                                ptx::tc_fence_after();
                                issue_qk_k(t, k + 2);
                            }
                        }
                    }
                }
                if (ok) {
                    ptx::tc_commit(bar(C::kBarO + 0));
                    ptx::tc_commit(bar(C::kBarO + 1));
                }
            } else {
                bool ok = ptx::mbar_wait_bounded(bar(C::kBarQ), 0, abort_flag, p.err, kErrMma, kTimeoutNs) &&
                          ptx::mbar_wait_bounded(bar(C::kBarKF), 0, abort_flag, p.err, kErrMma, kTimeoutNs);
                if (ok) {
                    ptx::tc_fence_after();
                    issue_qk(0, 0);
                    issue_qk(1, 0);
                    ptx::tc_commit(bar(C::kBarKE));
                }
                for (int j = 0; j < n_tiles && ok; ++j) {
                    const int vs = j % C::kVStages;
                    const int kn = (j + 1) % C::kKStages;
                    const uint32_t vpar = (j / C::kVStages) & 1;
                    ok = ptx::mbar_wait_bounded(bar(C::kBarP + 0), j & 1, abort_flag, p.err, kErrMma,
                                                kTimeoutNs);
                    for (int hf = 0; hf < C::kVParts && ok; ++hf) {
                        ok = ptx::mbar_wait_bounded(bar(C::kBarVF + C::kVParts * vs + hf), vpar, abort_flag,
                                                    p.err, kErrMma, kTimeoutNs);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        issue_pv_part(0, j, hf);
                    }
                    if (!ok) break;
                    if (j + 1 < n_tiles) {
                        ok = ptx::mbar_wait_bounded(bar(C::kBarKF + kn), ((j + 1) / C::kKStages) & 1,
                                                    abort_flag, p.err, kErrMma, kTimeoutNs);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        issue_qk(0, j + 1);
                    }
                    ok = ptx::mbar_wait_bounded(bar(C::kBarP + 1), j & 1, abort_flag, p.err, kErrMma,
                                                kTimeoutNs);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    for (int hf = 0; hf < C::kVParts; ++hf) {
                        issue_pv_part(1, j, hf);
                        ptx::tc_commit(bar(C::kBarVE + C::kVParts * vs + hf));  // this part of V(j) is free
                    }
                    if (j + 1 < n_tiles) {
                        issue_qk(1, j + 1);
                        ptx::tc_commit(bar(C::kBarKE + kn));
                    }
                }
                if (ok) {
                    ptx::tc_commit(bar(C::kBarO + 0));
                    ptx::tc_commit(bar(C::kBarO + 1));
                }
            }
            // every issued MMA must be finished before TMEM is released
            int dummy = 0;
            ptx::tc_commit(bar(C::kBarDrain));
            ptx::mbar_wait_bounded(bar(C::kBarDrain), 0, (volatile int *)&dummy, nullptr, 0,
                                   kTimeoutNs);
        }
    }  // warp 11 has no role
    } else {
        // ---------------------------------------------------------------- softmax
        const int t = warp >> 2;
        const SoftmaxBars sb{bar(C::kBarS + t), bar(C::kBarP + t), bar(C::kBarO + t)};
        // epilogue staging: 4 KB per softmax warp in the K stages, which no load or MMA
        // touches once the O-done barrier has completed (or when the split has no tile)
        float4 *stage = (float4 *)(gen_base + (sK - sQ)) + warp * 256;
        if constexpr (KVI) {
            // the two halves swap m and l through the Q tile's memory: every MMA has
            // finished once the O-done barrier completed (or no load was issued at all)
            float m_r = -INFINITY, l_r = 0.f;
            const bool ok_r = softmax_rows<T, DV, false, true>(p, si, b, h, s, pos0, t, tmem, kb, ke, n_tiles,
                                                              sb, abort_flag, o_part, lse_part, out, lse_out,
                                                              stage, &m_r, &l_r);
            kvi_epilogue<T, DV, DIRECT>(p, si, b, h, s, pos0, t, tmem, n_tiles, m_r, l_r, ok_r,
                                        (float *)gen_base, stage, o_part, lse_part, out, lse_out);
        } else {
            softmax_rows<T, DV, DIRECT>(p, si, b, h, s, pos0, t, tmem, kb, ke, n_tiles, sb,
                                        abort_flag, o_part, lse_part, out, lse_out, stage);
        }
        if constexpr (!DIRECT && !KVI) {
            // Fused merge: the CTA of this (sequence, head, M block) that writes its
            // partials last merges all splits. Every softmax thread takes part in both
            // barriers, also after an abort. Shared memory is free by now: every MMA and
            // load of this CTA has completed.
            if (tickets) {
                __threadfence();
                asm volatile("bar.sync 1, 256;" ::: "memory");
                if (threadIdx.x == 0) {
                    const int group = (b * p.H + h) * (int)gridDim.x + mb;
                    *fused_last = !*abort_flag && atomicAdd(tickets + group, 1) == p.S - 1;
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");
                if (*fused_last) {
                    __threadfence();
                    float *sW = (float *)gen_base;  // [kMaxFusedSplits][256]
                    merge_block<T, DV>(p, si, b, h, pos0, o_part, lse_part, out, lse_out, sW,
                                       sW + kMaxFusedSplits * 256, (int *)(sW + (kMaxFusedSplits + 1) * 256));
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}
static_assert(kLaunchRegs * kThreads <= 65536, "launch registers");

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
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)f;
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// [rows, H, D] (varlen: rows = total, one batch) or [B][rows][H][D] (dense), box of
// 64 elements x box_rows rows, 128-byte swizzle; out-of-range rows read as zero.
bool make_map(CUtensorMap *m, const TensorView &t, int dtype, int D, long long rows, int H,
                     int B, bool dense, unsigned box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows <= 0 || t.sr <= 0 || t.sh <= 0) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)(dense ? B : 1)};
    cuuint64_t strides[3] = {(cuuint64_t)t.sr * 2, (cuuint64_t)t.sh * 2,
                             (cuuint64_t)(dense ? t.sb : rows * t.sr) * 2};
    if (dense && t.sb <= 0) return false;
    cuuint32_t box[4] = {64, box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     4, t.ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename T, int DQK, int DV, bool DIRECT, bool LPT = false, bool KVI = false>
static cudaError_t launch_cfg(const Problem &p, const CUtensorMap &mq, const CUtensorMap &mk,
                              const CUtensorMap &mv, float *o_part, float *lse_part,
                              const TensorView &out, float *lse_out, int *tickets, cudaStream_t st) {
    using C = Cfg<DQK, DV, KVI>;
    auto kern = partial_tc_kernel<T, DQK, DV, DIRECT, LPT, KVI>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    dim3 grid((unsigned)((p.max_sq + kBM - 1) / kBM), (unsigned)p.H, (unsigned)(p.B * p.S));
    kern<<<grid, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, p, o_part, lse_part, out, lse_out, tickets);
    return cudaGetLastError();
}

static int sm_count_of_device();

// out without tickets: S == 1, the kernel writes the output directly. out with
// tickets: partials, merged by the last CTA of each M block. No out: partials only.
template <typename T, int DQK, int DV>
static cudaError_t launch_dims(const Problem &p, const CUtensorMap &mq, const CUtensorMap &mk,
                               const CUtensorMap &mv, float *o_part, float *lse_part,
                               const TensorView *out, float *lse_out, int *tickets, cudaStream_t st) {
    const long long units = (long long)p.B * p.S;
    if (out && !tickets) {
        // S == 1: the output is written directly
        if (p.max_sq <= kTileM && units <= kLptMaxUnits)
            return launch_cfg<T, DQK, DV, true, true, true>(p, mq, mk, mv, o_part, lse_part, *out, lse_out,
                                                            nullptr, st);
        if (p.max_sq <= kTileM)
            return launch_cfg<T, DQK, DV, true, false, true>(p, mq, mk, mv, o_part, lse_part, *out, lse_out,
                                                             nullptr, st);
        return launch_cfg<T, DQK, DV, true>(p, mq, mk, mv, o_part, lse_part, *out, lse_out, nullptr, st);
    }
    // partials only (no fused merge): single-M-block launches take their units longest first
    if (!(out && tickets) && p.max_sq <= kTileM && units <= kLptMaxUnits)
        return launch_cfg<T, DQK, DV, false, true, true>(p, mq, mk, mv, o_part, lse_part, TensorView{},
                                                         nullptr, nullptr, st);
    if (!(out && tickets) && p.max_sq <= kTileM)  // too many units to rank: index order
        return launch_cfg<T, DQK, DV, false, false, true>(p, mq, mk, mv, o_part, lse_part, TensorView{},
                                                          nullptr, nullptr, st);
    // Several sequences over more than one wave of CTAs: with ragged lengths, index order
    // leaves the units of the longest sequences for the last waves, so they go first
    // (long varlen prefill: 4.73 -> 4.61 ms at split 3). Within one wave, or with one
    // sequence, the ranking only delays each CTA's start.
    const long long ctas = (long long)((p.max_sq + kBM - 1) / kBM) * p.H * units;
    const int sms = sm_count_of_device();
    const bool ragged_waves = p.B > 1 && sms > 0 && ctas > sms;
    if (!(out && tickets) && units > 1 && units <= kLptMaxUnits && (p.max_sq <= kBM || ragged_waves))
        return launch_cfg<T, DQK, DV, false, true>(p, mq, mk, mv, o_part, lse_part, TensorView{}, nullptr,
                                                   nullptr, st);
    return launch_cfg<T, DQK, DV, false>(p, mq, mk, mv, o_part, lse_part, out ? *out : TensorView{},
                                         out ? lse_out : nullptr, out ? tickets : nullptr, st);
}

bool partial_tc_supported(const Problem &p, int dtype) {
    if (dtype != kBF16 && dtype != kF16) return false;
    if (!((p.d_qk == 64 && p.d_v == 64) || (p.d_qk == 128 && p.d_v == 128) ||
          (p.d_qk == 192 && p.d_v == 128)))
        return false;
    if (p.bm != kBM || p.total_k <= 0 || p.max_sk <= 0 || p.total_q <= 0) return false;
    if (p.max_sq < 1) return false;
    if ((long long)p.B * p.S > 65535 || p.H > 65535) return false;
    if (encode_fn() == nullptr) return false;
    return true;
}

// SM count of the current device (cached per device; 0 when it cannot be read).
static int sm_count_of_device() {
    static std::atomic<int> sms[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev < 0 || dev >= 64) return 0;
    int n = sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

bool persist_selected(const Problem &p) {
    const int sms = sm_count_of_device();
    return sms > 0 && persist_fits(p, sms);
}

cudaError_t launch_partial_tc(const Problem &p, int dtype, const TensorView &q, const TensorView &k,
                              const TensorView &v, float *o_part, float *lse_part,
                              const TensorView *out, float *lse_out, int *tickets, cudaStream_t st,
                              bool *launched) {
    *launched = false;
    if (tickets && (p.S < 2 || p.S > kMaxFusedSplits)) return cudaSuccess;  // not fusable
    const bool dense = p.cu_q == nullptr;
    CUtensorMap mq, mk, mv;
    const long long qrows = dense ? p.max_sq : p.total_q;
    const long long krows = dense ? p.max_sk : p.total_k;
    if (!make_map(&mq, q, dtype, p.d_qk, qrows, p.H, p.B, dense, 128) ||
        !make_map(&mk, k, dtype, p.d_qk, krows, p.H, p.B, dense, 128) ||
        !make_map(&mv, v, dtype, p.d_v, krows, p.H, p.B, dense, p.d_qk == 192 ? 64 : 128))
        return cudaSuccess;  // not expressible as TMA maps: the caller falls back
    *launched = true;
    // many short units: one CTA per SM takes them in turn (partial_tc_persist.cu)
    if (!tickets && persist_selected(p))
        return launch_partial_tc_persist(p, dtype, mq, mk, mv, o_part, lse_part, out, lse_out,
                                         sm_count_of_device(), st);
#define SK_TC_DIMS(T)                                                                              \
    if (p.d_qk == 192) return launch_dims<T, 192, 128>(p, mq, mk, mv, o_part, lse_part, out, lse_out, tickets, st); \
    if (p.d_qk == 128) return launch_dims<T, 128, 128>(p, mq, mk, mv, o_part, lse_part, out, lse_out, tickets, st); \
    return launch_dims<T, 64, 64>(p, mq, mk, mv, o_part, lse_part, out, lse_out, tickets, st);
    if (dtype == kBF16) { SK_TC_DIMS(__nv_bfloat16) }
    SK_TC_DIMS(__half)
#undef SK_TC_DIMS
}

}  // namespace tc
}  // namespace sk
