// partial_tc_persist.cu -- the tensor-core partial kernel in persistent form, for launches
// of many short (sequence, head, split, M block) units (D_QK = D_V = 64 or 128).
//
// [P1] Summary / Technical details: each unit computes, over the keys of its split's
// run, O_s = sum_j softmax(scale q.k_j) v_j and L_s = log sum_j exp(scale q.k_j) under
// the per-row masks (rows without a visible key: O_s = 0, L_s = -inf) -- exactly what
// partial_tc_kernel computes for one unit per CTA.
//
// When a unit holds only a few key tiles (causal masks with several splits), a CTA of
// partial_tc_kernel spends most of its time filling Q, K and V and writing its partial
// rows. Here one CTA per SM takes the units in turn, and the roles run ahead into the
// next unit while the softmax warps write the current one:
//   * warp 11 (one lane) loads the two Q tiles of each unit once every S MMA of the
//     previous unit is done (a Q-empty barrier);
//   * warps 8 and 10 (one lane each) stream K and V through rings whose stages and
//     phases run on across units, so the next unit's first tiles land during the
//     current unit's last steps;
//   * warp 9 (one lane) issues the MMAs in the order of partial_tc_kernel
//       S0(0) S1(0) | PV0(0) S0(1) | PV1(0) S1(1) | ...
//     and issues the next unit's S0(0) S1(0) as soon as its Q and K are in, while the
//     softmax warps still write the previous unit (its S / P columns are free once
//     PV_t(last) is issued: tcgen05 MMAs of one thread run in order; O_t is
//     overwritten only by PV_t(0) of the next unit, which waits for P_t(0), which the
//     softmax warps report after their epilogue);
//   * warps 0-7 run the online softmax and the epilogue of each unit (tc_softmax.cuh),
//     staging the partial rows in a shared-memory area of their own (the K stages are
//     busy with the next unit).
// Units are dealt out statically: unit u of CTA c in round i is i * grid + c in even
// rounds and i * grid + grid - 1 - c in odd ones, with the M blocks that see the most
// keys under causal masks (the last ones) first, so that the rounds balance.
// Every wait is bounded, as in partial_tc_kernel.
#include <float.h>

#include <mutex>
#include <type_traits>

#include "sk_common.cuh"
#include "sm100_ptx.cuh"
#include "sk_dispatch.h"
#include "tc_softmax.cuh"

namespace sk {
namespace tc {

namespace {
constexpr int kPersistMaxTiles = 16;  // key tiles per unit up to which the persistent form is used
constexpr int kPThreads = 384;
constexpr int kPKWarp = 8;      // K producer
constexpr int kPMmaWarp = 9;
constexpr int kPVWarp = 10;     // V producer
constexpr int kPQWarp = 11;     // Q producer
constexpr int kPLaunchRegs = 168;  // every warp keeps them (no reallocation, as in partial_tc)
}  // namespace

template <int DQK, int DV> struct PCfg {
    static constexpr int kQBytes = kTileM * DQK * 2;  // one 128-row Q tile
    static constexpr int kKBytes = kBN * DQK * 2;
    static constexpr int kVBytes = kBN * DV * 2;
    static constexpr int kVPanelBytes = kVBytes / (DV / 64);  // one 64-column panel of V
    static constexpr int kKStages = DQK == 128 ? 2 : 4;
    static constexpr int kVStages = DQK == 128 ? 2 : 4;
    static constexpr int kStageBytes = 8 * 32 * 128;  // 4 KB epilogue slice per softmax warp
    static constexpr int kBarQF = 0;
    static constexpr int kBarQE = 1;
    static constexpr int kBarKF = 2;
    static constexpr int kBarKE = kBarKF + kKStages;
    static constexpr int kBarVF = kBarKE + kKStages;
    static constexpr int kBarVE = kBarVF + kVStages;
    static constexpr int kBarS = kBarVE + kVStages;
    static constexpr int kBarP = kBarS + 2;
    static constexpr int kBarO = kBarP + 2;
    static constexpr int kBarDrain = kBarO + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kTileBytes = 2 * kQBytes + kKStages * kKBytes + kVStages * kVBytes + kStageBytes;
    static constexpr int kSmemBytes = 1024 + kTileBytes + kNumBars * 8 + 16;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert((DQK == 64 || DQK == 128) && DV == DQK, "head dims of the persistent form");
};

// One unit of work: (sequence b, head h, split s, M block mb) and its key tiles.
struct PUnit {
    int b, h, s, pos0, kb, ke, n_tiles;
    SeqInfo si;
    bool live;  // false: nothing to do (past the sequence, or an empty split that writes nothing)
};

// Unit u: M blocks outermost, the last (under causal masks the longest) first; then
// sequence, split and head.
template <bool DIRECT>
__device__ __forceinline__ PUnit unit_at(const Problem &p, int u, int n_mb) {
    PUnit U;
    const int per_mb = p.H * p.B * p.S;
    const int mb = n_mb - 1 - u / per_mb;
    int r = u % per_mb;
    U.h = r % p.H;
    r /= p.H;
    U.s = r % p.S;
    U.b = r / p.S;
    U.si = seq_info(p, U.b);
    U.pos0 = mb * kBM;
    U.live = U.pos0 < U.si.sq;
    U.kb = U.ke = U.n_tiles = 0;
    if (!U.live) return U;
    split_key_range(p, U.si.sq, U.si.last_valid, U.pos0, U.s, U.kb, U.ke);
    U.n_tiles = U.ke > U.kb ? (U.ke - U.kb + kBN - 1) / kBN : 0;
    if (!DIRECT && U.n_tiles == 0 && p.skip_empty) {  // real early exit: writes nothing
        U.live = false;
        return U;
    }
    const long long first = row_start(p, U.pos0);  // sliding window: skip leading tiles
    if (first > U.kb) {
        int skip = (int)((first - U.kb) / kBN);
        if (skip > U.n_tiles) skip = U.n_tiles;
        U.kb += skip * kBN;
        U.n_tiles -= skip;
    }
    return U;
}

// The unit of round i for CTA c of g (snake order), or -1 past the last unit.
__device__ __forceinline__ int unit_of_round(int i, int c, int g, int n_units) {
    const long long u = (long long)i * g + ((i & 1) ? g - 1 - c : c);
    return u < n_units ? (int)u : -1;
}

// The CTA's units of its first kTableRounds rounds, worked out once at the start by as
// many threads in parallel: looking a unit up needs the sequence's cu_seqlens, and a
// global load issued in the middle of the loop by the MMA thread (or the softmax warps)
// can wait thousands of cycles behind the CTA's own loads and stores.
constexpr int kTableRounds = 16;
struct PTable {
    PUnit unit[kTableRounds];
    int u[kTableRounds];  // unit index, -1 past the last unit
};

template <bool DIRECT>
__device__ __forceinline__ bool unit_of(const PTable &tab, const Problem &p, int i, int cta, int grid,
                                        int n_units, int n_mb, PUnit &U) {
    if (i < kTableRounds) {
        if (tab.u[i] < 0) return false;
        U = tab.unit[i];
        return true;
    }
    const int u = unit_of_round(i, cta, grid, n_units);
    if (u < 0) return false;
    U = unit_at<DIRECT>(p, u, n_mb);
    return true;
}

template <typename T, int DQK, int DV, bool DIRECT>
__global__ void __launch_bounds__(kPThreads, 1)
    partial_tc_persist_kernel(const __grid_constant__ CUtensorMap tmQ,
                              const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV, Problem p, float *o_part,
                              float *lse_part, TensorView out, float *lse_out, int n_mb,
                              int n_units) {
    using C = PCfg<DQK, DV>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    ptx::launch_dependents();  // the combine may be scheduled onto SMs this grid leaves idle

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, grid = gridDim.x;
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    const uint32_t sQ = (raw_u32 + 1023u) & ~1023u;
    const uint32_t sK = sQ + 2 * C::kQBytes;
    const uint32_t sV = sK + C::kKStages * C::kKBytes;
    const uint32_t sStage = sV + C::kVStages * C::kVBytes;
    const uint32_t bar0 = sStage + C::kStageBytes;
    uint8_t *const gen_base = smem_raw + (sQ - raw_u32);
    uint32_t *const tmem_holder = (uint32_t *)(gen_base + (bar0 - sQ) + C::kNumBars * 8);
    volatile int *const abort_flag = (volatile int *)(tmem_holder + 1);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    __shared__ PTable tab;
    if (threadIdx.x < kTableRounds) {
        const int u = unit_of_round(threadIdx.x, cta, grid, n_units);
        tab.u[threadIdx.x] = u;
        if (u >= 0) tab.unit[threadIdx.x] = unit_at<DIRECT>(p, u, n_mb);
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(C::kBarQF), 1);
        ptx::mbar_init(bar(C::kBarQE), 1);
        for (int i = 0; i < C::kKStages; ++i) {
            ptx::mbar_init(bar(C::kBarKF + i), 1);
            ptx::mbar_init(bar(C::kBarKE + i), 1);
        }
        for (int i = 0; i < C::kVStages; ++i) {
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
    if (warp == kPMmaWarp) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const bool dense = p.cu_q == nullptr;

    if (warp >= 8) {
        if (lane == 0 && (warp == kPKWarp || warp == kPVWarp || warp == kPQWarp)) {
            // ---------------------------------------------------------- TMA producers
            int quiet = 0;
            volatile int *no_abort = (volatile int *)&quiet;
            bool ok = true;
            int issued = 0;  // Q: units loaded; K / V: tiles loaded
            const CUtensorMap *map = warp == kPKWarp ? &tmK : (warp == kPVWarp ? &tmV : &tmQ);
            ptx::prefetch_tensormap(map);
            for (int i = 0; ok; ++i) {
                PUnit U;
                if (!unit_of<DIRECT>(tab, p, i, cta, grid, n_units, n_mb, U)) break;
                if (!U.live || U.n_tiles == 0) continue;
                const int cb = dense ? U.b : 0;
                if (warp == kPQWarp) {
                    if (issued > 0) {
                        ok = ptx::mbar_wait_bounded(bar(C::kBarQE), (issued - 1) & 1, abort_flag, p.err,
                                                    kErrProducer, kTimeoutNs);
                        if (!ok) break;
                    }
                    const int qrow = dense ? U.pos0 : U.si.q0 + U.pos0;
                    ptx::mbar_arrive_expect_tx(bar(C::kBarQF), 2 * C::kQBytes);
                    for (int t = 0; t < 2; ++t)
                        for (int c = 0; c < DQK / 64; ++c)
                            ptx::tma_load_4d(sQ + t * C::kQBytes + c * kChunkBytes, &tmQ, bar(C::kBarQF),
                                             c * 64, qrow + t * kTileM, U.h, cb);
                    ++issued;
                } else {
                    const bool isK = warp == kPKWarp;
                    const int stages = isK ? C::kKStages : C::kVStages;
                    const uint32_t base = isK ? sK : sV;
                    const uint32_t bytes = isK ? C::kKBytes : C::kVBytes;
                    const int full0 = isK ? C::kBarKF : C::kBarVF, empty0 = isK ? C::kBarKE : C::kBarVE;
                    const int d = isK ? DQK : DV;
                    const int krow = (dense ? 0 : U.si.k0) + U.kb;
                    for (int j = 0; j < U.n_tiles; ++j) {
                        const int st = issued % stages;
                        ok = ptx::mbar_wait_bounded(bar(empty0 + st), ((issued / stages) & 1) ^ 1, abort_flag,
                                                    p.err, kErrProducer, kTimeoutNs);
                        if (!ok) break;
                        ptx::mbar_arrive_expect_tx(bar(full0 + st), bytes);
                        for (int c = 0; c < d / 64; ++c)
                            ptx::tma_load_4d(base + st * bytes + c * kChunkBytes, map, bar(full0 + st), c * 64,
                                             krow + j * kBN, U.h, cb);
                        ++issued;
                    }
                }
            }
            if (!ok) {
                // drain: every load already issued must land before the CTA exits
                if (warp == kPQWarp) {
                    if (issued > 0)
                        ptx::mbar_wait_bounded(bar(C::kBarQF), (issued - 1) & 1, no_abort, nullptr, 0, kTimeoutNs);
                } else {
                    const int stages = warp == kPKWarp ? C::kKStages : C::kVStages;
                    const int full0 = warp == kPKWarp ? C::kBarKF : C::kBarVF;
                    for (int i = 0; i < stages && i < issued; ++i) {
                        const int last = i + ((issued - 1 - i) / stages) * stages;
                        ptx::mbar_wait_bounded(bar(full0 + i), (last / stages) & 1, no_abort, nullptr, 0,
                                               kTimeoutNs);
                    }
                }
            }
        } else if (warp == kPMmaWarp && lane == 0) {
            // -------------------------------------------------------------- MMA issuer
            constexpr uint32_t kIdescQK = ptx::idesc_f16(kBF16, false, false, kTileM, kBN);
            constexpr uint32_t kIdescPV = ptx::idesc_f16(kBF16, false, true, kTileM, DV);
            const uint32_t tS[2] = {tmem, tmem + 128u};
            const uint32_t tO[2] = {tmem + 256u, tmem + 384u};
            int kt = 0, vt = 0;  // K / V tiles consumed (ring position and phase)
            uint32_t g = 0;      // S / P phases used so far (the same for both tiles)
            int lu = 0;          // units with tiles so far (Q and O-done phases)
            bool ok = true;
            auto wait = [&](int b, uint32_t parity) {
                return ptx::mbar_wait_bounded(bar(b), parity, abort_flag, p.err, kErrMma, kTimeoutNs);
            };
            auto issue_qk = [&](int t, int ks) {
                const uint64_t kd = ptx::smem_desc_sw128(sK + ks * C::kKBytes, 16, 1024);
                const uint64_t qd = ptx::smem_desc_sw128(sQ + t * C::kQBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < DQK / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    ptx::mma_ss(tS[t], ptx::desc_advance(qd, off), ptx::desc_advance(kd, off), kIdescQK, kk > 0);
                }
                ptx::tc_commit(bar(C::kBarS + t));
            };
            auto issue_pv = [&](int t, int vs, bool first) {
                const uint64_t vd = ptx::smem_desc_sw128(sV + vs * C::kVBytes, C::kVPanelBytes, 1024);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    ptx::mma_ts(tO[t], tS[t] + kk * 8, ptx::desc_advance(vd, kk * 2048), kIdescPV,
                                (!first || kk > 0) ? 1u : 0u);
            };
            for (int i = 0; ok; ++i) {
                PUnit U;
                if (!unit_of<DIRECT>(tab, p, i, cta, grid, n_units, n_mb, U)) break;
                if (!U.live || U.n_tiles == 0) continue;
                const int n = U.n_tiles;
                ok = wait(C::kBarQF, lu & 1) && wait(C::kBarKF + kt % C::kKStages, (kt / C::kKStages) & 1);
                if (!ok) break;
                ptx::tc_fence_after();
                issue_qk(0, kt % C::kKStages);
                issue_qk(1, kt % C::kKStages);
                ptx::tc_commit(bar(C::kBarKE + kt % C::kKStages));
                ++kt;
                if (n == 1) ptx::tc_commit(bar(C::kBarQE));  // every S of the unit issued
                for (int j = 0; j < n && ok; ++j) {
                    const int vs = vt % C::kVStages;
                    ok = wait(C::kBarP + 0, (g + j) & 1) && wait(C::kBarVF + vs, (vt / C::kVStages) & 1);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    issue_pv(0, vs, j == 0);
                    if (j + 1 == n) ptx::tc_commit(bar(C::kBarO + 0));  // tile 0's epilogue may start
                    if (j + 1 < n) {
                        ok = wait(C::kBarKF + kt % C::kKStages, (kt / C::kKStages) & 1);
                        if (!ok) break;
                        ptx::tc_fence_after();
                        issue_qk(0, kt % C::kKStages);
                    }
                    ok = wait(C::kBarP + 1, (g + j) & 1);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    issue_pv(1, vs, j == 0);
                    ptx::tc_commit(bar(C::kBarVE + vs));  // V(j) is free
                    ++vt;
                    if (j + 1 < n) {
                        issue_qk(1, kt % C::kKStages);
                        ptx::tc_commit(bar(C::kBarKE + kt % C::kKStages));
                        ++kt;
                        if (j + 2 == n) ptx::tc_commit(bar(C::kBarQE));  // every S of the unit issued
                    }
                }
                if (!ok) break;
                ptx::tc_commit(bar(C::kBarO + 1));
                g += n;
                ++lu;
            }
            // every issued MMA must be finished before TMEM is released
            int dummy = 0;
            ptx::tc_commit(bar(C::kBarDrain));
            ptx::mbar_wait_bounded(bar(C::kBarDrain), 0, (volatile int *)&dummy, nullptr, 0, kTimeoutNs);
        }
    } else {
        // ---------------------------------------------------------------- softmax
        const int t = warp >> 2;
        const SoftmaxBars sb{bar(C::kBarS + t), bar(C::kBarP + t), bar(C::kBarO + t)};
        float4 *stage = (float4 *)(gen_base + (sStage - sQ)) + warp * 256;
        uint32_t g = 0;
        int lu = 0;
        for (int i = 0;; ++i) {
            PUnit U;
            if (!unit_of<DIRECT>(tab, p, i, cta, grid, n_units, n_mb, U)) break;
            if (!U.live) continue;
            const bool ok = softmax_rows<T, DV, DIRECT>(p, U.si, U.b, U.h, U.s, U.pos0, t, tmem, U.kb, U.ke,
                                                       U.n_tiles, sb, abort_flag, o_part, lse_part, out,
                                                       lse_out, stage, nullptr, nullptr, g, (uint32_t)(lu & 1));
            if (!ok) break;
            if (U.n_tiles > 0) {
                g += U.n_tiles;
                ++lu;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kPMmaWarp) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}
static_assert(kPLaunchRegs * kPThreads <= 65536, "launch registers");

template <typename T, int DQK, int DV, bool DIRECT>
static cudaError_t launch_persist(const Problem &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                  const CUtensorMap &mv, float *o_part, float *lse_part,
                                  const TensorView &out, float *lse_out, int ctas, cudaStream_t st) {
    using C = PCfg<DQK, DV>;
    auto kern = partial_tc_persist_kernel<T, DQK, DV, DIRECT>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
        attr_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    const int n_mb = (p.max_sq + kBM - 1) / kBM;
    const long long n_units = (long long)n_mb * p.H * p.B * p.S;
    if (n_units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int grid = (int)(n_units < ctas ? n_units : ctas);
    kern<<<grid, kPThreads, C::kSmemBytes, st>>>(mq, mk, mv, p, o_part, lse_part, out, lse_out, n_mb,
                                                 (int)n_units);
    return cudaGetLastError();
}

// Whether the persistent form takes this launch: head dims 64 or 128, M blocks of more
// than one 128-row tile, more units than SMs, and few key tiles per unit (an upper bound
// from max_seqlen_k, lastValid and the split count), where the fixed work of each unit
// outweighs its MMAs.
bool persist_fits(const Problem &p, int sm_count) {
    if (!((p.d_qk == 64 && p.d_v == 64) || (p.d_qk == 128 && p.d_v == 128))) return false;
    if (p.max_sq <= kTileM || p.bm != kBM) return false;
    const long long n_units = (long long)((p.max_sq + kBM - 1) / kBM) * p.H * p.B * p.S;
    if (n_units <= sm_count) return false;
    long long keys = p.max_sk;
    if (p.last_valid_kv_index >= 0 && p.last_valid_kv_index + 1LL < keys) keys = p.last_valid_kv_index + 1LL;
    const long long tiles_per_unit = (keys + (long long)p.S * kBN - 1) / ((long long)p.S * kBN);
    return tiles_per_unit <= kPersistMaxTiles;
}

cudaError_t launch_partial_tc_persist(const Problem &p, int dtype, const CUtensorMap &mq,
                                      const CUtensorMap &mk, const CUtensorMap &mv, float *o_part,
                                      float *lse_part, const TensorView *out, float *lse_out,
                                      int sm_count, cudaStream_t st) {
    const TensorView ov = out ? *out : TensorView{};
#define SK_P_LAUNCH(T, D)                                                                           \
    return out ? launch_persist<T, D, D, true>(p, mq, mk, mv, o_part, lse_part, ov, lse_out, sm_count, st) \
               : launch_persist<T, D, D, false>(p, mq, mk, mv, o_part, lse_part, ov, nullptr, sm_count, st);
    if (dtype == kBF16) {
        if (p.d_qk == 128) { SK_P_LAUNCH(__nv_bfloat16, 128) }
        SK_P_LAUNCH(__nv_bfloat16, 64)
    }
    if (p.d_qk == 128) { SK_P_LAUNCH(__half, 128) }
    SK_P_LAUNCH(__half, 64)
#undef SK_P_LAUNCH
}

}  // namespace tc
}  // namespace sk
