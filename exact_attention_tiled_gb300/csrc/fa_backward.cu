// fa_backward.cu -- gradients of exact attention on sm_103a tensor cores.
//
// What is computed ("Infra: Flash Attention", "Backward and recomputation"
// and "Blocked gradient computation"; CMU 10-423 Lecture 18, 5.3): with the
// forward's per-row log-sum-exp L and the upstream gradient dO,
//
//   P_ij  = exp(S_ij - L_i),  S = scale Q K^T      (recomputed tile by tile)
//   dP_ij = dO_i . V_j
//   D_i   = dO_i . O_i        (= sum_j P_ij dP_ij, so no pass over P)
//   dS_ij = P_ij (dP_ij - D_i)
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K
//
// Two kernels, no N x N matrix in global memory:
//   * bwd_pre_kernel: D = rowsum(dO o O) in fp32 (bandwidth bound).
//   * bwd_main_kernel: one grid of two kinds of CTA, which need only D and
//     so run side by side (the dQ CTAs fill the SMs the dK/dV CTAs leave idle
//     in their last wave):
//   * dK/dV CTAs: one per 128-key tile j of one (b, h).  K_j and V_j
//     stay in shared memory (at d = 64 also in TMEM, the A operands of the
//     S^T and dP^T products); the query tiles i stream through a ring together
//     with their dO_i, L_i and D_i.  Per half of a query tile (64 queries) the
//     tensor core forms S^T = K_j Q_i^T and dP^T = V_j dO_i^T in TMEM (keys on
//     the 128 TMEM lanes, queries on the columns); two compute warpgroups turn
//     them into P^T and dS^T (bf16, packed over the first half of each
//     warpgroup's columns), and the tensor core accumulates dV += P^T dO_i and
//     dK += dS^T Q_i in TMEM with A read straight from TMEM.  Each half has its
//     own TMEM buffer, so one half's exponentials overlap the other half's
//     products.  dV, dK leave once, at the end.
//   * dQ CTAs: one per 128-query tile i, the same half-step scheme
//     over key tiles: S = Q_i K_j^T and dP = dO_i V_j^T, dS in the compute
//     warpgroups, and dQ += dS K_j in TMEM.  Computing dQ in its own pass
//     (recomputing S and dP) keeps every gradient element written by exactly
//     one CTA: no atomics, and the result does not depend on scheduling.
// The dQ-accumulating variant (fa_backward_atomic_dq, d = 64) runs dK/dV
// CTAs only: each also forms dQ_i += dS_i K_j for every query tile it meets
// (dS^T copied to shared memory as the A operand) and adds it into an fp32
// dQ through TMA reductions; a last kernel scales and rounds it.  Less work,
// but the order of the fp32 additions depends on scheduling.
// Warp roles in both kinds of CTA (640 threads): warp 0 lane 0 issues the
// TMA copies, warp 1 is the MMA warp (converged, one elected lane issues),
// warps 4-19 are four compute warpgroups, one thread per TMEM lane (tile row);
// in the dQ variant warp 2 lane 0 issues the reductions.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_tmap.h"

namespace fa {
namespace {

constexpr int BT = 128;              // rows of a query or key tile (MMA M and N)
// warp 0 producer, warp 1 MMA, warps 2-3 idle, then four compute warpgroups that
// take 32 columns each of every step (query columns in the dK/dV kernel, key
// columns in the dQ kernel); warpgroups 2 hf and 2 hf + 1 serve half-step hf
constexpr int kComputeGroups = 4;
constexpr int kBwdThreads = 128 * (1 + kComputeGroups);
constexpr int kProd = 0, kMma = 1, kDqWarp = 2, kFirstCompute = 4;
constexpr float kLog2e = 1.4426950408889634f;

enum {
    kSiteBwKV = 0x401, kSiteBwQD = 0x402, kSiteBwS = 0x403, kSiteBwP = 0x404, kSiteBwDone = 0x405,
    kSiteBwEmpty = 0x406, kSiteBwDrain = 0x407, kSiteBwDqFree = 0x408, kSiteBwDqd = 0x409, kSiteBwStage = 0x40a
};

struct BwdMaps {
    CUtensorMap q, k, v, dO, dq, dk, dv;
    CUtensorMap dqa;   // fp32 dQ accumulator (the dQ-accumulating variant only)
};

// Row r, 16-byte chunk kc (8 bf16 columns) of a 128-row tile in the 128-byte
// swizzled layout of the tensor maps (64-column blocks of 128 x 128 bytes).
__device__ __forceinline__ uint32_t swz_chunk(uint32_t tile, int r, int kc) {
    return tile + (kc >> 3) * (BT * 128) + r * 128 + (static_cast<uint32_t>((kc & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ bool wait_abort(uint32_t bar, uint32_t parity, unsigned *err, int site,
                                           volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            report_timeout(err, site);
            *abort_flag = 1;
            return false;
        }
    }
}

// converged-warp form: every lane polls, the result is warp-uniform
__device__ __forceinline__ bool wait_abort_warp(uint32_t bar, uint32_t parity, unsigned *err, int site,
                                                volatile int *abort_flag) {
    return __all_sync(0xffffffffu, wait_abort(bar, parity, err, site, abort_flag));
}

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Row r of a 128-row bf16 tile held in shared memory in the tensor maps' 128-byte
// swizzled layout (16-byte chunk c of row r at c ^ (r & 7)) into this thread's TMEM
// lane as packed bf16 pairs, D / 2 columns from taddr: the row becomes the A operand
// of TS products.  Called by one full warpgroup, thread r of the tile on lane r.
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t *tile, int r, uint32_t taddr) {
#pragma unroll
    for (int cb = 0; cb < D / 64; ++cb) {
        const uint8_t *row = tile + cb * (BT * 128) + r * 128;
        uint32_t wv[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(row + ((c ^ (r & 7)) << 4));
            wv[4 * c] = v.x;
            wv[4 * c + 1] = v.y;
            wv[4 * c + 2] = v.z;
            wv[4 * c + 3] = v.w;
        }
        tmem_st32(taddr + cb * 32, wv);
    }
    tmem_wait_st();
}

template <int D, int Stages = 2>
struct BwdCfg {
    static constexpr int kColBlocks = D / 64;
    static constexpr int kTileBytes = BT * D * 2;
    static constexpr int kStages = Stages;
    // dkdv: K, V, then per stage {Q_i, dO_i}, then per stage {L_i * log2 e, D_i}
    // dq:   Q, dO, then per stage {K_j, V_j}
    static constexpr int kFixedOff = 0;
    static constexpr int kStageOff = 2 * kTileBytes;
    static constexpr int kVecOff = kStageOff + kStages * 2 * kTileBytes;
    static constexpr int kBarOff = kVecOff + kStages * 2 * BT * 4;
    static constexpr int kNumBars = 20;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // at least 120 KB, so one CTA per SM: each allocates all 512 TMEM columns
    static constexpr int kSmemUsed = kMiscOff + 16 + 1024;
    static constexpr int kSmemBytes = kSmemUsed > 120 * 1024 ? kSmemUsed : 120 * 1024;
};

// The dQ-accumulating variant of the dK/dV CTA (d = 64) adds two shared buffers of
// dS^T for a query tile (128 keys x 128 queries bf16, as the A operand of dQ = dS K:
// queries contiguous, two 64-query column blocks of 128 x 128 bytes), after the
// CTA's other shared state.
template <int D>
struct AtomicDqShape {
    using C = BwdCfg<D, 3>;
    static constexpr int kDsBytes = BT * BT * 2;
    static constexpr int kDsOff = (C::kMiscOff + 16 + 1023) / 1024 * 1024;
    static constexpr int kSmemBytes = kDsOff + 2 * kDsBytes + 1024;
    static_assert(D != 64 || kSmemBytes <= 227 * 1024, "shared memory per CTA");   // used at d = 64 only
};

// Both main kernels run a step (one 128-row tile of the streamed operand) as two
// half-steps of 64 columns.  TMEM holds kHalfBufs half-step buffers of 128
// columns (S half, then dP half) and then the accumulators; at d = 64 there is
// room for three buffers, at d = 128 for two (the dK/dV kernel trades the
// third for K_j and V_j, see dkdv_cta).  The streamed ring has one stage
// more at d = 64 (shared memory allows it), so the deeper lookahead does not
// wait on its loads.
template <int D>
struct HalfStepShape {
    static constexpr int kHalfBufs = D == 64 ? 3 : 2;
    static constexpr int kStages = D == 64 ? 3 : 2;
    static constexpr uint32_t kColAccum = 128u * kHalfBufs;   // dV; dK at + D
};

// ---------------------------------------------------------------------------
// D_i = sum_c dO_ic O_ic.  D/8 lanes per row, one 16-byte vector each.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16 *O, const __nv_bfloat16 *dO,
                                                      float *Dout, long long rows) {
    constexpr int LPR = D / 8;
    const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long row = gtid / LPR;
    const int part = static_cast<int>(gtid % LPR);
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = *reinterpret_cast<const uint4 *>(O + row * D + part * 8);
        const uint4 b = *reinterpret_cast<const uint4 *>(dO + row * D + part * 8);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(__uint_as_float(wa[i] << 16), __uint_as_float(wb[i] << 16), acc);
            acc = fmaf(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(wb[i] & 0xFFFF0000u), acc);
        }
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0) Dout[row] = acc;
    grid_launch_dependents();
}

// ---------------------------------------------------------------------------
// dK, dV of key tile jt of (batch, head) bh: one CTA (key tile 0 is the
// heaviest under causal masking: key tile j meets the query tiles i >= j).
// ---------------------------------------------------------------------------
// kAtomicDQ (d = 64 only): the CTA also forms dQ_i += dS_i K_j for every query tile
// it meets and adds it into the fp32 accumulator p.dq_accum with TMA reductions
// (through tm.dqa), so no dQ CTAs run.
template <int D, bool kAtomicDQ = false>
__device__ __forceinline__ void dkdv_cta(const BwdMaps &tm, const BwdParams &p, const int bh, const int jt) {
    using C = BwdCfg<D, HalfStepShape<D>::kStages>;
    static_assert(!kAtomicDQ || D == 64, "the dQ accumulator fits in TMEM at d = 64 only");
    // At d = 64 this kernel keeps two half-step buffers and copies K_j and V_j into
    // TMEM (packed bf16 rows, one key per lane), so S^T = K Q_h^T and dP^T = V dO_h^T
    // are TS products that read only Q_h and dO_h from shared memory (measured: d = 64
    // backward +0.7 % against three buffers and SS products).  At d = 128 the
    // accumulators leave no room: both operands come from shared memory.
    constexpr bool kKvTmem = D == 64;
    constexpr int NB = kKvTmem ? 2 : HalfStepShape<D>::kHalfBufs;
    constexpr uint32_t kColGrad = 128u * NB;
    constexpr uint32_t kColK = kColGrad + 2 * D, kColV = kColK + D / 2;
    static_assert(!kKvTmem || kColV + D / 2 <= 512, "TMEM columns");
    // dQ partial of the current query tile (queries on the lanes), after K_j and V_j
    constexpr uint32_t kColDq = kColV + D / 2;
    static_assert(!kAtomicDQ || kColDq + D <= 512, "TMEM columns");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t k_smem = sbase + C::kFixedOff, v_smem = k_smem + C::kTileBytes;
    auto q_stage = [&](int s) { return sbase + C::kStageOff + s * 2 * C::kTileBytes; };
    auto do_stage = [&](int s) { return q_stage(s) + C::kTileBytes; };
    float *vec = reinterpret_cast<float *>(smem + C::kVecOff);   // [stage][2][BT]: L*log2e, D
    const uint32_t bars = sbase + C::kBarOff;
    const uint32_t bar_kv = bars;
    auto bar_full = [&](int s) { return bars + 8u * (1 + s); };
    auto bar_empty = [&](int s) { return bars + 8u * (1 + C::kStages + s); };
    // Half-step u = 2n + hf covers query rows [64 hf, 64 hf + 64) of query tile
    // i_lo + n and uses TMEM buffer u % NB.  bar_st(b): S^T, dP^T of the buffer's
    // half-step are in TMEM; bar_ps(b): its two warpgroups have written P^T, dS^T.
    // A buffer's barriers complete once per use, and the next use is issued only
    // after the MMA warp saw bar_ps of the previous one, so no phase goes unseen.
    auto bar_st = [&](int bf) { return bars + 8u * (1 + 2 * C::kStages + bf); };
    auto bar_ps = [&](int bf) { return bars + 8u * (1 + 2 * C::kStages + NB + bf); };
    const uint32_t bar_done = bars + 8u * (1 + 2 * C::kStages + 2 * NB);
    const uint32_t bar_ktm = bar_done + 8u;   // K_j, V_j are in TMEM
    // dQ variant: bar_dqd(b) -- the dQ products of a query tile n with n % 2 == b are
    // complete; bar_dq_free -- every compute warp has read the previous tile's dQ out
    // of TMEM; bar_stage_full -- every compute warp has staged the tile's dQ (fp32)
    // in the tile's dS buffer; bar_stage_free(b) -- the reduction of the staged dQ
    // of the last tile that used buffer b has read it
    auto bar_dqd = [&](int b) { return bar_ktm + 8u * (1 + b); };
    const uint32_t bar_dq_free = bar_ktm + 24u;
    const uint32_t bar_stage_full = bar_ktm + 32u;
    auto bar_stage_free = [&](int b) { return bar_ktm + 8u * (5 + b); };
    static_assert(1 + 2 * C::kStages + 2 * NB + 2 + (kAtomicDQ ? 6 : 0) <= C::kNumBars, "barrier slots");
    auto ds_buf = [&](int b) { return sbase + AtomicDqShape<D>::kDsOff + b * AtomicDqShape<D>::kDsBytes; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = bh / p.H;
    const int N = p.N;
    const int T = (N + BT - 1) / BT;
    int klen = N;
    if (p.key_len) klen = clampi(p.key_len[b], 0, N);
    const int key0 = jt * BT;
    // query tiles this key tile meets; none when every key of the tile is masked
    const int i_lo = p.causal ? jt : 0;
    const int nsteps = key0 < klen ? T - i_lo : 0;

    if (threadIdx.x == 0) {
        mbar_init(bar_kv, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar_full(s), 2);    // TMA bytes + the producer warp's L/D stores
            mbar_init(bar_empty(s), 1);
        }
        for (int bf = 0; bf < NB; ++bf) {
            mbar_init(bar_st(bf), 1);
            mbar_init(bar_ps(bf), 8);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_ktm, 8);
        if (kAtomicDQ) {
            mbar_init(bar_dqd(0), 1);
            mbar_init(bar_dqd(1), 1);
            mbar_init(bar_dq_free, 16);
            mbar_init(bar_stage_full, 16);
            mbar_init(bar_stage_free(0), 1);
            mbar_init(bar_stage_free(1), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProd) {
        // ================================================= producer warp
        bool ok = true;
        if (nsteps > 0) {
            if (lane == 0) {
                prefetch_tmap(&tm.q);
                prefetch_tmap(&tm.k);
                prefetch_tmap(&tm.v);
                prefetch_tmap(&tm.dO);
                const uint64_t pol = l2_policy_evict_normal();
                mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes);
#pragma unroll
                for (int cb = 0; cb < C::kColBlocks; ++cb) {
                    tma_load_3d(k_smem + cb * (BT * 128), &tm.k, cb * 64, key0, bh, bar_kv, pol);
                    tma_load_3d(v_smem + cb * (BT * 128), &tm.v, cb * 64, key0, bh, bar_kv, pol);
                }
            }
            // D comes from bwd_pre_kernel, which this grid may overlap (programmatic
            // dependent launch): wait for it before the first read
            grid_dependency_wait();
            for (int n = 0; n < nsteps && ok; ++n) {
                const int s = n % C::kStages;
                const int i = i_lo + n;
                // L_i * log2(e) and D_i of this query tile, loaded before the stage
                // wait so their latency hides behind it (rows past N: never used)
                float lreg[BT / 32], dreg[BT / 32];
#pragma unroll
                for (int e = 0; e < BT / 32; ++e) {
                    const int q = i * BT + e * 32 + lane;
                    const size_t idx = static_cast<size_t>(bh) * N + (q < N ? q : 0);
                    lreg[e] = p.L[idx] * kLog2e;
                    dreg[e] = p.Dvec[idx];
                }
                if (n >= C::kStages)
                    ok = __all_sync(0xffffffffu, wait_abort(bar_empty(s), ((n / C::kStages) - 1) & 1, p.err,
                                                             kSiteBwEmpty, abort_flag));
                if (!ok) break;
                if (lane == 0) {
                    const uint64_t pol = l2_policy_evict_normal();
                    mbar_arrive_expect_tx(bar_full(s), 2 * C::kTileBytes);
#pragma unroll
                    for (int cb = 0; cb < C::kColBlocks; ++cb) {
                        tma_load_3d(q_stage(s) + cb * (BT * 128), &tm.q, cb * 64, i * BT, bh, bar_full(s), pol);
                        tma_load_3d(do_stage(s) + cb * (BT * 128), &tm.dO, cb * 64, i * BT, bh, bar_full(s), pol);
                    }
                }
                float *lv = vec + s * 2 * BT;
#pragma unroll
                for (int e = 0; e < BT / 32; ++e) {
                    lv[e * 32 + lane] = lreg[e];
                    lv[BT + e * 32 + lane] = dreg[e];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_full(s));
            }
            // no copy may be in flight when the CTA exits
            if (lane == 0) {
                mbar_wait(bar_kv, 0, p.err, kSiteBwDrain);
                const int first = nsteps > C::kStages ? nsteps - C::kStages : 0;
                for (int n = first; n < nsteps; ++n)
                    mbar_wait(bar_full(n % C::kStages), (n / C::kStages) & 1, p.err, kSiteBwDrain);
            }
        }
    } else if (warp == kMma) {
        // ================================================= MMA warp
        if (nsteps > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BT, BT / 2, 0, 0);   // M 128 keys, N 64 queries
            constexpr uint32_t idesc_g = idesc_bf16_f32(BT, D, 0, 1);
            const int nhalf = 2 * nsteps;
            bool ok = wait_abort_warp(kKvTmem ? bar_ktm : bar_kv, 0, p.err, kSiteBwKV, abort_flag);
            const uint64_t kd = sdesc_sw128(k_smem, 16, 1024), vd = sdesc_sw128(v_smem, 16, 1024);
            // S^T = K Q_h^T and dP^T = V dO_h^T into buffer u % NB (K-major A and B; the
            // half's 64 query rows start 8 swizzle atoms into each column block).  The
            // first half of a step waits for its Q_i, dO_i stage.
            auto issue_sdp = [&](int u) {
                const int hf = u & 1, n = u >> 1, s = n % C::kStages;
                const uint32_t col = 128u * (u % NB);
                if (hf == 0) {
                    if (!wait_abort_warp(bar_full(s), (n / C::kStages) & 1, p.err, kSiteBwQD, abort_flag))
                        return false;
                    tc_fence_after();
                }
                const uint32_t rows = hf * (BT / 2) * 128;
                const uint64_t qd = sdesc_sw128(q_stage(s) + rows, 16, 1024);
                const uint64_t od = sdesc_sw128(do_stage(s) + rows, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * (BT * 128) + (kk & 3) * 32) >> 4;
                    if constexpr (kKvTmem)
                        mma_ts_warp(tmem + col, tmem + kColK + kk * 8, qd + off, idesc_s, kk > 0 ? 1u : 0u);
                    else
                        mma_ss_warp(tmem + col, kd + off, qd + off, idesc_s, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * (BT * 128) + (kk & 3) * 32) >> 4;
                    if constexpr (kKvTmem)
                        mma_ts_warp(tmem + col + 64, tmem + kColV + kk * 8, od + off, idesc_s, kk > 0 ? 1u : 0u);
                    else
                        mma_ss_warp(tmem + col + 64, vd + off, od + off, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar_st(u % NB));
                return true;
            };
            // dV += P^T dO_h, dK += dS^T Q_h: A from TMEM (warpgroup 2 hf + w packed its 32
            // query columns into the first 16 of its own 32), B MN-major (d contiguous)
            auto issue_grad = [&](int u) {
                const int hf = u & 1, s = (u >> 1) % C::kStages;
                const uint32_t col = 128u * (u % NB);
                const uint64_t odm = sdesc_sw128(do_stage(s), BT * 128, 1024);
                const uint64_t qdm = sdesc_sw128(q_stage(s), BT * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acol = col + (kk >> 1) * 32 + (kk & 1) * 8;
                    const uint32_t boff = ((hf * 4 + kk) * 2048) >> 4;   // 16 query rows per step
                    mma_ts_warp(tmem + kColGrad, tmem + acol, odm + boff, idesc_g, (u > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acol = col + 64 + (kk >> 1) * 32 + (kk & 1) * 8;
                    const uint32_t boff = ((hf * 4 + kk) * 2048) >> 4;
                    mma_ts_warp(tmem + kColGrad + D, tmem + acol, qdm + boff, idesc_g, (u > 0 || kk > 0) ? 1u : 0u);
                }
            };
            for (int u = 0; u < NB && u < nhalf && ok; ++u) ok = issue_sdp(u);
            // The tensor core runs one thread's MMAs in issue order: S^T/dP^T of half-step
            // u + NB overwrite the buffer that dV/dK of half-step u read just before.
            for (int u = 0; u < nhalf && ok; ++u) {
                ok = wait_abort_warp(bar_ps(u % NB), (u / NB) & 1, p.err, kSiteBwP, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_grad(u);
                if (u & 1) mma_commit_warp(bar_empty((u >> 1) % C::kStages));   // Q_i, dO_i read
                if (u + NB < nhalf) ok = issue_sdp(u + NB);
                if constexpr (kAtomicDQ) {
                    if ((u & 1) && ok) {
                        // dQ_i (queries on the lanes) = dS_i K_j: A = dS^T of both halves from
                        // shared memory (published by the two ps barriers), MN-major; B = K_j,
                        // d contiguous.  The TMEM accumulator is free once every compute warp
                        // has read the previous tile's.
                        const int n = u >> 1;
                        if (n > 0) ok = wait_abort_warp(bar_dq_free, (n - 1) & 1, p.err, kSiteBwDqFree, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        constexpr uint32_t idesc_dq = idesc_bf16_f32(BT, D, 1, 1);
                        const uint64_t ad = sdesc_sw128(ds_buf(n & 1), BT * 128, 1024);
                        const uint64_t bd = sdesc_sw128(k_smem, BT * 128, 1024);
#pragma unroll
                        for (int kk = 0; kk < BT / 16; ++kk) {
                            const uint32_t off = (kk * 2048) >> 4;   // 16 key rows
                            mma_ss_warp(tmem + kColDq, ad + off, bd + off, idesc_dq, kk > 0 ? 1u : 0u);
                        }
                        mma_commit_warp(bar_dqd(n & 1));
                    }
                }
            }
            // every MMA has completed before the gradients are read and TMEM is freed
            mma_commit_warp(bar_done);
            mbar_wait(bar_done, 0, p.err, kSiteBwDone);
            __syncwarp();
        }
    } else if (kAtomicDQ && warp == kDqWarp) {
        // ================================================= dQ reduction warp (dQ variant)
        // Once every compute warp has staged query tile m's dQ partial, add it into the
        // fp32 accumulator (rows past N are skipped by the tensor map) and release the
        // buffer as soon as the reduction has read it.
        if (lane == 0 && nsteps > 0) {
            prefetch_tmap(&tm.dqa);
            for (int m = 0; m < nsteps; ++m) {
                if (!wait_abort(bar_stage_full, m & 1, p.err, kSiteBwStage, abort_flag)) break;
                const uint32_t stg = ds_buf(m & 1);
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb)
                    tma_reduce_add_3d(&tm.dqa, stg + cb * (BT * 128), cb * 32, (i_lo + m) * BT, bh);
                bulk_commit_group();
                bulk_wait_group_read0();
                mbar_arrive(bar_stage_free(m & 1));
            }
            // every addition has reached global memory before the CTA exits
            bulk_wait_group0();
        }
    } else if (warp >= kFirstCompute) {
        // ================================================= compute warpgroups
        // warpgroup h handles query columns [32h, 32h + 32) of every step, one
        // thread per key row (TMEM lane)
        const int h = (warp - kFirstCompute) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;      // key row of the tile
        const int key = key0 + r;
        const bool key_ok = key < klen;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        const float2 sl22 = make_float2(sl2, sl2);
        bool ok = true;
        const int hf = h >> 1;   // the half of every step this warpgroup serves
        const int w = h & 1;     // its 32 columns within the half
        if (kKvTmem && h < 2 && nsteps > 0) {
            // warpgroup 0 copies this thread's row of K_j, warpgroup 1 its row of V_j,
            // from the swizzled shared tile into TMEM as packed bf16 pairs
            ok = wait_abort_warp(bar_kv, 0, p.err, kSiteBwKV, abort_flag);
            if (ok)
                tile_row_to_tmem<D>(smem + C::kFixedOff + h * C::kTileBytes, r, tmem + lane_off + (h ? kColV : kColK));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ktm);
        }
        // dQ variant: this thread's 16 columns (16 h ..) of query tile m's dQ partial, on
        // its lane (query row r of the tile), staged as fp32 in the tile's dS buffer (the
        // dQ products are done with it) in the 128-byte swizzled layout of the
        // accumulator's tensor map; warp kDqWarp adds the staged tile into p.dq_accum
        auto dq_readout = [&](int m) -> bool {
            if (!wait_abort_warp(bar_dqd(m & 1), (m >> 1) & 1, p.err, kSiteBwDqd, abort_flag)) return false;
            tc_fence_after();
            __syncwarp();
            uint32_t a[16];
            tmem_ld16(tmem + lane_off + kColDq + 16 * h, a);
            tmem_wait_ld();
            reg_fence(a);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_dq_free);
            const uint32_t stg = ds_buf(m & 1) + (h >> 1) * (BT * 128);   // 32 fp32 columns per block
#pragma unroll
            for (int v = 0; v < 4; ++v)
                st_shared_v4(swz_chunk(stg, r, 4 * (h & 1) + v), a[4 * v], a[4 * v + 1], a[4 * v + 2], a[4 * v + 3]);
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_stage_full);
            return true;
        };
        for (int n = 0; n < nsteps && ok; ++n) {
            const int s = n % C::kStages;
            const int q0 = (i_lo + n) * BT;
            const int u = 2 * n + hf;
            const uint32_t col = 128u * (u % NB) + 32u * w;
            ok = wait_abort_warp(bar_st(u % NB), (u / NB) & 1, p.err, kSiteBwS, abort_flag);
            // the producer warp's L_i / D_i stores are published by the stage's
            // full barrier (already complete here: the MMAs behind bar_st waited on it)
            if (ok) ok = wait_abort_warp(bar_full(s), (n / C::kStages) & 1, p.err, kSiteBwQD, abort_flag);
            if (!ok) break;
            tc_fence_after();
            __syncwarp();
            const float *lv = vec + s * 2 * BT;     // L_i * log2 e
            const float *dv = lv + BT;              // D_i
            // masking only where the tile touches key_len, the sequence end or the diagonal
            const bool need_mask = key0 + BT > klen || q0 + BT > N || (p.causal && key0 + BT - 1 > q0);
            // P^T and dS^T of half hb (16 columns) of the 32-column chunk c from its S^T
            // and dP^T values, into words 8 hb .. 8 hb + 7 of pp and dp
            auto half = [&](int c, int hb, uint32_t (&sr)[16], const uint32_t (&dr)[16], uint32_t (&pp)[16],
                            uint32_t (&dp)[16]) {
                if (need_mask) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int q = q0 + c * 32 + hb * 16 + e;
                        if (!(key_ok && q < N && (!p.causal || key <= q))) sr[e] = __float_as_uint(-INFINITY);
                    }
                }
                const float4 *l4 = reinterpret_cast<const float4 *>(lv + c * 32 + hb * 16);
                const float4 *d4 = reinterpret_cast<const float4 *>(dv + c * 32 + hb * 16);
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    const float4 lq = l4[e >> 2], dq = d4[e >> 2];
                    const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl22,
                                                 make_float2(-lq.x, -lq.y));
                    const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])),
                                                 sl22, make_float2(-lq.z, -lq.w));
                    const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y)), p1 = make_float2(ex2(x1.x), ex2(x1.y));
                    const float2 g0 =
                        __fmul2_rn(p0, make_float2(__uint_as_float(dr[e]) - dq.x, __uint_as_float(dr[e + 1]) - dq.y));
                    const float2 g1 =
                        __fmul2_rn(p1, make_float2(__uint_as_float(dr[e + 2]) - dq.z, __uint_as_float(dr[e + 3]) - dq.w));
                    pp[8 * hb + (e >> 1)] = pack_bf16(p0.x, p0.y);
                    pp[8 * hb + (e >> 1) + 1] = pack_bf16(p1.x, p1.y);
                    dp[8 * hb + (e >> 1)] = pack_bf16(g0.x, g0.y);
                    dp[8 * hb + (e >> 1) + 1] = pack_bf16(g1.x, g1.y);
                }
            };
            // this warpgroup's S^T and dP^T columns, in two halves of 16 so that only
            // half of them is live at once (the second half loads while the first is
            // computed); P^T and dS^T are packed over the first 16 of the 32 columns
            uint32_t sa[16], da[16], sb[16], db[16];
            tmem_ld16(tmem + lane_off + col, sa);
            tmem_ld16(tmem + lane_off + col + 64, da);
            tmem_wait_ld();
            reg_fence(sa);
            reg_fence(da);
            tmem_ld16(tmem + lane_off + col + 16, sb);
            tmem_ld16(tmem + lane_off + col + 64 + 16, db);
            uint32_t pp[16], dp[16];
            half(h, 0, sa, da, pp, dp);
            tmem_wait_ld();
            reg_fence(sb);
            reg_fence(db);
            half(h, 1, sb, db, pp, dp);
            tmem_st16(tmem + lane_off + col, pp);
            tmem_st16(tmem + lane_off + col + 64, dp);
            if constexpr (kAtomicDQ) {
                // dS^T row r, query columns 32 h .. 32 h + 31, into this tile's shared dS
                // buffer, for the dQ products (the ps arrive below publishes it to them);
                // the buffer last held tile n - 2's staged dQ, whose reduction must have read it
                if (n >= 2 && !wait_abort_warp(bar_stage_free(n & 1), ((n - 2) >> 1) & 1, p.err, kSiteBwStage,
                                               abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t dsb = ds_buf(n & 1) + (h >> 1) * (BT * 128);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_shared_v4(swz_chunk(dsb, r, 4 * (h & 1) + c), dp[4 * c], dp[4 * c + 1], dp[4 * c + 2],
                                 dp[4 * c + 3]);
                fence_proxy_async_shared();
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ps(u % NB));
            if constexpr (kAtomicDQ) {
                if (n > 0 && !dq_readout(n - 1)) {
                    ok = false;
                    break;
                }
            }
        }
        if constexpr (kAtomicDQ) {
            if (ok && nsteps > 0) ok = dq_readout(nsteps - 1);
        }
        // ---- epilogue: dV and dK (x scale) to bf16; keys with no step get zeros
        if (ok && nsteps > 0) {
            ok = wait_abort_warp(bar_done, 0, p.err, kSiteBwDone, abort_flag);
            tc_fence_after();
            __syncwarp();
        }
        // dV and dK are staged in the shared tiles K_j and V_j held (free once
        // bar_done completed) and leave by TMA stores after the CTA's last barrier:
        // one thread per key row storing its own row to global memory would touch
        // 32 cache lines per store instruction.  Rows past N are clipped by the store.
        if (ok) {
            {
                // warpgroups 0, 1 stage the two column halves of dV, warpgroups 2, 3 of dK
                const int which = h >> 1;
                const uint32_t stage = which ? k_smem : v_smem;
                const float mul = which ? p.scale : 1.f;
#pragma unroll 1
                for (int c = (h & 1) * (D / 64); c < (h & 1) * (D / 64) + D / 64; ++c) {
                    uint32_t a[32];
                    if (nsteps > 0) {
                        tmem_ld32(tmem + lane_off + kColGrad + which * D + c * 32, a);
                        tmem_wait_ld();
                        reg_fence(a);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) a[e] = 0u;
                    }
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        st_shared_v4(swz_chunk(stage, r, c * 4 + v),
                                     pack_bf16(__uint_as_float(a[8 * v]) * mul, __uint_as_float(a[8 * v + 1]) * mul),
                                     pack_bf16(__uint_as_float(a[8 * v + 2]) * mul, __uint_as_float(a[8 * v + 3]) * mul),
                                     pack_bf16(__uint_as_float(a[8 * v + 4]) * mul, __uint_as_float(a[8 * v + 5]) * mul),
                                     pack_bf16(__uint_as_float(a[8 * v + 6]) * mul, __uint_as_float(a[8 * v + 7]) * mul));
                    __syncwarp();   // reconverge before the next warp-collective load
                }
            }
            fence_proxy_async_shared();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && !*abort_flag) {
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) {
            tma_store_3d(&tm.dv, v_smem + cb * (BT * 128), cb * 64, key0, bh);
            tma_store_3d(&tm.dk, k_smem + cb * (BT * 128), cb * 64, key0, bh);
        }
        bulk_commit_group();
        bulk_wait_group0();
    }
    if (warp == kMma) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// dQ of query tile rank `rank` of (batch, head) bh: one CTA; rank 0 is the
// last query tile, the heaviest under causal masking (query tile i meets the
// key tiles j <= i).
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void dq_cta(const BwdMaps &tm, const BwdParams &p, const int bh, const int rank) {
    using C = BwdCfg<D, HalfStepShape<D>::kStages>;
    constexpr int NB = HalfStepShape<D>::kHalfBufs;
    constexpr uint32_t kColGrad = HalfStepShape<D>::kColAccum;
    // Q_i and dO_i stay in TMEM as packed bf16 rows (one query per lane): the A
    // operands of S = Q K^T and dP = dO V^T, so those products read only K and V
    // from shared memory
    constexpr uint32_t kColQ = kColGrad + D, kColDO = kColQ + D / 2;
    static_assert(kColDO + D / 2 <= 512, "TMEM columns");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t q_smem = sbase + C::kFixedOff, do_smem = q_smem + C::kTileBytes;
    auto k_stage = [&](int s) { return sbase + C::kStageOff + s * 2 * C::kTileBytes; };
    auto v_stage = [&](int s) { return k_stage(s) + C::kTileBytes; };
    const uint32_t bars = sbase + C::kBarOff;
    const uint32_t bar_qd = bars;
    auto bar_full = [&](int s) { return bars + 8u * (1 + s); };
    auto bar_empty = [&](int s) { return bars + 8u * (1 + C::kStages + s); };
    // half-step u = 2n + hf: key rows [64 hf, 64 hf + 64) of key tile n, TMEM buffer
    // u % NB; the barriers follow the dK/dV kernel's
    auto bar_st = [&](int bf) { return bars + 8u * (1 + 2 * C::kStages + bf); };
    auto bar_ps = [&](int bf) { return bars + 8u * (1 + 2 * C::kStages + NB + bf); };
    const uint32_t bar_done = bars + 8u * (1 + 2 * C::kStages + 2 * NB);
    const uint32_t bar_qtm = bars + 8u * (2 + 2 * C::kStages + 2 * NB);   // Q_i, dO_i are in TMEM
    static_assert(2 + 2 * C::kStages + 2 * NB + 1 <= C::kNumBars, "barrier slots");
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = bh / p.H;
    const int N = p.N;
    const int T = (N + BT - 1) / BT;
    const int it = T - 1 - rank;
    const int q0 = it * BT;
    int klen = N;
    if (p.key_len) klen = clampi(p.key_len[b], 0, N);
    int kend = klen;
    if (p.causal) kend = min(kend, min(N, q0 + BT));
    const int nsteps = (kend + BT - 1) / BT;    // key tiles 0 .. nsteps-1

    if (threadIdx.x == 0) {
        mbar_init(bar_qd, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        for (int bf = 0; bf < NB; ++bf) {
            mbar_init(bar_st(bf), 1);
            mbar_init(bar_ps(bf), 8);
        }
        mbar_init(bar_done, 1);
        mbar_init(bar_qtm, 8);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProd) {
        if (lane == 0 && nsteps > 0) {
            prefetch_tmap(&tm.q);
            prefetch_tmap(&tm.k);
            prefetch_tmap(&tm.v);
            prefetch_tmap(&tm.dO);
            const uint64_t pol = l2_policy_evict_normal();
            mbar_arrive_expect_tx(bar_qd, 2 * C::kTileBytes);
#pragma unroll
            for (int cb = 0; cb < C::kColBlocks; ++cb) {
                tma_load_3d(q_smem + cb * (BT * 128), &tm.q, cb * 64, q0, bh, bar_qd, pol);
                tma_load_3d(do_smem + cb * (BT * 128), &tm.dO, cb * 64, q0, bh, bar_qd, pol);
            }
            bool ok = true;
            for (int n = 0; n < nsteps && ok; ++n) {
                const int s = n % C::kStages;
                if (n >= C::kStages) {
                    ok = wait_abort(bar_empty(s), ((n / C::kStages) - 1) & 1, p.err, kSiteBwEmpty, abort_flag);
                    if (!ok) break;
                }
                mbar_arrive_expect_tx(bar_full(s), 2 * C::kTileBytes);
#pragma unroll
                for (int cb = 0; cb < C::kColBlocks; ++cb) {
                    tma_load_3d(k_stage(s) + cb * (BT * 128), &tm.k, cb * 64, n * BT, bh, bar_full(s), pol);
                    tma_load_3d(v_stage(s) + cb * (BT * 128), &tm.v, cb * 64, n * BT, bh, bar_full(s), pol);
                }
            }
            mbar_wait(bar_qd, 0, p.err, kSiteBwDrain);
            const int first = nsteps > C::kStages ? nsteps - C::kStages : 0;
            for (int n = first; n < nsteps; ++n)
                mbar_wait(bar_full(n % C::kStages), (n / C::kStages) & 1, p.err, kSiteBwDrain);
        }
    } else if (warp == kMma) {
        if (nsteps > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BT, BT / 2, 0, 0);   // M 128 queries, N 64 keys
            constexpr uint32_t idesc_g = idesc_bf16_f32(BT, D, 0, 1);
            const int nhalf = 2 * nsteps;
            bool ok = wait_abort_warp(bar_qtm, 0, p.err, kSiteBwQD, abort_flag);
            // S = Q K_h^T, dP = dO V_h^T into buffer u % NB, A = Q or dO from TMEM; the
            // first half of a key tile waits for its K_j, V_j stage
            auto issue_sdp = [&](int u) {
                const int hf = u & 1, n = u >> 1, s = n % C::kStages;
                const uint32_t col = 128u * (u % NB);
                if (hf == 0) {
                    if (!wait_abort_warp(bar_full(s), (n / C::kStages) & 1, p.err, kSiteBwKV, abort_flag))
                        return false;
                    tc_fence_after();
                }
                const uint32_t rows = hf * (BT / 2) * 128;
                const uint64_t kd = sdesc_sw128(k_stage(s) + rows, 16, 1024);
                const uint64_t vd = sdesc_sw128(v_stage(s) + rows, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * (BT * 128) + (kk & 3) * 32) >> 4;
                    mma_ts_warp(tmem + col, tmem + kColQ + kk * 8, kd + off, idesc_s, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * (BT * 128) + (kk & 3) * 32) >> 4;
                    mma_ts_warp(tmem + col + 64, tmem + kColDO + kk * 8, vd + off, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit_warp(bar_st(u % NB));
                return true;
            };
            // dQ += dS K_h: A = dS from TMEM (packed over the first 16 of each warpgroup's
            // 32 dP columns), B = K_h MN-major
            auto issue_grad = [&](int u) {
                const int hf = u & 1, s = (u >> 1) % C::kStages;
                const uint32_t col = 128u * (u % NB) + 64;
                const uint64_t kdm = sdesc_sw128(k_stage(s), BT * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acol = col + (kk >> 1) * 32 + (kk & 1) * 8;
                    const uint32_t boff = ((hf * 4 + kk) * 2048) >> 4;   // 16 key rows per step
                    mma_ts_warp(tmem + kColGrad, tmem + acol, kdm + boff, idesc_g, (u > 0 || kk > 0) ? 1u : 0u);
                }
            };
            for (int u = 0; u < NB && u < nhalf && ok; ++u) ok = issue_sdp(u);
            // S/dP of half-step u + NB overwrite the buffer that dQ of half-step u read
            // just before (the tensor core runs one thread's MMAs in issue order)
            for (int u = 0; u < nhalf && ok; ++u) {
                ok = wait_abort_warp(bar_ps(u % NB), (u / NB) & 1, p.err, kSiteBwP, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_grad(u);
                if (u & 1) mma_commit_warp(bar_empty((u >> 1) % C::kStages));   // K_j, V_j read
                if (u + NB < nhalf) ok = issue_sdp(u + NB);
            }
            mma_commit_warp(bar_done);
            mbar_wait(bar_done, 0, p.err, kSiteBwDone);
            __syncwarp();
        }
    } else if (warp >= kFirstCompute) {
        // warpgroup h handles key columns [32h, 32h + 32) of every key tile (half-step
        // h / 2, columns 32 (h & 1) of its buffer), one thread per query row
        const int h = (warp - kFirstCompute) >> 2;
        const int hf = h >> 1, w = h & 1;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int q = q0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        float lrow = 0.f, drow = 0.f;
        grid_dependency_wait();   // D of bwd_pre_kernel (programmatic dependent launch)
        if (q < N) {
            lrow = p.L[static_cast<size_t>(bh) * N + q] * kLog2e;
            drow = p.Dvec[static_cast<size_t>(bh) * N + q];
        }
        const float2 sl22 = make_float2(sl2, sl2), nl2 = make_float2(-lrow, -lrow);
        const float2 ndr2 = make_float2(-drow, -drow);
        bool ok = true;
        if (h < 2 && nsteps > 0) {
            // warpgroup 0 copies this thread's row of Q_i, warpgroup 1 its row of dO_i,
            // from the swizzled shared tile (16-byte chunk c of row r sits at c ^ (r & 7))
            // into TMEM columns as packed bf16 pairs
            ok = wait_abort_warp(bar_qd, 0, p.err, kSiteBwQD, abort_flag);
            if (ok)
                tile_row_to_tmem<D>(smem + C::kFixedOff + h * C::kTileBytes, r, tmem + lane_off + (h ? kColDO : kColQ));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_qtm);
        }
        for (int n = 0; n < nsteps && ok; ++n) {
            const int u = 2 * n + hf;
            const uint32_t col = 128u * (u % NB) + 32u * w;
            ok = wait_abort_warp(bar_st(u % NB), (u / NB) & 1, p.err, kSiteBwS, abort_flag);
            if (!ok) break;
            tc_fence_after();
            __syncwarp();
            const int kb = n * BT + h * 32;   // first key of this warpgroup's columns
            // masking only where the key tile touches key_len, the diagonal or the row tail
            const bool need_mask = n * BT + BT > klen || q0 + BT > N || (p.causal && n * BT + BT - 1 > q0);
            uint32_t sr[32], dr[32];
            tmem_ld32(tmem + lane_off + col, sr);
            tmem_ld32(tmem + lane_off + col + 64, dr);
            tmem_wait_ld();
            reg_fence(sr);
            reg_fence(dr);
            if (need_mask) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int key = kb + e;
                    if (!(q < N && key < klen && (!p.causal || key <= q))) sr[e] = __float_as_uint(-INFINITY);
                }
            }
            // dS = P (dP - D), P = 2^(S scale log2 e - L log2 e), packed over the first 16
            // of this warpgroup's dP columns
            uint32_t dp[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl22, nl2);
                const float2 pr = make_float2(ex2(x.x), ex2(x.y));
                const float2 g =
                    __fmul2_rn(pr, __fadd2_rn(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), ndr2));
                dp[e >> 1] = pack_bf16(g.x, g.y);
            }
            tmem_st16(tmem + lane_off + col + 64, dp);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ps(u % NB));
        }
        if (ok && nsteps > 0) {
            ok = wait_abort_warp(bar_done, 0, p.err, kSiteBwDone, abort_flag);
            tc_fence_after();
            __syncwarp();
        }
        // dQ is staged in the shared tile Q_i held (free since Q_i was copied into
        // TMEM) and leaves by TMA stores after the CTA's last barrier; rows past N
        // are clipped by the store
        if (ok) {
            // warpgroup h stages dQ columns [32c, 32c + 32) for c = h, h + 4, ...
#pragma unroll 1
            for (int c = h; c < D / 32; c += kComputeGroups) {
                uint32_t a[32];
                if (nsteps > 0) {
                    tmem_ld32(tmem + lane_off + kColGrad + c * 32, a);
                    tmem_wait_ld();
                    reg_fence(a);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) a[e] = 0u;
                }
                const float mul = p.scale;
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    st_shared_v4(swz_chunk(q_smem, r, c * 4 + v),
                                 pack_bf16(__uint_as_float(a[8 * v]) * mul, __uint_as_float(a[8 * v + 1]) * mul),
                                 pack_bf16(__uint_as_float(a[8 * v + 2]) * mul, __uint_as_float(a[8 * v + 3]) * mul),
                                 pack_bf16(__uint_as_float(a[8 * v + 4]) * mul, __uint_as_float(a[8 * v + 5]) * mul),
                                 pack_bf16(__uint_as_float(a[8 * v + 6]) * mul, __uint_as_float(a[8 * v + 7]) * mul));
                __syncwarp();   // reconverge before the next warp-collective load
            }
            fence_proxy_async_shared();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && !*abort_flag) {
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) tma_store_3d(&tm.dq, q_smem + cb * (BT * 128), cb * 64, q0, bh);
        bulk_commit_group();
        bulk_wait_group0();
    }
    if (warp == kMma) tmem_dealloc(tmem, 512);
}

// dK/dV and dQ in one grid of B*H*2T CTAs (T = ceil(N/128)): for each (b, h), T
// dK/dV CTAs and T dQ CTAs.  The two kinds are independent (both need only D), so
// dQ CTAs fill the SMs that the dK/dV CTAs leave idle in their last wave instead
// of waiting for a second launch.
template <int D, bool kAtomicDQ = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_main_kernel(const __grid_constant__ BwdMaps tm, const BwdParams p) {
    if constexpr (kAtomicDQ) {
        // grid (B*H, T): every unit's key tile y, units innermost
        dkdv_cta<D, true>(tm, p, static_cast<int>(blockIdx.x), static_cast<int>(blockIdx.y));
    } else {
        const int T = (p.N + BT - 1) / BT;
        // CTA order: (b, h) units in groups of p.head_group; inside a group the CTA
        // kinds and tiles run in order, heaviest first, with the group's units innermost.
        // With small groups the CTAs running at once touch few units' Q, K, V and dO,
        // which then stay in L2.
        const unsigned G = static_cast<unsigned>(p.head_group);
        const unsigned per_group = G * static_cast<unsigned>(2 * T);
        const unsigned g = blockIdx.x / per_group, rem = blockIdx.x % per_group;
        const unsigned in_group = min(G, static_cast<unsigned>(p.B * p.H) - g * G);   // the last group may be short
        const int y = static_cast<int>(rem / in_group);
        const int bh = static_cast<int>(g * G + rem % in_group);
        if (y < T)
            dkdv_cta<D>(tm, p, bh, y);
        else
            dq_cta<D>(tm, p, bh, y - T);
    }
}

// dQ = bf16(scale * dQ accumulated in fp32), 8 elements per thread
__global__ void __launch_bounds__(256) dq_finalize_kernel(const float4 *acc, uint4 *dq, float scale, long long n8) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const float4 a = acc[2 * i], b = acc[2 * i + 1];
    dq[i] = make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                       pack_bf16(b.x * scale, b.y * scale), pack_bf16(b.z * scale, b.w * scale));
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams &p, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.B) * p.H * p.N;
    constexpr bool kCanAtomic = D == 64;
    const bool atomic_dq = p.dq_accum != nullptr;
    if (atomic_dq && !kCanAtomic) return cudaErrorInvalidValue;
    if (atomic_dq) {
        const cudaError_t e = cudaMemsetAsync(p.dq_accum, 0, static_cast<size_t>(rows) * D * sizeof(float), stream);
        if (e != cudaSuccess) return e;
    }
    {
        constexpr int LPR = D / 8;
        const long long threads = rows * LPR;
        const long long blocks = (threads + 255) / 256;
        if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
        bwd_pre_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(p.O), static_cast<const __nv_bfloat16 *>(p.dO), p.Dvec, rows);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    BwdMaps tm;
    std::memset(&tm, 0, sizeof tm);
    const int BH = p.B * p.H;
    if (!make_map(&tm.q, p.Q, BH, p.N, D) || !make_map(&tm.k, p.K, BH, p.N, D) ||
        !make_map(&tm.v, p.V, BH, p.N, D) || !make_map(&tm.dO, p.dO, BH, p.N, D) ||
        !make_map(&tm.dq, p.dQ, BH, p.N, D) || !make_map(&tm.dk, p.dK, BH, p.N, D) ||
        !make_map(&tm.dv, p.dV, BH, p.N, D))
        return cudaErrorInvalidValue;
    if (atomic_dq && !make_map_f32(&tm.dqa, p.dq_accum, BH, p.N, D)) return cudaErrorInvalidValue;
    int smem = BwdCfg<D, HalfStepShape<D>::kStages>::kSmemBytes;
    const void *kern = reinterpret_cast<const void *>(bwd_main_kernel<D>);
    if constexpr (kCanAtomic) {
        if (atomic_dq) {
            smem = AtomicDqShape<D>::kSmemBytes;
            kern = reinterpret_cast<const void *>(bwd_main_kernel<D, true>);
        }
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int T = (p.N + BT - 1) / BT;
    // launched as a programmatic dependent of bwd_pre_kernel: its CTAs set up
    // (barriers, TMEM, the first K/V or Q/dO loads) while D is still being written
    cudaLaunchConfig_t cfg = {};
    if (atomic_dq) {
        if (T > 65535) return cudaErrorInvalidValue;
        cfg.gridDim = dim3(static_cast<unsigned>(BH), static_cast<unsigned>(T), 1);
    } else {
        const long long ctas = static_cast<long long>(BH) * 2 * T;
        if (ctas > 0x7fffffffll) return cudaErrorInvalidValue;
        cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    }
    // Groups of (b, h) units whose Q, K, V and dO fill about 32 MiB of L2 (measured: causal
    // B1 H32 N8192 d128 backward 1522 -> 1395 us against all units interleaved; unchanged at
    // d = 64, where a group holds 32 or more units).  The dQ-accumulating variant keeps all
    // units interleaved (measured faster, also with head-major and grouped orders).
    BwdParams pg = p;
    {
        const long long per_unit = 4ll * p.N * D * 2;
        long long grp = (32ll << 20) / per_unit;
        if (grp < 1) grp = 1;
        if (grp > BH) grp = BH;
        pg.head_group = static_cast<int>(grp);
    }
    cfg.blockDim = dim3(kBwdThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (kCanAtomic) {
        if (atomic_dq) {
            e = cudaLaunchKernelEx(&cfg, bwd_main_kernel<D, true>, tm, pg);
            if (e != cudaSuccess) return e;
            const long long n8 = rows * D / 8;
            const long long blocks = (n8 + 255) / 256;
            if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
            dq_finalize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
                reinterpret_cast<const float4 *>(p.dq_accum), static_cast<uint4 *>(p.dQ), p.scale, n8);
            return cudaGetLastError();
        }
    }
    return cudaLaunchKernelEx(&cfg, bwd_main_kernel<D>, tm, pg);
}

}  // namespace

cudaError_t launch_backward(const BwdParams &p, int d, cudaStream_t stream) {
    return d == 128 ? launch_bwd_d<128>(p, stream) : launch_bwd_d<64>(p, stream);
}

}  // namespace fa
