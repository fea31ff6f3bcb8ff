// fa_prefill.cu -- exact attention forward on sm_103a tensor cores.
//
// What is computed ("Infra: Flash Attention", Algorithm 1 "FlashAttention
// forward", in the FlashAttention-2 order: query tiles outside, KV tiles
// inside, normalisation delayed to the end):
//
//   for each query tile Q_i:  m = -inf, l = 0, U = 0
//     for each KV tile j:     S = Q_i K_j^T * scale           (tensor cores)
//                             mask S (rows with no valid key skip the update)
//                             m' = max(m, rowmax S), alpha = exp(m - m')
//                             W = exp(S - m'), l = alpha l + rowsum W
//                             U = alpha U + W V_j              (tensor cores)
//                             m = m'
//     O_i = U / l,  L_i = m + log l
//
// Causal masking skips KV tiles wholly in the future and masks the diagonal
// tile on chip (same page, the causal figure; CMU 10-423 Lecture 18, 4.3).
//
// How it maps onto one GB300 SM (the FlashAttention-4 arrangement described
// on the same page, section "FlashAttention-4": two query tiles per CTA so
// the tensor core works on one tile's GEMM while the other tile's softmax
// runs):
//   * warp 0, one lane: TMA producer.  Loads Q for both query tiles once,
//     then streams K_0, V_0, K_1, V_1, ... through a ring of shared-memory
//     slots (128-byte swizzled, 64-column boxes).
//   * warp 1: allocates tensor memory; one lane issues every tcgen05.mma:
//       S_t = Q_t K_j^T        (A, B from shared memory, fp32 into TMEM)
//       O_t += P_t V_j         (A = P from TMEM, B = V from shared memory)
//     and signals completion through tcgen05.commit -> mbarrier.
//   * warps 4-7 / 8-11: softmax warpgroups for query tile 0 / 1, one thread
//     per query row.  They read S from TMEM with tcgen05.ld.red, an sm_103a
//     load that also returns each row's maximum over the loaded columns
//     (tiles with masked entries reduce the masked row instead), mask,
//     update (m, l), write
//     P = bf16(exp2(S*scale*log2e - m)) over the first half of S's TMEM
//     columns, and rescale O in TMEM by alpha when some row's max moved.
//     At the end they normalise O by 1/l, stage it in shared memory in the
//     layout of the O tensor map, and one thread stores the tile with TMA;
//     each thread writes its L.
//   Warps 0-3 form the first warpgroup (at d = 128 warps 2 and 3 have no
//   role; at d = 64 warp 2 issues the P V products, see below); it hands
//   registers to the softmax warpgroups with setmaxnreg so the softmax can
//   hold a whole 128-column score row without spilling.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 after it.
//
// The MMA issue order per KV step is PV_0(j), S_0(j+1), PV_1(j), S_1(j+1):
// (KV ring slots are released by a softmax thread once it sees S_t(j), which
// covers every MMA that read K_j and V_{j-1}; a tcgen05.commit per release
// would stall the MMA issue stream.)
// S_t(j+1) overwrites the P_t(j) that PV_t(j) reads, which relies on the
// tensor core executing one CTA's MMAs in issue order; and the barrier that
// announces S_t(j+1) also covers PV_t(j), so the softmax may rescale O_t
// as soon as it sees S_t(j+1).
//
// d = 64 runs a lookahead schedule instead.  TMEM then has room for P in
// its own columns (S_0, S_1 [0,256), O_0, O_1 [256,384), P_0, P_1
// [384,512)), so S_t(j+1) no longer has to wait for PV_t(j):
//   * a softmax warp signals s_cons[t] as soon as S_t(j) is in its registers,
//     and warp 1 then issues S_t(j+1), which runs during that softmax;
//   * warp 2 issues PV_t(j) on p_ready[t] and commits pv_done[t];
//   * the softmax waits for pv_done[t] (PV_t(j-1) complete) only before it
//     stores P_t(j) or rescales O_t.
// Each tile's next softmax step then starts as soon as the previous one ends,
// instead of after its P V and S products.  S and P V come from two
// issuing warps because one warp issuing all 24 MMAs of a KV step, on an
// SMSP that also runs two softmax warps, falls behind.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_tmap.h"

namespace fa {
namespace {

constexpr int BM = 128;          // query rows per tile (MMA M)
constexpr int BN = 128;          // keys per KV tile (MMA N of Q K^T, K of P V)
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kPvWarp = 2;           // P V issuer of the d = 64 lookahead schedule
constexpr int kThreads = 384;        // 3 warpgroups: softmax 0, softmax 1, producer/MMA (+2 idle warps)
// Per-thread registers after setmaxnreg: the softmax warpgroups and the
// producer/MMA warpgroup (2*200 + 104 = 504 = 3 * 168 at launch).  Measured:
// 200/104 is ~1 % faster than 208/88 at causal d = 128 since the row max comes
// with the TMEM load; 192/120 and 216/72 are slower, and 72 spilled the MMA
// loop state.
constexpr int kRegsSoftmax = 200;
constexpr int kRegsAux = 104;
constexpr int kTmemCols = 512;
constexpr long long kL2BlockBytes = 16ll << 20;  // K+V budget of a block of (batch, head) units
constexpr int kPrefetchTiles = 4;   // L2 prefetch distance of the KV stream, in KV tiles
// At d = 64 the next item's Q and first kPrefetchTiles K/V tiles are prefetched
// into L2 this many KV steps before the current item ends (d64 +3 %, measured);
// at d = 128 (long causal items) the Q prefetch stays at the item's start and
// the first K/V tiles at the next item's start (measured: no gain there).
template <int D>
constexpr int kNextItemPrefetchSteps = D == 64 ? 8 : 0;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleLog2 = 8.0f;  // move the exponent base only when the max grows by > 2^8

enum {
    kSiteQ = 0x201, kSiteKvFull = 0x202, kSiteKvEmpty = 0x203, kSiteP = 0x204, kSiteS = 0x205,
    kSiteO = 0x206, kSiteDrain = 0x207, kSiteMmaDone = 0x208
};

template <int D>
struct Cfg {
    static constexpr int kColBlocks = D / 64;                 // 128-byte swizzle atoms per row
    static constexpr int kTileBytes = BM * D * 2;             // one 128-row bf16 tile
    static constexpr int kSlots = (D == 128) ? 4 : 8;         // KV ring slots (K and V alternate)
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = 2 * kTileBytes;
    // O staging for the TMA store of the epilogue: one buffer per query tile at
    // d = 64, one shared by both tiles (they finish in turn) at d = 128
    static constexpr int kOStageBufs = (D == 64) ? 2 : 1;
    static constexpr int kOStageOff = kRingOff + kSlots * kTileBytes;
    static constexpr int kBarOff = kOStageOff + kOStageBufs * kTileBytes;
    // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], p_ready[2], o_final[2], mma_done,
    //           q_free, o_free[2]
    // d = 64 lookahead adds s_cons[2], pv_done[2] and the second issuer's mma_done;
    // the O staging adds ostage_full[2], ostage_free[2]
    static constexpr int kNumBars = 1 + 2 * kSlots + 19;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;    // tmem base + abort flag
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;   // +1024 for base alignment
    static constexpr uint32_t kPCol = 384;  // d = 64 lookahead: P_t at columns [384 + 64 t, 448 + 64 t)
    static_assert(D != 64 || kPCol + 2 * 64 <= kTmemCols, "P_0, P_1 must fit beside S and O");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

struct TmapSet {
    CUtensorMap q, k, v, o;
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, unsigned *err, int site,
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

// wait_or_abort for a whole converged warp: every lane polls, and the result
// is made warp-uniform so the warp never diverges around its elected issues.
__device__ __forceinline__ bool wait_or_abort_warp(uint32_t bar, uint32_t parity, unsigned *err, int site,
                                                   volatile int *abort_flag) {
    const bool ok = wait_or_abort(bar, parity, err, site, abort_flag);
    return __all_sync(0xffffffffu, ok);
}

// One work item = one (b, h, pair of 128-row query tiles).
struct Item {
    int b, h, bh, klen, ntot, t_rel;
    int row0[2], nkv[2];
};

// Item order: (batch, head) units are taken in blocks of `upb`; inside a
// block the heaviest causal pairs come first and the block's units share each
// pair index, so concurrently running CTAs read the same K/V tiles from L2.
__device__ __forceinline__ Item item_info(const PrefillParams &p, int k, int npairs, int upb) {
    Item it;
    const int units = p.B * p.H;
    const int block = k / (npairs * upb);
    const int first = block * upb;
    const int in_block = min(upb, units - first);
    const int rem = k - block * npairs * upb;
    const int pair = npairs - 1 - rem / in_block;
    it.bh = first + rem % in_block;
    it.b = it.bh / p.H;
    it.h = it.bh % p.H;
    const int N = p.N;
    it.klen = N;
    if (p.key_len) {
        const int v = p.key_len[it.b];
        it.klen = v < 0 ? 0 : (v > N ? N : v);
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        it.row0[t] = pair * 2 * BM + t * BM;
        if (it.row0[t] >= N) {
            it.nkv[t] = 0;
            continue;
        }
        int kend = it.klen;
        if (p.causal) kend = min(kend, min(N, it.row0[t] + BM));
        it.nkv[t] = (kend + BN - 1) / BN;
    }
    it.ntot = max(it.nkv[0], it.nkv[1]);
    it.t_rel = it.nkv[1] > 0 ? 1 : 0;  // the tile active in every KV step of the item
    return it;
}

// Static schedule of a persistent CTA: round r takes item r*G + c, or
// r*G + G-1-c on odd rounds, so the heavy-first order is dealt out evenly.
__device__ __forceinline__ int item_of_round(int r, int G, int c) {
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// kCount: the counting instantiation of fa_forward_count_tiles, which adds per
// (batch, head) the tile products it issues to p.tile_count; the kernels of the
// other entry points are compiled without it.
template <int D, bool QK8 = false, bool kCount = false>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ TmapSet tm, const PrefillParams p, int num_items, int npairs, int upb) {
    using C = Cfg<D>;
    // QK8: Q and K are E4M3 (one byte per element) and S = Q K^T runs as
    // tcgen05.mma kind::f8f6f4; V, P and O stay bf16.  A row of an FP8 tile
    // at d = 128 is one 128-byte swizzle atom.
    constexpr int kQKBlocks = QK8 ? D / 128 : C::kColBlocks;      // 128-byte column blocks
    constexpr int kQKBlockElems = QK8 ? 128 : 64;
    constexpr uint32_t kQTileBytes = QK8 ? BM * D : C::kTileBytes;
    constexpr uint32_t kKTileBytes = QK8 ? BN * D : C::kTileBytes;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzled tiles need 1024-byte aligned bases.
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t q_smem = sbase + C::kQOff;
    const uint32_t ring = sbase + C::kRingOff;
    const uint32_t bars = sbase + C::kBarOff;
    const uint32_t bar_q = bars;
    auto bar_kv_full = [&](int s) { return bars + 8u * (1 + s); };
    auto bar_kv_empty = [&](int s) { return bars + 8u * (1 + C::kSlots + s); };
    auto bar_s_full = [&](int t) { return bars + 8u * (1 + 2 * C::kSlots + t); };
    auto bar_p_ready = [&](int t) { return bars + 8u * (3 + 2 * C::kSlots + t); };
    auto bar_o_final = [&](int t) { return bars + 8u * (5 + 2 * C::kSlots + t); };
    const uint32_t bar_mma_done = bars + 8u * (7 + 2 * C::kSlots);
    const uint32_t bar_q_free = bars + 8u * (8 + 2 * C::kSlots);
    auto bar_o_free = [&](int t) { return bars + 8u * (9 + 2 * C::kSlots + t); };
    auto bar_s_cons = [&](int t) { return bars + 8u * (11 + 2 * C::kSlots + t); };
    auto bar_pv_done = [&](int t) { return bars + 8u * (13 + 2 * C::kSlots + t); };
    const uint32_t bar_mma_done_pv = bars + 8u * (15 + 2 * C::kSlots);
    auto bar_ostage_full = [&](int b) { return bars + 8u * (16 + 2 * C::kSlots + b); };
    auto bar_ostage_free = [&](int b) { return bars + 8u * (18 + 2 * C::kSlots + b); };
    // the d = 64 lookahead schedule (see the top of this file)
    constexpr bool kLA = (D == 64) && !QK8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int N = p.N;

    // ---- set-up: barriers, TMEM
    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(bar_kv_full(s), 1);
            mbar_init(bar_kv_empty(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar_s_full(t), 1);
            mbar_init(bar_p_ready(t), 4);
            mbar_init(bar_o_final(t), 1);
            mbar_init(bar_o_free(t), 4);
            mbar_init(bar_s_cons(t), 4);
            mbar_init(bar_pv_done(t), 1);
            mbar_init(bar_ostage_full(t), 4);
            mbar_init(bar_ostage_free(t), 1);
        }
        mbar_init(bar_mma_done, 1);
        mbar_init(bar_mma_done_pv, 1);
        mbar_init(bar_q_free, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Move registers from the producer/MMA warpgroup to the softmax warpgroups
    // (the host checks 2*128*kRegsSoftmax + 128*kRegsAux <= 384 * launch registers).
    if (warp < 4) {
        setmaxnreg_dec<kRegsAux>();
        if (warp == kProducerWarp) {
            // ================================================= TMA producer
            if (lane == 0) {
                prefetch_tmap(&tm.q);
                prefetch_tmap(&tm.k);
                prefetch_tmap(&tm.v);
                const uint64_t pol_q = l2_policy_evict_first();
                const uint64_t pol_kv = l2_policy_evict_normal();
                int g = 0;       // running index of K/V tiles in the ring (all items)
                int qi = 0;      // items with work so far (phase of q_full / q_free)
                bool ok = true;
                for (int r = 0; ok; ++r) {
                    const int k = item_of_round(r, G, cta);
                    if (k >= num_items) break;
                    const Item it = item_info(p, k, npairs, upb);
                    if (it.ntot == 0) continue;
                    // Q of the next item of this CTA: warm L2 while this one runs
                    constexpr int kNextPf = kNextItemPrefetchSteps<D>;
                    const int kn = item_of_round(r + 1, G, cta);
                    if (kNextPf == 0 && kn < num_items) {
                        const Item nx = item_info(p, kn, npairs, upb);
#pragma unroll
                        for (int t = 0; t < 2; ++t)
#pragma unroll
                            for (int cb = 0; cb < kQKBlocks; ++cb)
                                tma_prefetch_3d(&tm.q, cb * kQKBlockElems, nx.row0[t], nx.bh);
                    }
                    // Q smem is free once the previous item's last S MMA completed
                    if (qi > 0 && !wait_or_abort(bar_q_free, (qi - 1) & 1, p.err, kSiteQ, abort_flag)) break;
                    mbar_arrive_expect_tx(bar_q, 2 * kQTileBytes);
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int cb = 0; cb < kQKBlocks; ++cb)
                            tma_load_3d(q_smem + t * C::kTileBytes + cb * (BM * 128), &tm.q, cb * kQKBlockElems,
                                        it.row0[t],
                                        it.bh, bar_q, pol_q);
                    ++qi;
                    // this item's first K/V tiles (unless the previous item prefetched them)
                    if (kNextPf == 0 || qi == 1)
                        for (int j = 0; j < kPrefetchTiles && j < it.ntot; ++j)
#pragma unroll
                            for (int cb = 0; cb < C::kColBlocks; ++cb) {
                                if (cb < kQKBlocks) tma_prefetch_3d(&tm.k, cb * kQKBlockElems, j * BN, it.bh);
                                tma_prefetch_3d(&tm.v, cb * 64, j * BN, it.bh);
                            }
                    for (int j = 0; ok && j < it.ntot; ++j) {
                        if (kNextPf > 0 && j == (it.ntot > kNextPf ? it.ntot - kNextPf : 0) && kn < num_items) {
                            // the next item's Q and first K/V tiles, a few steps before this item ends
                            const Item nx = item_info(p, kn, npairs, upb);
#pragma unroll
                            for (int t = 0; t < 2; ++t)
#pragma unroll
                                for (int cb = 0; cb < kQKBlocks; ++cb)
                                    tma_prefetch_3d(&tm.q, cb * kQKBlockElems, nx.row0[t], nx.bh);
                            for (int jj = 0; jj < kPrefetchTiles && jj < nx.ntot; ++jj)
#pragma unroll
                                for (int cb = 0; cb < C::kColBlocks; ++cb) {
                                    if (cb < kQKBlocks) tma_prefetch_3d(&tm.k, cb * kQKBlockElems, jj * BN, nx.bh);
                                    tma_prefetch_3d(&tm.v, cb * 64, jj * BN, nx.bh);
                                }
                        }
                        for (int kv = 0; kv < 2; ++kv) {  // K_j then V_j
                            const int s = g % C::kSlots;
                            if (g >= C::kSlots &&
                                !wait_or_abort(bar_kv_empty(s), ((g / C::kSlots) - 1) & 1, p.err, kSiteKvEmpty,
                                               abort_flag)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(bar_kv_full(s), kv ? C::kTileBytes : kKTileBytes);
                            const CUtensorMap *map = kv ? &tm.v : &tm.k;
                            const int nblk = kv ? C::kColBlocks : kQKBlocks;
                            const int belems = kv ? 64 : kQKBlockElems;
#pragma unroll
                            for (int cb = 0; cb < C::kColBlocks; ++cb)
                                if (cb < nblk)
                                    tma_load_3d(ring + s * C::kTileBytes + cb * (BN * 128), map, cb * belems,
                                                j * BN, it.bh, bar_kv_full(s), pol_kv);
                            // Warm L2 with the same tensor's tile kPrefetchTiles steps
                            // ahead: the CTAs of one head walk the KV tiles in step, so
                            // a tile's first touch would otherwise stall them on DRAM.
                            if (j + kPrefetchTiles < it.ntot)
#pragma unroll
                                for (int cb = 0; cb < C::kColBlocks; ++cb)
                                    if (cb < nblk) tma_prefetch_3d(map, cb * belems, (j + kPrefetchTiles) * BN, it.bh);
                            ++g;
                        }
                    }
                }
                // Drain: no copy may still be in flight when the CTA exits.
                if (qi > 0) mbar_wait(bar_q, (qi - 1) & 1, p.err, kSiteDrain);
                const int first = g > C::kSlots ? g - C::kSlots : 0;
                for (int item = first; item < g; ++item)
                    mbar_wait(bar_kv_full(item % C::kSlots), (item / C::kSlots) & 1, p.err, kSiteDrain);
            }
        } else if (warp == kMmaWarp || (kLA && warp == kPvWarp)) {
            // ================================================= MMA issuer(s)
            // The whole warp runs the loop (warp-uniform control flow and
            // operands); one elected lane issues each MMA and commit.  With
            // the lookahead schedule warp 1 issues the S products and warp 2
            // the P V products; otherwise warp 1 issues both.
            const bool do_s = !kLA || warp == kMmaWarp;
            bool issued_any = false;
            {
                constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0, 0);
                constexpr uint32_t idesc_s8 = idesc_e4m3_f32(BM, BN);
                constexpr uint32_t idesc_o = idesc_bf16_f32(BM, D, 0, 1);
                // A descriptor advanced by a byte offset: the start-address
                // field holds address >> 4 and never carries (SMEM < 256 KB).
                // per (batch, head): the S and the P V tile products issued
                auto count = [&](int bh, int which) {
                    if constexpr (kCount) {
                        if (lane == 0) atomicAdd(p.tile_count + 2 * bh + which, 1u);
                    }
                };
                auto issue_s = [&](int t, uint32_t kslot) {
                    const uint64_t qd = sdesc_sw128(q_smem + t * C::kTileBytes, 16, 1024);
                    const uint64_t kd = sdesc_sw128(kslot, 16, 1024);
                    if constexpr (QK8) {
                        // K = 32 one-byte elements per instruction: 32-byte steps along the atom
#pragma unroll
                        for (int kk = 0; kk < D / 32; ++kk) {
                            const uint32_t off = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
                            mma_ss_f8_warp(tmem + t * 128, qd + off, kd + off, idesc_s8, kk > 0 ? 1u : 0u);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
                            mma_ss_warp(tmem + t * 128, qd + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
                        }
                    }
                };
                auto issue_pv = [&](int t, uint32_t vslot, int j) {
                    const uint64_t vd = sdesc_sw128(vslot, BN * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint32_t pcol = kLA ? C::kPCol + t * 64 : t * 128u;
                        mma_ts_warp(tmem + 256 + t * D, tmem + pcol + kk * 8, vd + ((kk * 2048) >> 4), idesc_o,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    }
                };
                int g = 0;                 // running ring index of this item's K_0
                int qi = 0;                // items with work so far
                int pcnt[2] = {0, 0};      // PV_t issued so far (phase of p_ready[t])
                int scons[2] = {0, 0};     // s_cons[t] phases consumed (lookahead)
                int uses[2] = {0, 0};      // items in which tile t had work (o_final / o_free phases)
                bool ok = true;
                for (int r = 0; ok; ++r) {
                    const int k = item_of_round(r, G, cta);
                    if (k >= num_items) break;
                    const Item it = item_info(p, k, npairs, upb);
                    if (it.ntot == 0) continue;
                    if (do_s) {
                        ok = wait_or_abort_warp(bar_q, qi & 1, p.err, kSiteQ, abort_flag);
                        if (ok) ok = wait_or_abort_warp(bar_kv_full(g % C::kSlots), (g / C::kSlots) & 1, p.err,
                                                        kSiteKvFull, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        // S_t(0) may overwrite the previous item's S_t / P_t: the softmax has
                        // read its last S_t (lookahead: s_cons consumed) and its PV was issued.
#pragma unroll
                        for (int t = 0; t < 2; ++t)
                            if (it.nkv[t] > 0) {
                                issue_s(t, ring + (g % C::kSlots) * C::kTileBytes);
                                count(it.bh, 0);
                                mma_commit_warp(bar_s_full(t));
                            }
                        if (it.ntot == 1) mma_commit_warp(bar_q_free);  // the item's last S MMA is issued
                    }
                    issued_any = true;
                    for (int j = 0; ok && j < it.ntot; ++j) {
                        const int iv = g + 2 * j + 1, ik = g + 2 * j + 2;
                        const int sv = iv % C::kSlots, sk = ik % C::kSlots;
                        const uint32_t vslot = ring + sv * C::kTileBytes;
                        const uint32_t kslot = ring + sk * C::kTileBytes;
                        if constexpr (kLA) {
                            if (do_s) {
                                // S_t(j+1) as soon as softmax t has S_t(j) in registers
                                bool k_ready = false;
#pragma unroll
                                for (int t = 0; t < 2; ++t) {
                                    if (!ok || j >= it.nkv[t]) continue;
                                    ok = wait_or_abort_warp(bar_s_cons(t), scons[t] & 1, p.err, kSiteS, abort_flag);
                                    if (!ok) break;
                                    ++scons[t];
                                    if (j + 1 < it.nkv[t]) {
                                        if (!k_ready) {
                                            ok = wait_or_abort_warp(bar_kv_full(sk), (ik / C::kSlots) & 1, p.err,
                                                                    kSiteKvFull, abort_flag);
                                            if (!ok) break;
                                            k_ready = true;
                                        }
                                        tc_fence_after();
                                        issue_s(t, kslot);
                                        count(it.bh, 0);
                                        mma_commit_warp(bar_s_full(t));
                                    }
                                }
                                if (ok && j + 2 == it.ntot) mma_commit_warp(bar_q_free);  // last S MMA of the item issued
                            } else {
                                ok = wait_or_abort_warp(bar_kv_full(sv), (iv / C::kSlots) & 1, p.err, kSiteKvFull,
                                                        abort_flag);
#pragma unroll
                                for (int t = 0; t < 2; ++t) {
                                    if (!ok || j >= it.nkv[t]) continue;
                                    // O_t is overwritten by PV_t(0): the previous item's epilogue must have read it
                                    if (j == 0 && uses[t] > 0) {
                                        ok = wait_or_abort_warp(bar_o_free(t), (uses[t] - 1) & 1, p.err, kSiteO,
                                                                abort_flag);
                                        if (!ok) break;
                                    }
                                    ok = wait_or_abort_warp(bar_p_ready(t), pcnt[t] & 1, p.err, kSiteP, abort_flag);
                                    if (!ok) break;
                                    ++pcnt[t];
                                    tc_fence_after();
                                    issue_pv(t, vslot, j);
                                    count(it.bh, 1);
                                    // the item's last PV_t is announced by o_final, the others by pv_done
                                    mma_commit_warp(j + 1 == it.nkv[t] ? bar_o_final(t) : bar_pv_done(t));
                                }
                            }
                            continue;
                        }
                        ok = wait_or_abort_warp(bar_kv_full(sv), (iv / C::kSlots) & 1, p.err, kSiteKvFull, abort_flag);
                        bool k_ready = false;
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            if (!ok) break;
                            if (j < it.nkv[t]) {
                                // O_t is overwritten by PV_t(0): the previous item's epilogue must have read it
                                if (j == 0 && uses[t] > 0) {
                                    ok = wait_or_abort_warp(bar_o_free(t), (uses[t] - 1) & 1, p.err, kSiteO, abort_flag);
                                    if (!ok) break;
                                }
                                ok = wait_or_abort_warp(bar_p_ready(t), pcnt[t] & 1, p.err, kSiteP, abort_flag);
                                if (!ok) break;
                                ++pcnt[t];
                                tc_fence_after();
                                issue_pv(t, vslot, j);
                                count(it.bh, 1);
                                if (j + 1 == it.nkv[t]) mma_commit_warp(bar_o_final(t));
                            }
                            if (j + 1 < it.nkv[t]) {
                                if (!k_ready) {
                                    ok = wait_or_abort_warp(bar_kv_full(sk), (ik / C::kSlots) & 1, p.err, kSiteKvFull,
                                                       abort_flag);
                                    if (!ok) break;
                                    tc_fence_after();
                                    k_ready = true;
                                }
                                issue_s(t, kslot);
                                count(it.bh, 0);
                                mma_commit_warp(bar_s_full(t));
                            }
                        }
                        if (ok && j + 2 == it.ntot) mma_commit_warp(bar_q_free);  // last S MMA of the item issued
                    }
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (it.nkv[t] > 0) ++uses[t];
                    g += 2 * it.ntot;
                    ++qi;
                }
                if (issued_any) {
                    // every MMA issued above has completed before TMEM is released
                    const uint32_t bd = warp == kMmaWarp ? bar_mma_done : bar_mma_done_pv;
                    mma_commit_warp(bd);
                    mbar_wait(bd, 0, p.err, kSiteMmaDone);
                    __syncwarp();
                }
            }
            __syncwarp();
        }  // warp 3 (and warp 2 at d = 128): no role
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ================================================= softmax warpgroups
        const int t = (warp >> 2) - 1;        // query tile of this warpgroup
        const int quarter = warp & 3;         // TMEM lane quarter
        const int r = quarter * 32 + lane;    // row within the tile
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + t * 128;
        const uint32_t o_addr = tmem + lane_off + 256 + t * D;
        const float sl2 = p.scale_log2;
        int scnt = 0;   // S_t completions consumed (phase of s_full[t])
        int pvcnt = 0;  // pv_done[t] phases consumed (lookahead)
        // O staging: buffer ob; its uses are counted in the order both warpgroups
        // take them (tile 0, then tile 1, item by item)
        const int ob = C::kOStageBufs == 2 ? t : 0;
        const uint32_t ostage = sbase + C::kOStageOff + ob * C::kTileBytes;
        int ouse = 0;   // uses of buffer ob before the current item
        const uint32_t p_addr = kLA ? tmem + lane_off + C::kPCol + t * 64 : s_addr;
        int uses = 0;   // items in which this tile had work (phase of o_final[t])
        int g = 0;      // running ring index of the item's K_0
        bool ok = true;
        for (int rr = 0; ok; ++rr) {
            const int k = item_of_round(rr, G, cta);
            if (k >= num_items) break;
            const Item it = item_info(p, k, npairs, upb);
            const int my_row0 = t ? it.row0[1] : it.row0[0];
            const int my_nkv = t ? it.nkv[1] : it.nkv[0];
            const int klen = it.klen;
            const int qi = my_row0 + r;           // query index
            const bool store = qi < N && my_row0 < N;
            __nv_bfloat16 *orow =
                static_cast<__nv_bfloat16 *>(p.O) + (static_cast<size_t>(it.bh) * N + qi) * D;

            // Conditional rescaling ("Infra: Flash Attention", "Conditional
            // rescaling invariant"): l and U are kept relative to a base r that
            // only moves when the row max exceeds r + kRescaleLog2; u(r)/l(r) does
            // not depend on r, and with r within kRescaleLog2 of the max every
            // weight stays <= 2^kRescaleLog2.  r is in log2 units of the scaled score.
            float r_base = -INFINITY;
            float l_run = 0.f;
            for (int j = 0; j < my_nkv; ++j) {
                ok = __all_sync(0xffffffffu, wait_or_abort(bar_s_full(t), scnt & 1, p.err, kSiteS, abort_flag));
                if (!ok) break;
                ++scnt;
                // S_t(j) complete implies every MMA its issuer issued before it is
                // complete: the releasing tile (the one active in every KV step)
                // hands K_j (and, with one issuer, V_{j-1}) back to the producer
                // with a plain arrive.  With the lookahead schedule V_{j-1} is
                // released below, once PV(j-1) is known complete.
                if (t == it.t_rel && quarter == 0 && lane == 0) {
                    mbar_arrive(bar_kv_empty((g + 2 * j) % C::kSlots));
                    if (!kLA && j > 0) mbar_arrive(bar_kv_empty((g + 2 * j - 1) % C::kSlots));
                }
                tc_fence_after();
                __syncwarp();
                // S_t(j) row into registers; the load also reduces the row to its
                // maximum (tcgen05.ld.red), so unmasked tiles need no max pass.
                // One 128-column load at d = 64, four 32-column loads at d = 128
                // (the faster register allocation of each, measured).
                uint32_t sr[4][32];
                float hmax;
                if constexpr (D == 64) {
                    hmax = tmem_ld128_max(s_addr, reinterpret_cast<uint32_t (&)[128]>(sr));
                    tmem_wait_ld();
                    reg_fence_f(hmax);
                } else {
                    float hm[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) hm[c] = tmem_ld32_max(s_addr + c * 32, sr[c]);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 4; ++c) reg_fence_f(hm[c]);
                    hmax = fmaxf(fmaxf(hm[0], hm[1]), fmaxf(hm[2], hm[3]));
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
                if constexpr (kLA) {
                    // S_t(j) is in registers: S_t(j+1) may be written
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_s_cons(t));
                }

                // mask: keys beyond key_len / the sequence, and the causal future
                const int kbase = j * BN;
                const bool need_mask = (kbase + BN > klen) || (p.causal && kbase + BN > my_row0);
                if (need_mask) {
                    int lim = klen - kbase;
                    if (p.causal) lim = min(lim, qi - kbase + 1);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (c * 32 + e >= lim) sr[c][e] = __float_as_uint(-INFINITY);
                }
                // row max: from the load, or, on a tile with masked entries, over the
                // masked row in four independent chains of three-input maxima
                float mrow = hmax;
                if (need_mask) {
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 32; e += 2)
                            mx[(e >> 1) & 3] = fmax3(mx[(e >> 1) & 3], __uint_as_float(sr[c][e]),
                                                     __uint_as_float(sr[c][e + 1]));
                    mrow = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                }
                mrow *= sl2;
                const bool resc = mrow > r_base + kRescaleLog2;   // always true on the first valid tile
                const float r_new = resc ? mrow : r_base;
                // a row that has seen no valid key keeps a finite base, so no
                // -inf - (-inf) appears; its weights are then all zero
                const float r_use = (r_new == -INFINITY) ? 0.f : r_new;
                const float alpha = resc ? ex2(r_base - r_use) : 1.f;  // 0 when r_base = -inf
                const float2 nr2 = make_float2(-r_use, -r_use);
                const float2 sl22 = make_float2(sl2, sl2);

                float2 ls[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) ls[a] = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 x = __ffma2_rn(
                            make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), sl22, nr2);
                        const float2 w = make_float2(ex2(x.x), ex2(x.y));
                        ls[(e >> 1) & 3] = __fadd2_rn(ls[(e >> 1) & 3], w);
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(w.x, w.y);
                        pk[e >> 1] = *reinterpret_cast<const uint32_t *>(&pr);
                    }
                    // P columns 16c .. 16c+15 of this tile's P (over S, or its own columns at d = 64)
#pragma unroll
                    for (int e = 0; e < 16; ++e) sr[c][e] = pk[e];
                }
                {
                    uint32_t lo[32], hi[32];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        lo[e] = sr[0][e];
                        lo[16 + e] = sr[1][e];
                        hi[e] = sr[2][e];
                        hi[16 + e] = sr[3][e];
                    }
                    if (kLA && j > 0) {
                        // PV_t(j-1) complete: P_t may be overwritten and O_t rescaled.  On the
                        // releasing tile it also covers the other tile's PV(j-1), so V_{j-1} is free.
                        ok = __all_sync(0xffffffffu,
                                        wait_or_abort(bar_pv_done(t), pvcnt & 1, p.err, kSiteP, abort_flag));
                        if (!ok) break;
                        ++pvcnt;
                        tc_fence_after();
                        if (t == it.t_rel && quarter == 0 && lane == 0)
                            mbar_arrive(bar_kv_empty((g + 2 * j - 1) % C::kSlots));
                    }
                    tmem_st32(p_addr + 0, lo);
                    tmem_st32(p_addr + 32, hi);
                }
                const float2 s01 = __fadd2_rn(__fadd2_rn(ls[0], ls[1]), __fadd2_rn(ls[2], ls[3]));
                l_run = fmaf(l_run, alpha, s01.x + s01.y);
                r_base = r_new;

                // correction U <- alpha U, only when some row of the warp moved its
                // base (O holds the complete PV(j-1) at this point)
                if (j > 0 && __any_sync(0xffffffffu, resc)) {
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int c = 0; c < D / 32; c += 2) {
                        uint32_t o0[32], o1[32];
                        tmem_ld32(o_addr + c * 32, o0);
                        tmem_ld32(o_addr + (c + 1) * 32, o1);
                        tmem_wait_ld();
                        reg_fence(o0);
                        reg_fence(o1);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float2 v0 = __fmul2_rn(make_float2(__uint_as_float(o0[e]), __uint_as_float(o0[e + 1])), a2);
                            float2 v1 = __fmul2_rn(make_float2(__uint_as_float(o1[e]), __uint_as_float(o1[e + 1])), a2);
                            o0[e] = __float_as_uint(v0.x);
                            o0[e + 1] = __float_as_uint(v0.y);
                            o1[e] = __float_as_uint(v1.x);
                            o1[e + 1] = __float_as_uint(v1.y);
                        }
                        tmem_st32(o_addr + c * 32, o0);
                        tmem_st32(o_addr + (c + 1) * 32, o1);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_ready(t));
            }
            if (!ok) break;

            // ---- epilogue: O = U / l, L = m + log l
            if (my_nkv > 0) {
                ok = __all_sync(0xffffffffu, wait_or_abort(bar_o_final(t), uses & 1, p.err, kSiteO, abort_flag));
                if (!ok) break;
                ++uses;
                tc_fence_after();
                __syncwarp();
                // the last V tile of the item is free once the item's last PV completed
                if (t == it.t_rel && quarter == 0 && lane == 0)
                    mbar_arrive(bar_kv_empty((g + 2 * it.ntot - 1) % C::kSlots));
                uint32_t o[D / 32][32];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_ld32(o_addr + c * 32, o[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) reg_fence(o[c]);
                // O_t has been read: the next item's PV_t(0) may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_o_free(t));
                // O goes out through shared memory and a TMA store: one thread per row
                // writing its own 2d-byte row straight to global memory touches 32 cache
                // lines per store instruction, which kept the epilogue (and the barrier
                // polls queued behind those stores) slow.
                const int ui = ouse + ((C::kOStageBufs == 1 && t == 1 && it.nkv[0] > 0) ? 1 : 0);
                if (ui > 0) {
                    ok = __all_sync(0xffffffffu, wait_or_abort(bar_ostage_free(ob), (ui - 1) & 1, p.err, kSiteO,
                                                               abort_flag));
                    if (!ok) break;
                }
                {
                    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 pr =
                                    __floats2bfloat162_rn(__uint_as_float(o[c][v * 8 + 2 * e]) * inv,
                                                          __uint_as_float(o[c][v * 8 + 2 * e + 1]) * inv);
                                w[e] = *reinterpret_cast<const uint32_t *>(&pr);
                            }
                            // 16-byte chunk kc of row r in the 128-byte-swizzled layout of the O map
                            const int kc = c * 4 + v;
                            const uint32_t addr = ostage + (kc >> 3) * (BM * 128) + r * 128 +
                                                  (static_cast<uint32_t>((kc & 7) ^ (r & 7)) << 4);
                            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_ostage_full(ob));
                if (quarter == 0 && lane == 0) {
                    // all four warps have staged their rows; rows past N are clipped by the store
                    if (wait_or_abort(bar_ostage_full(ob), ui & 1, p.err, kSiteO, abort_flag)) {
#pragma unroll
                        for (int cb = 0; cb < D / 64; ++cb)
                            tma_store_3d(&tm.o, ostage + cb * (BM * 128), cb * 64, my_row0, it.bh);
                        bulk_commit_group();
                        bulk_wait_group_read0();
                    }
                    mbar_arrive(bar_ostage_free(ob));
                }
                if (store && p.L)
                    p.L[static_cast<size_t>(it.bh) * N + qi] =
                        l_run > 0.f ? (r_base + __log2f(l_run)) * kLn2 : -INFINITY;
            } else if (store) {
                // no valid key for this row (key_len = 0): O = 0, L = -inf
                uint4 *dst = reinterpret_cast<uint4 *>(orow);
                for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
                if (p.L) p.L[static_cast<size_t>(it.bh) * N + qi] = -INFINITY;
            }
            ouse += C::kOStageBufs == 2 ? (my_nkv > 0 ? 1 : 0) : (it.nkv[0] > 0 ? 1 : 0) + (it.nkv[1] > 0 ? 1 : 0);
            g += 2 * it.ntot;
        }
        // the O stores this thread issued are complete before the CTA exits
        if (quarter == 0 && lane == 0) bulk_wait_group0();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
template <int D, bool QK8 = false, bool kCount = false>
cudaError_t launch_d(const PrefillParams &p, cudaStream_t stream) {
    TmapSet tm;
    std::memset(&tm, 0, sizeof tm);
    const int BH = p.B * p.H;
    const bool maps = QK8 ? make_map_u8(&tm.q, p.Q, BH, p.N, D) && make_map_u8(&tm.k, p.K, BH, p.N, D)
                          : make_map(&tm.q, p.Q, BH, p.N, D) && make_map(&tm.k, p.K, BH, p.N, D);
    if (!maps || !make_map(&tm.v, p.V, BH, p.N, D) || !make_map(&tm.o, p.O, BH, p.N, D)) return cudaErrorInvalidValue;
    const int smem = Cfg<D>::kSmemBytes;
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<D, QK8, kCount>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc only completes when the registers it asks for exist in
    // the block's launch allocation: refuse to launch a build where they do not.
    // (a property of the compiled kernel, the same on every device: computed once)
    static std::atomic<int> regs_ok{-1};
    if (regs_ok.load() < 0) {
        cudaFuncAttributes fa_attr;
        e = cudaFuncGetAttributes(&fa_attr, prefill_kernel<D, QK8, kCount>);
        if (e != cudaSuccess) return e;
        const long long have = static_cast<long long>(fa_attr.numRegs) * kThreads;
        const long long want = 2ll * 128 * kRegsSoftmax + 128ll * kRegsAux;
        regs_ok.store((have >= want && fa_attr.numRegs >= kRegsAux && fa_attr.numRegs <= kRegsSoftmax) ? 1 : 0);
    }
    if (!regs_ok.load()) return cudaErrorInvalidConfiguration;
    const int npairs = (p.N + 2 * BM - 1) / (2 * BM);
    const long long items = static_cast<long long>(npairs) * p.H * p.B;
    if (items > (1ll << 30)) return cudaErrorInvalidValue;
    int sms = 0;
    e = current_sm_count(&sms);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (shared memory and TMEM allow no more)
    const int grid = static_cast<int>(items < sms ? items : sms);
    // (batch, head) units per L2 block.  Non-causal items all cost the same,
    // so blocks whose K+V take <= kL2BlockBytes keep the concurrently running
    // CTAs on shared K/V tiles.  Causal items differ up to 64x in cost: there
    // the whole problem is one block, ordered heaviest first, because the
    // static schedule balances only a globally sorted order (measured: head
    // blocks cost more in balance than they gain in L2 hits).
    const long long kv_unit = 2ll * p.N * D * 2;
    long long upb = p.causal ? BH : kL2BlockBytes / (kv_unit > 0 ? kv_unit : 1);
    if (upb < 1) upb = 1;
    if (upb > static_cast<long long>(BH)) upb = BH;
    prefill_kernel<D, QK8, kCount><<<grid, kThreads, smem, stream>>>(tm, p, static_cast<int>(items), npairs,
                                                              static_cast<int>(upb));
    return cudaGetLastError();
}

// E4M3 -> bf16, 8 elements per thread.  Every E4M3 value (|x| <= 448, down to
// 2^-9) is a bf16 value, so the widening is exact.
__global__ void __launch_bounds__(256) e4m3_to_bf16_kernel(const uint2 *src, uint4 *dst, long long n8) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const uint2 v = src[i];
    const uint32_t w[2] = {v.x, v.y};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint16_t pair = static_cast<uint16_t>(w[k >> 1] >> (16 * (k & 1)));
        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
        o[k] = *reinterpret_cast<const uint32_t *>(&b);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

cudaError_t launch_e4m3_to_bf16(const void *src, void *dst, long long n, cudaStream_t stream) {
    if (n % 8 != 0) return cudaErrorInvalidValue;
    const long long n8 = n / 8;
    const long long blocks = (n8 + 255) / 256;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    if (blocks == 0) return cudaSuccess;
    e4m3_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const uint2 *>(src),
                                                                          static_cast<uint4 *>(dst), n8);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams &p, int d, cudaStream_t stream) {
    if (p.qk_e4m3) return d == 128 && !p.tile_count ? launch_d<128, true>(p, stream) : cudaErrorInvalidValue;
    if (p.tile_count) return d == 128 ? launch_d<128, false, true>(p, stream) : launch_d<64, false, true>(p, stream);
    return d == 128 ? launch_d<128>(p, stream) : launch_d<64>(p, stream);
}

}  // namespace fa
