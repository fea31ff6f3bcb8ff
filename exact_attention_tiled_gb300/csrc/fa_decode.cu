// fa_decode.cu -- Flash-Decoding for sm_103a: split-KV partial kernel and the
// log-sum-exp merge kernel.
//
// "science-depth M4-055: Flash-Decoding", "Flash-Decoding Algorithm":
//   1. the cache of length L is cut into chunks;
//   2. one thread block per (batch, head, chunk) computes the chunk's partial
//      output O^(k) and its normaliser (m^(k), l^(k));
//   3. a reduction kernel combines the partials:
//      m = max_k m^(k), l = sum_k l^(k) exp(m^(k) - m),
//      O = sum_k O^(k) l^(k) exp(m^(k) - m) / l.
// Within a chunk the scan is the online softmax of "Infra: Flash Attention"
// ("Merging block states", "Accumulating the weighted sum").
//
// The path is bound by HBM bandwidth (one multiply-add per two bytes of
// cache), so the split kernel is built around moving bytes: a producer warp
// streams each chunk's K and V rows into a ring of shared-memory stages with
// bulk TMA copies (a chunk of one (b, h) is contiguous in memory, so each
// stage is two plain bulk copies), and four consumer warps read them from
// shared memory with 128-bit loads.  Chunk data is read once, so the copies
// carry an L2 evict-first hint.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kStages = 2;           // ring depth (2 x 32 KB per stage at d = 128): 3 CTAs per SM
constexpr int kConsumerWarps = 4;
constexpr int kSplitThreads = (kConsumerWarps + 1) * 32;
constexpr int kMergeThreads = 256;
constexpr float kLn2 = 0.69314718055994530942f;

// Error-word sites in this file.
enum { kSiteDecodeFull = 0x101, kSiteDecodeEmpty = 0x102, kSiteDecodeDrain = 0x103, kSiteDecodeTable = 0x104 };
constexpr int kTableWin = 256;       // block-table entries staged in shared memory (paged cache)

__device__ __forceinline__ int clamp_len(int len, int lmax) {
    return len < 0 ? 0 : (len > lmax ? lmax : len);
}

// Chunk length of a sequence of `len` tokens (multiple of the granule).
__device__ __forceinline__ int chunk_tokens(int len, const DecodeParams &p) {
    if (p.num_splits > 0) {
        int c = (len + p.num_splits - 1) / p.num_splits;
        c = (c + kDecodeGranule - 1) / kDecodeGranule * kDecodeGranule;
        return c < kDecodeGranule ? kDecodeGranule : c;
    }
    return p.chunk_len;
}

__device__ __forceinline__ int num_chunks(int len, const DecodeParams &p) {
    if (len <= 0) return 0;
    const int c = chunk_tokens(len, p);
    const int n = (len + c - 1) / c;
    return n < p.smax ? n : p.smax;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Online-softmax state of one token group: running max m (log2 units of the
// scaled score), sum l and unnormalised output o over this lane's 8 dims.
struct State {
    float m, l, o[8];
};

// Merge state b into a ("Merging block states": alpha = 2^(m_a - m), beta = 2^(m_b - m)).
__device__ __forceinline__ void merge_into(State &a, const State &b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return;  // both empty
    const float fa = (a.m == -INFINITY) ? 0.f : ex2(a.m - m);
    const float fb = (b.m == -INFINITY) ? 0.f : ex2(b.m - m);
    a.l = fa * a.l + fb * b.l;
#pragma unroll
    for (int e = 0; e < 8; ++e) a.o[e] = fa * a.o[e] + fb * b.o[e];
    a.m = m;
}

__device__ __forceinline__ State shfl_xor_state(const State &s, int mask) {
    State r;
    r.m = __shfl_xor_sync(0xffffffffu, s.m, mask);
    r.l = __shfl_xor_sync(0xffffffffu, s.l, mask);
#pragma unroll
    for (int e = 0; e < 8; ++e) r.o[e] = __shfl_xor_sync(0xffffffffu, s.o[e], mask);
    return r;
}

// ---------------------------------------------------------------------------
// Split kernel: grid (smax, H, B); one CTA per (b, h, chunk).
// Warps 0..3 consume, warp 4 produces.  Each consumer warp owns 16 tokens of
// every 64-token tile; LPT = D/8 lanes cooperate on one token (8 dims each),
// so a warp covers 32/LPT tokens per step.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kSplitThreads) decode_split_kernel(const DecodeParams p) {
    constexpr int kRowBytes = D * 2;
    constexpr int kTileBytes = kDecodeTile * kRowBytes;
    constexpr int LPT = D / 8;                  // lanes per token
    constexpr int TPI = 32 / LPT;               // tokens per warp step
    constexpr int ITERS = 16 / TPI;             // steps per tile per warp

    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *k_stage = smem;                                  // [kStages][kTileBytes]
    uint8_t *v_stage = smem + kStages * kTileBytes;           // [kStages][kTileBytes]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + 2 * kStages * kTileBytes);
    uint64_t *empty = full + kStages;
    State *xwarp = reinterpret_cast<State *>(empty + kStages);  // [kConsumerWarps][LPT]
    int *tbl = reinterpret_cast<int *>(xwarp + kConsumerWarps * LPT);  // [kTableWin] (paged cache)

    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int len = clamp_len(p.seqlens[b], p.Lmax);
    const int nchunk = num_chunks(len, p);
    if (chunk >= nchunk) return;  // CTA-uniform, before any barrier use
    const int ctok = chunk_tokens(len, p);
    const int t0 = chunk * ctok;
    const int t1 = min(len, t0 + ctok);
    const int ntiles = (t1 - t0 + kDecodeTile - 1) / kDecodeTile;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t bh = static_cast<size_t>(b) * p.H + h;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ producer warp
        // Lane 0 issues the copies.  With a paged cache the whole warp first
        // stages a window of the sequence's block table in shared memory; a
        // tile then takes one bulk copy per physical block it touches
        // (CMU 10-423 Lecture 18, section 7.3: blocks found through the table).
        const uint64_t pol = l2_policy_evict_first();
        const size_t row0 = p.block_table ? 0 : bh * p.Lmax + t0;  // contiguous cache only
        const uint8_t *kbase = static_cast<const uint8_t *>(p.K) + row0 * kRowBytes;
        const uint8_t *vbase = static_cast<const uint8_t *>(p.V) + row0 * kRowBytes;
        int issued = 0;
        bool ok = true;
        int win0 = -1;  // first logical block held in tbl
        for (int i = 0; i < ntiles && ok; ++i) {
            const int rows = min(kDecodeTile, t1 - t0 - i * kDecodeTile);
            const int tok0 = t0 + i * kDecodeTile;
            if (p.block_table) {
                const int blo = tok0 / p.block_size, bhi = (tok0 + rows - 1) / p.block_size;
                if (win0 < 0 || bhi >= win0 + kTableWin) {
                    __syncwarp();
                    win0 = blo;
                    const int last = (t1 - 1) / p.block_size;  // last block of this chunk (< max_blocks)
                    for (int e = lane; e < kTableWin; e += 32) {
                        const int lb = win0 + e;
                        int phys = 0;
                        if (lb <= last) {
                            phys = p.block_table[static_cast<size_t>(b) * p.max_blocks + lb];
                            if (phys < 0 || phys >= p.num_blocks) {
                                report_invalid(p.err, kSiteDecodeTable);
                                phys = 0;   // never dereference an entry outside the pool
                            }
                        }
                        tbl[e] = phys;
                    }
                    __syncwarp();
                }
            }
            if (lane == 0) {
                const int s = i % kStages;
                if (i >= kStages)
                    ok = mbar_wait(smem_u32(&empty[s]), ((i / kStages) - 1) & 1, p.err, kSiteDecodeEmpty);
                if (ok) {
                    const uint32_t bytes = static_cast<uint32_t>(rows) * kRowBytes;
                    mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * bytes);
                    if (!p.block_table) {
                        bulk_g2s(smem_u32(k_stage + s * kTileBytes), kbase + static_cast<size_t>(i) * kTileBytes,
                                 bytes, smem_u32(&full[s]), pol);
                        bulk_g2s(smem_u32(v_stage + s * kTileBytes), vbase + static_cast<size_t>(i) * kTileBytes,
                                 bytes, smem_u32(&full[s]), pol);
                    } else {
                        for (int r = 0; r < rows;) {
                            const int tok = tok0 + r;
                            const int lb = tok / p.block_size, rin = tok % p.block_size;
                            const int n = min(rows - r, p.block_size - rin);
                            const int phys = tbl[lb - win0];
                            const size_t src = ((static_cast<size_t>(phys) * p.H + h) * p.block_size + rin) * kRowBytes;
                            const uint32_t nb = static_cast<uint32_t>(n) * kRowBytes;
                            bulk_g2s(smem_u32(k_stage + s * kTileBytes + r * kRowBytes),
                                     static_cast<const uint8_t *>(p.K) + src, nb, smem_u32(&full[s]), pol);
                            bulk_g2s(smem_u32(v_stage + s * kTileBytes + r * kRowBytes),
                                     static_cast<const uint8_t *>(p.V) + src, nb, smem_u32(&full[s]), pol);
                            r += n;
                        }
                    }
                    ++issued;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        // Never leave the CTA with copies in flight: wait (bounded) for the
        // last copies issued into each stage.
        if (lane == 0) {
            const int first = issued > kStages ? issued - kStages : 0;
            for (int i = first; i < issued; ++i)
                mbar_wait(smem_u32(&full[i % kStages]), (i / kStages) & 1, p.err, kSiteDecodeDrain);
        }
    } else {
        // ------------------------------------------------ consumers
        const int sub = lane / LPT;   // token slot within a warp step
        const int cl = lane % LPT;    // 16-byte column chunk
        float q8[8];
        {
            const uint4 raw = *reinterpret_cast<const uint4 *>(
                static_cast<const uint8_t *>(p.q) + bh * kRowBytes + cl * 16);
            bf16x8_to_f32(raw, q8);
#pragma unroll
            for (int e = 0; e < 8; ++e) q8[e] *= p.scale_log2;
        }
        State st;
        st.m = -INFINITY;
        st.l = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) st.o[e] = 0.f;

        for (int i = 0; i < ntiles; ++i) {
            const int s = i % kStages;
            if (!mbar_wait(smem_u32(&full[s]), (i / kStages) & 1, p.err, kSiteDecodeFull)) break;
            const uint8_t *ks = k_stage + s * kTileBytes;
            const uint8_t *vs = v_stage + s * kTileBytes;
            const int valid = t1 - t0 - i * kDecodeTile;  // tokens of this tile that exist
            float sc[ITERS];
            float tmax = -INFINITY;
#pragma unroll
            for (int it = 0; it < ITERS; ++it) {
                const int tok = warp * 16 + it * TPI + sub;
                const uint4 raw = *reinterpret_cast<const uint4 *>(ks + tok * kRowBytes + cl * 16);
                float kf[8];
                bf16x8_to_f32(raw, kf);
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(q8[e], kf[e], acc);
#pragma unroll
                for (int off = LPT / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                sc[it] = (tok < valid) ? acc : -INFINITY;
                tmax = fmaxf(tmax, sc[it]);
            }
            const float m_new = fmaxf(st.m, tmax);
            if (m_new != -INFINITY) {
                const float alpha = ex2(st.m - m_new);  // 0 on the first valid tile
                st.l *= alpha;
#pragma unroll
                for (int e = 0; e < 8; ++e) st.o[e] *= alpha;
#pragma unroll
                for (int it = 0; it < ITERS; ++it) {
                    const int tok = warp * 16 + it * TPI + sub;
                    // rows past the chunk end hold stale shared memory: never read them
                    if (tok < valid) {
                        const float pw = ex2(sc[it] - m_new);
                        st.l += pw;
                        const uint4 raw = *reinterpret_cast<const uint4 *>(vs + tok * kRowBytes + cl * 16);
                        float vf[8];
                        bf16x8_to_f32(raw, vf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) st.o[e] = fmaf(pw, vf[e], st.o[e]);
                    }
                }
                st.m = m_new;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }
        // merge the TPI token groups of this warp
#pragma unroll
        for (int mask = LPT; mask < 32; mask <<= 1) merge_into(st, shfl_xor_state(st, mask));
        if (lane < LPT) xwarp[warp * LPT + lane] = st;
    }
    __syncthreads();

    if (warp == 0 && lane < LPT) {
        State acc = xwarp[lane];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) merge_into(acc, xwarp[w * LPT + lane]);
        const size_t slot = bh * p.smax + chunk;
        const float inv = acc.l > 0.f ? 1.f / acc.l : 0.f;
        float4 *dst = reinterpret_cast<float4 *>(p.part_o + slot * D + lane * 8);
        dst[0] = make_float4(acc.o[0] * inv, acc.o[1] * inv, acc.o[2] * inv, acc.o[3] * inv);
        dst[1] = make_float4(acc.o[4] * inv, acc.o[5] * inv, acc.o[6] * inv, acc.o[7] * inv);
        if (lane == 0) {
            // (m, l) with m in natural-log units of the scaled score
            p.part_ml[2 * slot] = acc.m * kLn2;
            p.part_ml[2 * slot + 1] = acc.l;
        }
    }
    grid_launch_dependents();
}

// ---------------------------------------------------------------------------
// Merge kernel: grid (H, B); the log-sum-exp reduction of step 3,
//   m = max_k m_k,  l = sum_k l_k e^(m_k - m),  O = sum_k O_k l_k e^(m_k - m) / l,
// evaluated as the pages' block-state merge ("Merging block states"): each warp
// folds its chunks into a running (m, l, o) with a moving maximum, and the
// warps' states are combined at the end with one shared maximum.  The result is
// the same sum; no pass over the chunks waits for the global maximum first.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeParams p) {
    constexpr int kWarps = kMergeThreads / 32;
    constexpr int DPL = D / 32;  // dims per lane
    __shared__ float wm[kWarps], wl[kWarps];
    __shared__ float accs[kWarps][D];

    // the lengths are inputs: read them before waiting for the split kernel
    const int h = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len = clamp_len(p.seqlens[b], p.Lmax);
    const int n = num_chunks(len, p);
    const size_t bh = static_cast<size_t>(b) * p.H + h;
    const float *ml = p.part_ml + bh * p.smax * 2;
    const float *po = p.part_o + bh * p.smax * D;

    grid_dependency_wait();  // partials of the split kernel are visible after this

    // this warp's chunks k = warp, warp + kWarps, ...: running maximum m (natural
    // units), l = sum l_k e^(m_k - m), o = sum O_k l_k e^(m_k - m)
    float m = -INFINITY, l = 0.f;
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
#pragma unroll 2
    for (int k = warp; k < n; k += kWarps) {
        const float2 mlk = *reinterpret_cast<const float2 *>(ml + 2 * k);
        float v[DPL];
        const float *src = po + static_cast<size_t>(k) * D + lane * DPL;
        if constexpr (DPL == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(src);
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2 *>(src);
            v[0] = t.x; v[1] = t.y;
        }
        if (!(mlk.y > 0.f)) continue;   // an empty chunk has weight 0
        if (mlk.x > m) {
            const float c = __expf(m - mlk.x);   // 0 while m = -inf
            l *= c;
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[e] *= c;
            m = mlk.x;
        }
        const float wk = mlk.y * __expf(mlk.x - m);
        l += wk;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wk, v[e], acc[e]);
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) accs[warp][lane * DPL + e] = acc[e];
    if (lane == 0) {
        wm[warp] = m;
        wl[warp] = l;
    }
    __syncthreads();

    if (threadIdx.x < D) {
        float m_f = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) m_f = fmaxf(m_f, wm[w]);
        float l_f = 0.f, o = 0.f;
        if (m_f != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                if (wm[w] == -INFINITY) continue;   // a warp without a non-empty chunk
                const float c = __expf(wm[w] - m_f);
                l_f = fmaf(wl[w], c, l_f);
                o = fmaf(accs[w][threadIdx.x], c, o);
            }
        }
        const float out = l_f > 0.f ? o / l_f : 0.f;
        static_cast<__nv_bfloat16 *>(p.O)[bh * D + threadIdx.x] = __float2bfloat16_rn(out);
        if (threadIdx.x == 0 && p.L) p.L[bh] = l_f > 0.f ? m_f + logf(l_f) : -INFINITY;
    }
}

template <int D>
constexpr size_t split_smem_bytes() {
    return 2 * kStages * kDecodeTile * D * 2 + 2 * kStages * sizeof(uint64_t) +
           kConsumerWarps * (D / 8) * sizeof(State) + kTableWin * sizeof(int);
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams &p, cudaStream_t stream) {
    const size_t smem = split_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(p.smax, p.H, p.B);
    decode_split_kernel<D><<<grid, kSplitThreads, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.H, p.B, 1);
    cfg.blockDim = dim3(kMergeThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, p);
}

template <int D>
int ctas_per_sm_d() {
    const size_t smem = split_smem_bytes<D>();
    if (cudaFuncSetAttribute(decode_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<D>, kSplitThreads, smem) !=
        cudaSuccess)
        return 0;
    return n;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, int d, cudaStream_t stream) {
    return d == 128 ? launch_decode_d<128>(p, stream) : launch_decode_d<64>(p, stream);
}

int decode_ctas_per_sm(int d) { return d == 128 ? ctas_per_sm_d<128>() : ctas_per_sm_d<64>(); }

}  // namespace fa
