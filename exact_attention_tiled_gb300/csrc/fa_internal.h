// fa_internal.h -- launch interfaces between the C ABI layer (fa_api.cu) and
// the kernel translation units.  Host-side only; no torch types anywhere.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

// ------------------------------------------------------------------ decode
struct DecodeParams {
    const void *q;          // bf16 [B, H, d]
    const void *K;          // bf16 [B, H, Lmax, d]
    const void *V;          // bf16 [B, H, Lmax, d]
    const int32_t *seqlens; // device [B]
    float *part_o;          // fp32 [B, H, smax, d]   O_k = u_k / l_k
    float *part_ml;         // fp32 [B, H, smax, 2]   (m_k, l_k), natural-log units
    void *O;                // bf16 [B, H, d]
    float *L;               // fp32 [B, H] or nullptr
    int B, H, Lmax;
    int num_splits;         // > 0: fixed chunk count per sequence
    int chunk_len;          // tokens per chunk when num_splits <= 0 (multiple of 64)
    int smax;               // partial slots per (b, h)
    float scale_log2;       // scale * log2(e)
    unsigned *err;          // device error word
    // paged cache (block_table != nullptr): K and V are pools [num_blocks, H, block_size, d]
    // and token t of sequence b lives in block block_table[b * max_blocks + t / block_size]
    const int32_t *block_table;
    int block_size, max_blocks, num_blocks;
};

constexpr int kDecodeTile = 64;      // tokens per staged tile
constexpr int kDecodeGranule = 64;   // chunk lengths are multiples of this

// Launch the split kernel and the merge kernel on `stream`.
cudaError_t launch_decode(const DecodeParams &p, int d, cudaStream_t stream);
// Resident split-kernel CTAs per SM for head dimension d (0 on error).
int decode_ctas_per_sm(int d);

// ------------------------------------------------------------------ prefill
struct PrefillParams {
    const void *Q, *K, *V;  // bf16 [B, H, N, d]
    void *O;                // bf16 [B, H, N, d]
    float *L;               // fp32 [B, H, N] or nullptr
    const int32_t *key_len; // device [B] or nullptr
    int B, H, N;
    int causal;
    float scale_log2;       // scale * log2(e)
    unsigned *err;
    int qk_e4m3;            // Q and K are E4M3 [B, H, N, d] (d = 128); V stays bf16
    unsigned *tile_count;   // nullptr, or device [B * H][2]: S and P V tile products issued
};

cudaError_t launch_prefill(const PrefillParams &p, int d, cudaStream_t stream);
// SM count of the current device (looked up once per device).
cudaError_t current_sm_count(int *out);
// Forget the fa_decode_noalloc array's per-device addresses (fa_shutdown).
void reset_noalloc_addresses();
// E4M3 -> bf16 (exact) for n elements; n a multiple of 8, both pointers 16-byte aligned.
cudaError_t launch_e4m3_to_bf16(const void *src, void *dst, long long n, cudaStream_t stream);

// ------------------------------------------------------------------ backward
struct BwdParams {
    const void *Q, *K, *V, *O, *dO;   // bf16 [B, H, N, d]
    const float *L;                   // fp32 [B, H, N], the forward's natural-log LSE
    float *Dvec;                      // fp32 [B, H, N] scratch: D_i = dO_i . O_i
    void *dQ, *dK, *dV;               // bf16 [B, H, N, d]
    const int32_t *key_len;           // device [B] or nullptr
    int B, H, N;
    int causal;
    float scale;                      // score multiplier
    float scale_log2;                 // scale * log2(e)
    unsigned *err;
    float *dq_accum;                  // nullptr, or fp32 [B, H, N, d]: dQ accumulated by the dK/dV CTAs
    int head_group;                   // (b, h) units per group of the main grid's CTA order (set at launch)
};

cudaError_t launch_backward(const BwdParams &p, int d, cudaStream_t stream);

// ------------------------------------------------------------------ self-test
constexpr int kSiteSelfTest = 0x301;
cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned *err, cudaStream_t stream);

}  // namespace fa
