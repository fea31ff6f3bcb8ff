/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * The operations, all defined by the pages this library follows:
 *
 *   fa_forward  exact scaled-dot-product attention O = softmax(Q K^T * scale) V,
 *               computed tile by tile with the online-softmax state (m, l, U)
 *               so that the N x N scores S and weights P never reach global
 *               memory; it also returns the per-row log-sum-exp
 *               L = m + log l = log sum_j exp(S_ij).
 *               ("Infra: Flash Attention", sections "Attention and its scope",
 *               "Tiled computation and the forward pass" with Algorithm 1
 *               "FlashAttention forward", and "Backward and recomputation"
 *               for L.)
 *
 *   fa_decode   Flash-Decoding: one query per (batch, head) over a long KV
 *               cache.  The cache is split into chunks; one kernel writes a
 *               partial state (m_k, l_k, O_k) per chunk and a second kernel
 *               merges them with the log-sum-exp reduction
 *               m = max_k m_k, l = sum_k l_k exp(m_k - m),
 *               O = sum_k O_k l_k exp(m_k - m) / l.
 *               ("science-depth M4-055: Flash-Decoding", "Flash-Decoding
 *               Algorithm" steps 1-3 and trade-off 3 on the chunk count.)
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never frees or retains them.  bf16 = IEEE bfloat16 (2 bytes).
 *   - Layouts are dense row-major with the last dimension contiguous.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and performs no host synchronisation.
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing and returns FA_ERR_INVALID_ARG or
 *     FA_ERR_UNSUPPORTED.  A failed CUDA launch returns FA_ERR_CUDA.
 *   - Device pointers must be 16-byte aligned (tensor-memory-accelerator
 *     copies require it).
 *   - Kernels bound every wait on a barrier.  A wait that runs out sets a
 *     device-side error word and the kernel returns early; the outputs of
 *     that call are then undefined.  fa_device_error() reports it.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size or flag */
    FA_ERR_UNSUPPORTED = 2,     /* valid request this build does not handle (e.g. d not 64/128) */
    FA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed */
    FA_ERR_WORKSPACE = 4,       /* workspace missing or smaller than required */
    FA_ERR_DEVICE_TIMEOUT = 5   /* a bounded in-kernel wait ran out (see fa_device_error) */
} fa_status;

typedef void *fa_stream_t; /* cudaStream_t */

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

/*
 * fa_forward -- exact attention forward, one pass over Q tiles.
 *
 *   Q, K, V  bf16 [B, H, N, d], contiguous.
 *   O        bf16 [B, H, N, d] output: O_i = sum_j P_ij V_j, rounded to
 *            nearest-even bf16 from fp32.
 *   L        float [B, H, N] output, natural-log LSE of the scaled scores,
 *            or NULL to skip it.  A query row with no valid key gets O = 0
 *            and L = -inf (the pages leave that case to the operator).
 *   B, H, N  batch, heads, sequence length (queries and keys); all >= 1,
 *            B * H <= 65535 * 65535.
 *   d        head dimension, 64 or 128 (others: FA_ERR_UNSUPPORTED).
 *   causal   0: every query sees every key; 1: query i sees keys j <= i
 *            (upper-left aligned, square).  Key tiles wholly in the future
 *            are skipped, diagonal tiles are masked on chip.
 *   scale    score multiplier; <= 0 selects 1/sqrt(d).
 *   key_len  NULL, or a DEVICE int32 [B]: keys j >= key_len[b] of batch b
 *            are masked (right key padding).  Values are clamped to
 *            [0, N]; key_len[b] = 0 leaves every row of b without keys.
 *   stream   cudaStream_t.
 *
 * Arithmetic: bf16 inputs, fp32 tensor-core accumulation of Q K^T and of
 * W V, fp32 softmax state; P is rounded to bf16 before the W V product.
 */
FA_API fa_status fa_forward(const void *Q, const void *K, const void *V, void *O, float *L,
                     int B, int H, int N, int d, int causal, float scale,
                     const int32_t *key_len, fa_stream_t stream);

/*
 * fa_forward_count_tiles -- fa_forward that also counts, per (batch, head),
 * the 128 x 128 tile products the kernel issues: tile_counts[2 * (b * H + h)]
 * the S = Q K^T products and tile_counts[2 * (b * H + h) + 1] the P V
 * products.  It makes the causal tile skipping of "Infra: Flash Attention"
 * (section "Symbols and boundary conditions", the causal figure) and "CMU
 * 10-423 Lecture 18" (section 4.3, exercise 4: T(T+1)/2 of T^2 tiles)
 * observable; the outputs are those of fa_forward.
 *
 *   tile_counts  DEVICE uint32 [B * H * 2], 4-byte aligned, zero-filled by
 *                the call (on `stream`) before the kernel adds to it.
 * Other arguments, results and errors: as in fa_forward.  The counting adds
 * one atomic per tile product, so this call is for checking, not timing.
 */
FA_API fa_status fa_forward_count_tiles(const void *Q, const void *K, const void *V, void *O, float *L,
                                        int B, int H, int N, int d, int causal, float scale,
                                        const int32_t *key_len, unsigned *tile_counts, fa_stream_t stream);

/*
 * fa_forward_host -- fa_forward over HOST buffers, with the host<->device
 * copies inside the call.  The (batch, head) slices are independent problems
 * ("Infra: Flash Attention", "Attention and its scope": each head attends on
 * its own), so the call splits them into groups of `heads_per_group`
 * consecutive heads of one batch element and pipelines, on internal streams,
 * the copy of a group's Q, K, V to the device, fa_forward on it, and the copy
 * of its O (and L) back, so that the copies of one group overlap the compute
 * and copies of the others.  The results are bit-identical to fa_forward on
 * the same data (every (batch, head) is computed by the same kernel code).
 *
 *   Qh, Kh, Vh  HOST bf16 [B, H, N, d], contiguous; page-locked (pinned)
 *               memory lets the copies run asynchronously and overlap, other
 *               host memory works but each copy then blocks the host.
 *   Oh          HOST bf16 [B, H, N, d] output.
 *   Lh          HOST float [B, H, N] output, or NULL.
 *   key_len_host  NULL, or a HOST int32 [B] (read before the call returns).
 *   heads_per_group  0 = automatic (the largest divisor of H whose Q slice
 *               is at most 16 MiB); otherwise a divisor of H.
 *   workspace   DEVICE scratch, 256-byte aligned, at least
 *               fa_forward_host_workspace_bytes(B, H, N, d, heads_per_group)
 *               bytes; it holds up to three groups' Q, K, V, O, L in flight.
 *   stream      work is ordered after what `stream` already holds, and
 *               `stream` waits for the whole call (the last copy to Oh/Lh)
 *               before any later work; the host does not wait, so Oh and Lh
 *               are complete once `stream` is synchronised.
 * Other arguments and the arithmetic are those of fa_forward.
 * Errors: FA_ERR_INVALID_ARG (null pointers, shapes, heads_per_group not
 * dividing H), FA_ERR_UNSUPPORTED (d), FA_ERR_WORKSPACE, FA_ERR_CUDA (a copy
 * or launch failed; some groups may then be missing from Oh).
 */
FA_API fa_status fa_forward_host(const void *Qh, const void *Kh, const void *Vh, void *Oh, float *Lh,
                                 int B, int H, int N, int d, int causal, float scale,
                                 const int32_t *key_len_host, int heads_per_group, void *workspace,
                                 size_t workspace_bytes, fa_stream_t stream);

/* Device scratch bytes fa_forward_host needs; 0 for an invalid shape. */
FA_API size_t fa_forward_host_workspace_bytes(int B, int H, int N, int d, int heads_per_group);

/*
 * fa_forward_fp8 -- fa_forward with FP8 (E4M3) inputs.  ("Infra: Flash
 * Attention", "FlashAttention-3": FA3 explores FP8 and its quantisation error
 * has to be evaluated on its own.)  The attention computed is exactly
 * fa_forward's over the E4M3 values of Q, K and V:
 *   S = Q K^T * scale runs on the FP8 tensor cores (tcgen05.mma kind::f8f6f4,
 *   E4M3 x E4M3, fp32 accumulation: every product is exact);
 *   V is widened to bf16 (exact for every E4M3 value) into `workspace`, and
 *   P V runs as in fa_forward (P rounded to bf16, fp32 accumulation).
 * So the kernel's rounding is that of fa_forward on the same values; the
 * error of quantising real-valued inputs to E4M3 is the caller's.
 *
 *   Q8, K8, V8  E4M3 codes (one byte each) [B, H, N, d], contiguous; d = 128
 *               (others: FA_ERR_UNSUPPORTED).  No scale factors: the codes are
 *               the values.
 *   O, L, B, H, N, causal, scale, key_len: as in fa_forward.
 *   workspace   device scratch of at least fa_forward_fp8_workspace_bytes()
 *               bytes, 256-byte aligned (the bf16 copy of V).
 */
FA_API fa_status fa_forward_fp8(const void *Q8, const void *K8, const void *V8, void *O, float *L,
                                int B, int H, int N, int d, int causal, float scale,
                                const int32_t *key_len, void *workspace, size_t workspace_bytes,
                                fa_stream_t stream);

/* Workspace bytes fa_forward_fp8 needs (0 for arguments it would reject). */
FA_API size_t fa_forward_fp8_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_backward -- gradients of exact attention ("Infra: Flash Attention",
 * sections "Backward and recomputation" and "Blocked gradient computation";
 * CMU 10-423 Lecture 18 notes, 5.3).  With S = scale Q K^T (masked as in
 * fa_forward), P_ij = exp(S_ij - L_i), dP = dO V^T, D_i = dO_i . O_i and
 * dS_ij = P_ij (dP_ij - D_i):
 *     dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
 * P, dP and dS are recomputed tile by tile on chip and never reach global
 * memory.
 *
 *   Q, K, V, O, dO  bf16 [B, H, N, d]: the forward's inputs and output and the
 *                   upstream gradient of O.
 *   L               float [B, H, N]: the forward's L for the same inputs.
 *   dQ, dK, dV      bf16 [B, H, N, d] outputs, fully written (keys that no
 *                   query sees, and query rows with no valid key, get 0).
 *   B, H, N, d, causal, scale, key_len: as in fa_forward (same values as the
 *                   forward call that produced O and L).
 *   workspace       device scratch of at least fa_backward_workspace_bytes()
 *                   bytes, 256-byte aligned (holds D); not read before written.
 *
 * Arithmetic: fp32 tensor-core accumulation; P and dS are rounded to bf16
 * before the products with dO, Q and K; D from the bf16 O.  Every gradient
 * element is written by one thread block (no atomics): results do not
 * depend on scheduling.
 */
FA_API fa_status fa_backward(const void *Q, const void *K, const void *V, const void *O,
                             const void *dO, const float *L, void *dQ, void *dK, void *dV,
                             int B, int H, int N, int d, int causal, float scale,
                             const int32_t *key_len, void *workspace, size_t workspace_bytes,
                             fa_stream_t stream);

/* Workspace bytes fa_backward needs (0 for arguments it would reject). */
FA_API size_t fa_backward_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_backward_atomic_dq -- fa_backward with dQ accumulated across key tiles by
 * fp32 atomic additions.  (The pages compute dQ_i = scale sum_j dS_ij K_j by
 * blocks, "Blocked gradient computation"; this entry point is a different order
 * of that sum, not a different result.)
 *
 * The thread block of key tile j, which already holds K_j and forms dS for
 * every query tile it meets, also forms dQ_i += dS_i K_j in TMEM and adds it
 * into an fp32 copy of dQ in the workspace; a last kernel scales it and
 * rounds it to bf16.  No second pass recomputes S, dP and dS per query tile,
 * so it does less work than fa_backward; but the order of the fp32 additions
 * into dQ depends on scheduling, so dQ may differ from run to run in its last
 * bits (dK and dV do not: they are produced as in fa_backward).
 *
 * Arguments as fa_backward, except: d must be 64 (FA_ERR_UNSUPPORTED
 * otherwise: at d = 128 the dQ accumulator does not fit beside dK and dV in
 * tensor memory), and the workspace holds at least
 * fa_backward_atomic_dq_workspace_bytes() bytes (D, then the fp32 dQ).
 */
FA_API fa_status fa_backward_atomic_dq(const void *Q, const void *K, const void *V, const void *O,
                                       const void *dO, const float *L, void *dQ, void *dK, void *dV,
                                       int B, int H, int N, int d, int causal, float scale,
                                       const int32_t *key_len, void *workspace, size_t workspace_bytes,
                                       fa_stream_t stream);

/* Workspace bytes fa_backward_atomic_dq needs (0 for arguments it would reject). */
FA_API size_t fa_backward_atomic_dq_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_decode -- split-KV single-query attention (Flash-Decoding).
 *
 *   q             bf16 [B, H, d]: one query per (b, h).
 *   Kcache,Vcache bf16 [B, H, Lmax, d]; row t of (b, h) holds token t.
 *   seqlens       DEVICE int32 [B]: tokens 0 .. seqlens[b]-1 are attended;
 *                 values are clamped to [0, Lmax].
 *   seqlens_host  HOST copy of seqlens used to plan the split without a
 *                 device synchronisation, or NULL (then every sequence is
 *                 planned as if it were Lmax long; results are identical).
 *   O             bf16 [B, H, d] output.  L: float [B, H] natural-log LSE or
 *                 NULL.  A sequence of length 0 gets O = 0, L = -inf.
 *   d             64 or 128.  scale <= 0 selects 1/sqrt(d).
 *   num_splits    > 0: every sequence is cut into num_splits chunks of
 *                 ceil(len / num_splits) tokens rounded up to a multiple of
 *                 64 (so a short sequence may use fewer chunks);
 *                 <= 0: automatic, one chunk length for the whole batch
 *                 chosen from the SM count and the sequence lengths, which
 *                 gives each sequence its own chunk count.
 *   workspace     device scratch of at least fa_decode_workspace_bytes(...)
 *                 bytes, 256-byte aligned; holds the per-chunk partials.
 *                 Not read before it is written; may be reused across calls
 *                 that are ordered on the GPU.
 */
FA_API fa_status fa_decode(const void *q, const void *Kcache, const void *Vcache,
                    const int32_t *seqlens, const int32_t *seqlens_host,
                    void *O, float *L,
                    int B, int H, int Lmax, int d, float scale, int num_splits,
                    void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Workspace bytes that suffice for every fa_decode call with these B, H,
 * Lmax, d and num_splits, whatever the sequence lengths and seqlens_host
 * (NULL included) and whatever the SM count: a buffer of this size can be
 * allocated once and reused.  With num_splits > 0 it is exact; with automatic
 * chunking it is the bound B * H * s_max * (d + 2) * 4 bytes (plus alignment),
 * s_max = max(ceil(Lmax / 256), min(ceil(Lmax / 64), 1024)) chunks per
 * sequence.  Returns 0 for arguments fa_decode would reject.
 */
FA_API size_t fa_decode_workspace_bytes(int B, int H, int Lmax, int d, int num_splits);

/*
 * The exact workspace bytes of one fa_decode call on the current device:
 * same arguments as there (seqlens_host may be NULL), never more than
 * fa_decode_workspace_bytes(B, H, Lmax, d, num_splits).  Returns 0 for
 * arguments fa_decode would reject.
 */
FA_API size_t fa_decode_workspace_bytes_for_lengths(int B, int H, int Lmax, int d, int num_splits,
                                                    const int32_t *seqlens_host);

/*
 * The split plan fa_decode would use: writes the chunk length in tokens and
 * the largest per-sequence chunk count.  num_sms <= 0 asks the current
 * device; a positive value plans for that many SMs (host-only, no CUDA
 * call).  Returns FA_OK or FA_ERR_INVALID_ARG.
 */
FA_API fa_status fa_decode_plan(int B, int H, int Lmax, int d, int num_splits,
                         const int32_t *seqlens_host, int num_sms,
                         int *chunk_len, int *max_chunks);

/*
 * fa_decode_noalloc -- fa_decode for callers that cannot allocate device
 * memory when they decode (a runtime that gives all device memory to its
 * own pool at start-up and forbids later allocations, a plugin whose host
 * application owns the memory budget, a token loop where cudaMalloc or
 * cudaFree could synchronise the device).  The pages have no counterpart of
 * this entry point; it only changes where the split partials are kept.
 *
 * Arguments and results are those of fa_decode without `workspace` and
 * `workspace_bytes`: the partials go to one array of
 * FA_DECODE_NOALLOC_MAX_BYTES that the library keeps in device memory on
 * every GPU that loads it, until the process exits.  The call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 *   - A request whose fa_decode_workspace_bytes_for_lengths() exceeds
 *     FA_DECODE_NOALLOC_MAX_BYTES returns FA_ERR_WORKSPACE and launches
 *     nothing; use fa_decode with your own workspace for it.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept until fa_shutdown(); after a cudaDeviceReset()
 *     without fa_shutdown() first it is stale, as is the device error word's.
 *   - Every call on a device uses the same array.  Nothing in it needs to
 *     start at zero (each partial is written before it is read), but two
 *     calls that overlap on the GPU, e.g. on two streams, race on it: order
 *     them on one stream or with events.
 */
#define FA_DECODE_NOALLOC_MAX_BYTES (8u << 20) /* 8 MiB */

FA_API fa_status fa_decode_noalloc(const void *q, const void *Kcache, const void *Vcache,
                                   const int32_t *seqlens, const int32_t *seqlens_host,
                                   void *O, float *L,
                                   int B, int H, int Lmax, int d, float scale, int num_splits,
                                   fa_stream_t stream);

/*
 * fa_decode_paged -- fa_decode over a paged KV cache ("CMU 10-423 Lecture 18",
 * section 7 "Efficient decoding I: PagedAttention": the cache is a pool of
 * fixed-size blocks and each sequence reaches its blocks through a block
 * table, so logically consecutive tokens need not be adjacent in memory).
 * The attention computed is exactly fa_decode's over the gathered keys and
 * values; only the addressing differs.
 *
 *   Kpool,Vpool   bf16 [num_blocks, H, block_size, d]: row r of head h in
 *                 physical block p holds one token's key (value).
 *   block_table   DEVICE int32 [B, max_blocks]: token t of sequence b lives
 *                 in physical block block_table[b * max_blocks + t / block_size]
 *                 at row t % block_size.  Only the entries of blocks that
 *                 hold attended tokens are read; the rest may hold anything.
 *   max_blocks    table row length, >= 1; max_blocks * block_size <= 2^30.
 *   seqlens       DEVICE int32 [B], clamped to [0, max_blocks * block_size];
 *                 seqlens_host as in fa_decode.
 *   num_blocks    pool size in blocks, >= 1.
 *   block_size    tokens per block, 1 .. FA_PAGED_MAX_BLOCK_SIZE.  Any value
 *                 is exact; a multiple of 16 keeps each copy >= 2 KB.
 *   O, L, d, scale, num_splits, workspace, stream: as in fa_decode, with
 *                 Lmax = max_blocks * block_size in the workspace queries
 *                 (fa_decode_workspace_bytes and ..._for_lengths).
 *
 * A table entry read on the device that lies outside [0, num_blocks) is
 * never dereferenced: block 0 is read in its place and the device error
 * word records it, so a following fa_device_error() returns
 * FA_ERR_INVALID_ARG with *site = 0x104; the outputs of that call are
 * undefined.
 */
#define FA_PAGED_MAX_BLOCK_SIZE 65536

FA_API fa_status fa_decode_paged(const void *q, const void *Kpool, const void *Vpool,
                                 const int32_t *block_table, int max_blocks,
                                 const int32_t *seqlens, const int32_t *seqlens_host,
                                 void *O, float *L,
                                 int B, int H, int num_blocks, int block_size, int d,
                                 float scale, int num_splits,
                                 void *workspace, size_t workspace_bytes, fa_stream_t stream);

/* Human-readable name of a status code (static string). */
FA_API const char *fa_status_string(fa_status s);

/*
 * Device-side error word of the current device: FA_OK when nothing has
 * been recorded since the last clear; FA_ERR_DEVICE_TIMEOUT when a bounded
 * wait ran out; FA_ERR_INVALID_ARG when a kernel met invalid device data
 * (a paged-cache table entry outside the pool).  The first event recorded
 * wins; its site goes to *site (may be NULL).  Synchronises the device.
 * clear != 0 resets the word.
 */
FA_API fa_status fa_device_error(int clear, int *site);

/*
 * fa_get_last_device_error -- the device error word of the current device,
 * read and then reset, like cudaGetLastError: FA_OK, FA_ERR_DEVICE_TIMEOUT or
 * FA_ERR_INVALID_ARG as in fa_device_error (which also reports the site and
 * can leave the word set).  Synchronises the device.
 */
FA_API fa_status fa_get_last_device_error(void);

/*
 * fa_selftest_wait_timeout -- exercise the bounded-wait failure path.
 * (No counterpart on the pages: a check of this library's failure handling.)
 * Launches one thread that waits, for limit_us microseconds (1 .. 100000),
 * on a barrier nothing arrives at.  The wait gives up, records site 0x301 in
 * the device error word and returns; the context stays usable.  A following
 * fa_device_error() returns FA_ERR_DEVICE_TIMEOUT with *site = 0x301.
 */
FA_API fa_status fa_selftest_wait_timeout(unsigned limit_us, fa_stream_t stream);

/*
 * fa_shutdown -- release what the library keeps between calls.  (No
 * counterpart on the pages: the resource lifetime of this boundary.)
 * That is the streams and events fa_forward_host creates per device, and
 * the per-device lookups every call shares: the device error word's and the
 * fa_decode_noalloc array's addresses, the SM count and the decode CTAs per
 * SM.  It first waits for the work queued on those streams.  Call it with no
 * other library call running on any host thread; the next call sets
 * everything up again.  Call it before cudaDeviceReset(), after which the
 * cached addresses would be stale.  Returns FA_ERR_CUDA if a device could not
 * be selected or synchronised (the remaining state is still released), else
 * FA_OK; with nothing cached it touches no device.
 */
FA_API fa_status fa_shutdown(void);

/* Library ABI version (major * 100 + minor). */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
