// fa_api.cu -- the C ABI of libfa.so: argument validation, split planning,
// workspace layout and kernel launches.  Everything here runs on the host;
// the arithmetic of the method lives in the kernels.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

// Device error word written by bounded waits (see fa_ptx.cuh).
__device__ unsigned g_device_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned *g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
int g_decode_ctas[kMaxDevices][2] = {};

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fa_status current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// Address of the error word on the current device (looked up once per device).
fa_status error_word(unsigned **out) {
    int dev;
    fa_status s = current_device(&dev);
    if (s != FA_OK) return s;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return FA_ERR_CUDA;
        g_err_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_err_ptr[dev];
    return FA_OK;
}

fa_status device_sm_count(int *out) {
    int dev;
    fa_status s = current_device(&dev);
    if (s != FA_OK) return s;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return FA_ERR_CUDA;
        g_sm_count[dev] = n;
    }
    *out = g_sm_count[dev];
    return FA_OK;
}

fa_status device_decode_ctas(int d, int *out) {
    int dev;
    fa_status s = current_device(&dev);
    if (s != FA_OK) return s;
    const int idx = d == 128 ? 1 : 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_decode_ctas[dev][idx]) {
        const int n = decode_ctas_per_sm(d);
        if (n <= 0) return FA_ERR_CUDA;
        g_decode_ctas[dev][idx] = n;
    }
    *out = g_decode_ctas[dev][idx];
    return FA_OK;
}

int clamp_len(int v, int lmax) { return v < 0 ? 0 : (v > lmax ? lmax : v); }

}  // namespace

cudaError_t current_sm_count(int *out) {
    return device_sm_count(out) == FA_OK ? cudaSuccess : cudaErrorInvalidDevice;
}

namespace {

int round_up(long long v, int g) { return static_cast<int>((v + g - 1) / g * g); }

// Split plan ("science-depth M4-055", trade-off 3: the chunk count is chosen
// from the SM count and the sequence length; too many chunks make the
// reduction dominate).  Pure host arithmetic.
//
//   fixed (num_splits > 0): every sequence gets num_splits chunks of
//     ceil(len / num_splits) tokens rounded up to the granule; smax = num_splits.
//   automatic, equal lengths: choose the per-sequence chunk count S that
//     minimises waves(S) * (chunk(S) + overhead), waves counted against the
//     resident CTA slots, so the work divides into whole waves.
//   automatic, mixed lengths: one chunk length c for the batch that balances
//     the per-chunk overhead against the tail of the last wave:
//     c = sqrt(2 * overhead * total_tokens / slots); each sequence then gets
//     ceil(len / c) chunks.
constexpr int kOverheadTokens = 96;  // fixed cost of one CTA, in token-equivalents

void plan_decode(int B, int H, int Lmax, int num_splits, const int32_t *seqlens_host, int slots,
                 int *chunk_len, int *smax) {
    long long total = 0;
    int max_len = 0, min_len = Lmax;
    for (int b = 0; b < B; ++b) {
        const int len = seqlens_host ? clamp_len(seqlens_host[b], Lmax) : Lmax;
        total += len;
        max_len = len > max_len ? len : max_len;
        min_len = len < min_len ? len : min_len;
    }
    total *= H;
    if (max_len <= 0) {  // nothing to attend: one (empty) slot per (b, h)
        *chunk_len = kDecodeGranule;
        *smax = 1;
        return;
    }
    if (num_splits > 0) {
        int c = round_up((max_len + num_splits - 1) / num_splits, kDecodeGranule);
        *chunk_len = c;
        *smax = num_splits;
        return;
    }
    if (slots < 1) slots = 1;
    int c;
    if (min_len == max_len && static_cast<long long>(B) * H * 20 <= 17ll * slots) {
        // equal lengths and room for at least one chunk per sequence in 85 % of the
        // slots: one wave of as many chunks (>= 256 tokens each) as fit in 85 % of
        // the slots.  Measured on B1 H32 L32768 at 3 CTAs per SM: one wave of 256 to
        // 384 CTAs streams 5.85-5.96 TB/s, a full wave (448) 5.78, and a partial
        // second wave (512 or 608 CTAs) 4.8-5.4.
        const long long units = static_cast<long long>(B) * H;
        long long s_fit = (17ll * slots) / (20 * units);
        const long long s_len = (max_len + 4 * kDecodeGranule - 1) / (4 * kDecodeGranule);
        if (s_fit > s_len) s_fit = s_len;
        if (s_fit < 1) s_fit = 1;
        c = round_up((max_len + s_fit - 1) / s_fit, kDecodeGranule);
    } else if (min_len == max_len) {
        const long long units = static_cast<long long>(B) * H;
        const int max_s = (max_len + kDecodeGranule - 1) / kDecodeGranule;
        double best = 1e300;
        c = round_up(max_len, kDecodeGranule);
        for (int s = 1; s <= max_s && s <= 1024; ++s) {
            const int cs = round_up((max_len + s - 1) / s, kDecodeGranule);
            const int ns = (max_len + cs - 1) / cs;
            const long long ctas = units * ns;
            const long long waves = (ctas + slots - 1) / slots;
            const double cost = static_cast<double>(waves) * (cs + kOverheadTokens);
            if (cost < best - 1e-9) {
                best = cost;
                c = cs;
            }
        }
    } else {
        const double opt = std::sqrt(2.0 * kOverheadTokens * static_cast<double>(total) / slots);
        c = round_up(static_cast<long long>(opt), kDecodeGranule);
        if (c < 4 * kDecodeGranule) c = 4 * kDecodeGranule;
        const int cmax = round_up(max_len, kDecodeGranule);
        if (c > cmax) c = cmax;
    }
    *chunk_len = c;
    *smax = (max_len + c - 1) / c;
}

// The largest per-sequence chunk count plan_decode can return for sequences of
// at most Lmax tokens, whatever the lengths and the SM count: a fixed count is
// used as given; the automatic plans use chunks of >= 4 granules (one wave, or
// mixed lengths), or of >= 1 granule with at most 1024 chunks (several waves of
// equal lengths).
int smax_bound(int Lmax, int num_splits) {
    if (num_splits > 0) return num_splits;
    const long long g1 = (static_cast<long long>(Lmax) + kDecodeGranule - 1) / kDecodeGranule;
    const long long g4 = (static_cast<long long>(Lmax) + 4 * kDecodeGranule - 1) / (4 * kDecodeGranule);
    long long s = g1 < 1024 ? g1 : 1024;
    if (g4 > s) s = g4;
    return static_cast<int>(s < 1 ? 1 : s);
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

size_t workspace_for(int B, int H, int smax, int d) {
    const size_t slots = static_cast<size_t>(B) * H * smax;
    return align256(slots * d * sizeof(float)) + align256(slots * 2 * sizeof(float));
}

bool decode_shape_ok(int B, int H, int Lmax, int d) {
    return B >= 1 && H >= 1 && Lmax >= 1 && B <= 65535 && H <= 65535 && (d == 64 || d == 128);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 101; }

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    }
    return "FA_ERR_UNKNOWN";
}

fa_status fa_device_error(int clear, int *site) {
    unsigned *ptr = nullptr;
    fa_status s = error_word(&ptr);
    if (s != FA_OK) return s;
    if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, ptr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    if (clear) {
        const unsigned zero = 0;
        if (cudaMemcpy(ptr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (site) *site = static_cast<int>(v & 0x3FFFFFFFu);
    if (!v) return FA_OK;
    return (v & 0x40000000u) ? FA_ERR_INVALID_ARG : FA_ERR_DEVICE_TIMEOUT;
}

fa_status fa_selftest_wait_timeout(unsigned limit_us, fa_stream_t stream) {
    if (limit_us < 1 || limit_us > 100000) return FA_ERR_INVALID_ARG;
    unsigned *err = nullptr;
    fa_status s = error_word(&err);
    if (s != FA_OK) return s;
    if (launch_wait_selftest(1000ull * limit_us, err, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

fa_status fa_decode_plan(int B, int H, int Lmax, int d, int num_splits, const int32_t *seqlens_host,
                         int num_sms, int *chunk_len, int *max_chunks) {
    if (!chunk_len || !max_chunks || !decode_shape_ok(B, H, Lmax, d)) return FA_ERR_INVALID_ARG;
    int slots = 1;
    if (num_splits > 0) {
        // a fixed chunk count needs no device information
    } else if (num_sms > 0) {
        slots = num_sms * 3;   // the split kernel's two-stage ring fits three CTAs per SM
    } else {
        int sms = 0, per = 0;
        fa_status s = device_sm_count(&sms);
        if (s != FA_OK) return s;
        s = device_decode_ctas(d, &per);
        if (s != FA_OK) return s;
        slots = sms * per;
    }
    plan_decode(B, H, Lmax, num_splits, seqlens_host, slots, chunk_len, max_chunks);
    return FA_OK;
}

size_t fa_decode_workspace_bytes_for_lengths(int B, int H, int Lmax, int d, int num_splits,
                                             const int32_t *seqlens_host) {
    if (!decode_shape_ok(B, H, Lmax, d)) return 0;
    int chunk = 0, smax = 0;
    if (num_splits > 0) {
        smax = num_splits;
    } else if (fa_decode_plan(B, H, Lmax, d, num_splits, seqlens_host, 0, &chunk, &smax) != FA_OK) {
        return 0;
    }
    return workspace_for(B, H, smax, d);
}

size_t fa_decode_workspace_bytes(int B, int H, int Lmax, int d, int num_splits) {
    if (!decode_shape_ok(B, H, Lmax, d)) return 0;
    return workspace_for(B, H, smax_bound(Lmax, num_splits), d);
}

fa_status fa_get_last_device_error(void) { return fa_device_error(1, nullptr); }

}  // extern "C"

namespace fa {
namespace {

// Shared body of fa_decode and fa_decode_paged: `paged` carries the block
// table (nullptr for a contiguous cache), in which case Lmax = max_blocks * bs.
struct PagedArgs {
    const int32_t *block_table;
    int block_size, max_blocks, num_blocks;
};

fa_status decode_impl(const void *q, const void *Kcache, const void *Vcache, const int32_t *seqlens,
                      const int32_t *seqlens_host, void *O, float *L, int B, int H, int Lmax, int d,
                      float scale, int num_splits, void *workspace, size_t workspace_bytes,
                      const PagedArgs &paged, cudaStream_t stream) {
    if (!q || !Kcache || !Vcache || !seqlens || !O) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Lmax < 1 || B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(Kcache, 16) || !aligned(Vcache, 16) || !aligned(O, 16) ||
        !aligned(seqlens, 4) || (L && !aligned(L, 4)))
        return FA_ERR_INVALID_ARG;
    if (!(std::isfinite(scale))) return FA_ERR_INVALID_ARG;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d));

    int chunk = 0, smax = 0;
    fa_status s = fa_decode_plan(B, H, Lmax, d, num_splits, seqlens_host, 0, &chunk, &smax);
    if (s != FA_OK) return s;
    if (smax < 1 || smax > 65535 * 32) return FA_ERR_UNSUPPORTED;
    const size_t need = workspace_for(B, H, smax, d);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return FA_ERR_WORKSPACE;

    unsigned *err = nullptr;
    s = error_word(&err);
    if (s != FA_OK) return s;

    DecodeParams p;
    std::memset(&p, 0, sizeof p);
    const size_t slots = static_cast<size_t>(B) * H * smax;
    p.q = q;
    p.K = Kcache;
    p.V = Vcache;
    p.seqlens = seqlens;
    p.part_o = static_cast<float *>(workspace);
    p.part_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                          align256(slots * d * sizeof(float)));
    p.O = O;
    p.L = L;
    p.B = B;
    p.H = H;
    p.Lmax = Lmax;
    p.num_splits = num_splits > 0 ? num_splits : 0;
    p.chunk_len = chunk;
    p.smax = smax;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    p.block_table = paged.block_table;
    p.block_size = paged.block_size;
    p.max_blocks = paged.max_blocks;
    p.num_blocks = paged.num_blocks;
    if (launch_decode(p, d, stream) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_decode(const void *q, const void *Kcache, const void *Vcache, const int32_t *seqlens,
                    const int32_t *seqlens_host, void *O, float *L, int B, int H, int Lmax, int d,
                    float scale, int num_splits, void *workspace, size_t workspace_bytes,
                    fa_stream_t stream) {
    const PagedArgs contiguous = {nullptr, 0, 0, 0};
    return decode_impl(q, Kcache, Vcache, seqlens, seqlens_host, O, L, B, H, Lmax, d, scale, num_splits,
                       workspace, workspace_bytes, contiguous, static_cast<cudaStream_t>(stream));
}

fa_status fa_decode_paged(const void *q, const void *Kpool, const void *Vpool, const int32_t *block_table,
                          int max_blocks, const int32_t *seqlens, const int32_t *seqlens_host, void *O,
                          float *L, int B, int H, int num_blocks, int block_size, int d, float scale,
                          int num_splits, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    if (!block_table || !aligned(block_table, 4)) return FA_ERR_INVALID_ARG;
    if (max_blocks < 1 || num_blocks < 1 || block_size < 1 || block_size > FA_PAGED_MAX_BLOCK_SIZE)
        return FA_ERR_INVALID_ARG;
    const long long cap = static_cast<long long>(max_blocks) * block_size;
    if (cap > (1ll << 30)) return FA_ERR_UNSUPPORTED;
    const PagedArgs paged = {block_table, block_size, max_blocks, num_blocks};
    return decode_impl(q, Kpool, Vpool, seqlens, seqlens_host, O, L, B, H, static_cast<int>(cap), d, scale,
                       num_splits, workspace, workspace_bytes, paged, static_cast<cudaStream_t>(stream));
}

size_t fa_forward_fp8_workspace_bytes(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || B > 65535 || H > 65535 || d != 128) return 0;
    return align256(static_cast<size_t>(B) * H * N * d * 2);
}

fa_status fa_forward_fp8(const void *Q8, const void *K8, const void *V8, void *O, float *L, int B, int H,
                         int N, int d, int causal, float scale, const int32_t *key_len, void *workspace,
                         size_t workspace_bytes, fa_stream_t stream) {
    if (!Q8 || !K8 || !V8 || !O) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(Q8, 16) || !aligned(K8, 16) || !aligned(V8, 16) || !aligned(O, 16) || (L && !aligned(L, 4)) ||
        (key_len && !aligned(key_len, 4)))
        return FA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * N > (1ll << 40)) return FA_ERR_UNSUPPORTED;
    if (!(std::isfinite(scale))) return FA_ERR_INVALID_ARG;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d));
    const size_t need = fa_forward_fp8_workspace_bytes(B, H, N, d);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return FA_ERR_WORKSPACE;

    unsigned *err = nullptr;
    fa_status s = error_word(&err);
    if (s != FA_OK) return s;
    const long long n = static_cast<long long>(B) * H * N * d;
    if (launch_e4m3_to_bf16(V8, workspace, n, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;

    PrefillParams p;
    std::memset(&p, 0, sizeof p);
    p.Q = Q8;
    p.K = K8;
    p.V = workspace;
    p.O = O;
    p.L = L;
    p.key_len = key_len;
    p.B = B;
    p.H = H;
    p.N = N;
    p.causal = causal;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    p.qk_e4m3 = 1;
    if (launch_prefill(p, d, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

size_t fa_backward_workspace_bytes(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1 || B > 65535 || H > 65535 || (d != 64 && d != 128)) return 0;
    return align256(static_cast<size_t>(B) * H * N * sizeof(float));
}

size_t fa_backward_atomic_dq_workspace_bytes(int B, int H, int N, int d) {
    const size_t dbytes = fa_backward_workspace_bytes(B, H, N, d);
    if (d != 64 || dbytes == 0) return 0;
    return dbytes + align256(static_cast<size_t>(B) * H * N * d * sizeof(float));
}

}  // extern "C"

namespace {

// fa_backward and fa_backward_atomic_dq: the same validation and parameters; the
// second also hands the dK/dV CTAs an fp32 dQ accumulator after D in the workspace.
fa_status backward_impl(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *L,
                        void *dQ, void *dK, void *dV, int B, int H, int N, int d, int causal, float scale,
                        const int32_t *key_len, void *workspace, size_t workspace_bytes, fa_stream_t stream,
                        bool atomic_dq) {
    if (!Q || !K || !V || !O || !dO || !L || !dQ || !dK || !dV) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (atomic_dq && d != 64) return FA_ERR_UNSUPPORTED;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(dO, 16) ||
        !aligned(dQ, 16) || !aligned(dK, 16) || !aligned(dV, 16) || !aligned(L, 4) ||
        (key_len && !aligned(key_len, 4)))
        return FA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * N > (1ll << 40)) return FA_ERR_UNSUPPORTED;
    if (!(std::isfinite(scale))) return FA_ERR_INVALID_ARG;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d));
    const size_t need =
        atomic_dq ? fa_backward_atomic_dq_workspace_bytes(B, H, N, d) : fa_backward_workspace_bytes(B, H, N, d);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return FA_ERR_WORKSPACE;

    unsigned *err = nullptr;
    fa_status s = error_word(&err);
    if (s != FA_OK) return s;

    BwdParams p;
    std::memset(&p, 0, sizeof p);
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.O = O;
    p.dO = dO;
    p.L = L;
    p.Dvec = static_cast<float *>(workspace);
    p.dQ = dQ;
    p.dK = dK;
    p.dV = dV;
    p.key_len = key_len;
    p.B = B;
    p.H = H;
    p.N = N;
    p.causal = causal;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    if (atomic_dq)
        p.dq_accum = reinterpret_cast<float *>(static_cast<char *>(workspace) + fa_backward_workspace_bytes(B, H, N, d));
    if (launch_backward(p, d, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_backward(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                      const float *L, void *dQ, void *dK, void *dV, int B, int H, int N, int d, int causal,
                      float scale, const int32_t *key_len, void *workspace, size_t workspace_bytes,
                      fa_stream_t stream) {
    return backward_impl(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, causal, scale, key_len, workspace,
                         workspace_bytes, stream, false);
}

fa_status fa_backward_atomic_dq(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                                const float *L, void *dQ, void *dK, void *dV, int B, int H, int N, int d,
                                int causal, float scale, const int32_t *key_len, void *workspace,
                                size_t workspace_bytes, fa_stream_t stream) {
    return backward_impl(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, d, causal, scale, key_len, workspace,
                         workspace_bytes, stream, true);
}

}  // extern "C"

namespace {

fa_status forward_impl(const void *Q, const void *K, const void *V, void *O, float *L, int B, int H, int N, int d,
                       int causal, float scale, const int32_t *key_len, unsigned *tile_count,
                       cudaStream_t stream) {
    if (!Q || !K || !V || !O) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
        (L && !aligned(L, 4)) || (key_len && !aligned(key_len, 4)))
        return FA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * N > (1ll << 40)) return FA_ERR_UNSUPPORTED;
    if (!(std::isfinite(scale))) return FA_ERR_INVALID_ARG;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d));

    unsigned *err = nullptr;
    fa_status s = error_word(&err);
    if (s != FA_OK) return s;

    PrefillParams p;
    std::memset(&p, 0, sizeof p);
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.O = O;
    p.L = L;
    p.key_len = key_len;
    p.B = B;
    p.H = H;
    p.N = N;
    p.causal = causal;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    p.tile_count = tile_count;
    if (tile_count &&
        cudaMemsetAsync(tile_count, 0, static_cast<size_t>(B) * H * 2 * sizeof(unsigned), stream) != cudaSuccess)
        return FA_ERR_CUDA;
    if (launch_prefill(p, d, stream) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_forward(const void *Q, const void *K, const void *V, void *O, float *L, int B, int H,
                     int N, int d, int causal, float scale, const int32_t *key_len,
                     fa_stream_t stream) {
    return forward_impl(Q, K, V, O, L, B, H, N, d, causal, scale, key_len, nullptr,
                        static_cast<cudaStream_t>(stream));
}

fa_status fa_forward_count_tiles(const void *Q, const void *K, const void *V, void *O, float *L, int B, int H,
                                 int N, int d, int causal, float scale, const int32_t *key_len,
                                 unsigned *tile_counts, fa_stream_t stream) {
    if (!tile_counts || !aligned(tile_counts, 4)) return FA_ERR_INVALID_ARG;
    return forward_impl(Q, K, V, O, L, B, H, N, d, causal, scale, key_len, tile_counts,
                        static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// fa_forward_host: a group is `hg` consecutive heads of one batch element; a
// slot holds one group's Q, K, V, O and L on the device.
constexpr size_t kHostGroupBytes = 16u << 20;  // automatic group: Q slice <= 16 MiB
constexpr int kHostSlots = 3;                  // groups in flight

struct HostPlan {
    int hg = 0;            // heads per group
    int groups = 0;        // B * H / hg
    int slots = 0;
    size_t tile = 0;       // bytes of one group's Q (= K = V = O) slice, 256-aligned
    size_t lrows = 0;      // bytes of one group's L slice, 256-aligned
    size_t slot = 0;       // 4 * tile + lrows
    size_t keylen = 0;     // device copy of key_len
    size_t total = 0;
};

bool host_plan(int B, int H, int N, int d, int heads_per_group, HostPlan *pl) {
    if (B < 1 || H < 1 || N < 1 || B > 65535 || H > 65535 || (d != 64 && d != 128)) return false;
    if (static_cast<long long>(B) * H * N > (1ll << 40)) return false;
    const size_t head = static_cast<size_t>(N) * d * 2;
    int hg = heads_per_group;
    if (hg == 0) {
        hg = 1;
        for (int c = 1; c <= H; ++c)
            if (H % c == 0 && static_cast<size_t>(c) * head <= kHostGroupBytes) hg = c;
    }
    if (hg < 1 || hg > H || H % hg != 0) return false;
    pl->hg = hg;
    pl->groups = static_cast<int>(static_cast<long long>(B) * H / hg);
    pl->slots = pl->groups < kHostSlots ? pl->groups : kHostSlots;
    pl->tile = align256(static_cast<size_t>(hg) * head);
    pl->lrows = align256(static_cast<size_t>(hg) * N * sizeof(float));
    pl->slot = 4 * pl->tile + pl->lrows;
    pl->keylen = align256(static_cast<size_t>(B) * sizeof(int32_t));
    pl->total = pl->slots * pl->slot + pl->keylen;
    return true;
}

// Internal streams and events of fa_forward_host, created once per device.
// up copies every group's Q, K, V in, in group order, so the first group's
// inputs are complete after one group's worth of copy time.  Slot stream
// st[i] runs the kernel of each group that uses slot i and copies its O and L
// out; the groups' kernels overlap across slots.  Per slot: h2d (inputs
// landed), d2h (outputs left, the slot may be refilled).
struct HostStreams {
    cudaStream_t up, st[kHostSlots];
    cudaEvent_t start, h2d[kHostSlots], d2h[kHostSlots];
    // Held by a call while it enqueues on these streams and records these
    // events, so calls from several host threads on one device queue their
    // work one after the other instead of interleaving event records.
    std::mutex enqueue;
};

// fa_forward_host's streams and events, created on a device's first call and
// kept until fa_shutdown
std::mutex g_host_mu;
HostStreams *g_host[kMaxDevices] = {};

void destroy_host_streams(HostStreams *h) {
    cudaStreamDestroy(h->up);
    for (int i = 0; i < kHostSlots; ++i) {
        cudaStreamDestroy(h->st[i]);
        cudaEventDestroy(h->h2d[i]);
        cudaEventDestroy(h->d2h[i]);
    }
    cudaEventDestroy(h->start);
    delete h;
}

cudaError_t host_streams(HostStreams **out) {
    auto &per_dev = g_host;
    auto &mu = g_host_mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!per_dev[dev]) {
        HostStreams *h = new HostStreams;
        e = cudaStreamCreateWithFlags(&h->up, cudaStreamNonBlocking);
        for (int i = 0; i < kHostSlots && e == cudaSuccess; ++i) {
            e = cudaStreamCreateWithFlags(&h->st[i], cudaStreamNonBlocking);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->h2d[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->d2h[i], cudaEventDisableTiming);
        }
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->start, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;   // (the partial set is leaked: creation failing is fatal anyway)
        per_dev[dev] = h;
    }
    *out = per_dev[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t fa_forward_host_workspace_bytes(int B, int H, int N, int d, int heads_per_group) {
    HostPlan pl;
    return host_plan(B, H, N, d, heads_per_group, &pl) ? pl.total : 0;
}

fa_status fa_forward_host(const void *Qh, const void *Kh, const void *Vh, void *Oh, float *Lh, int B, int H,
                          int N, int d, int causal, float scale, const int32_t *key_len_host,
                          int heads_per_group, void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    if (!Qh || !Kh || !Vh || !Oh) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * H * N > (1ll << 40)) return FA_ERR_UNSUPPORTED;
    if (!(std::isfinite(scale))) return FA_ERR_INVALID_ARG;
    HostPlan pl;
    if (!host_plan(B, H, N, d, heads_per_group, &pl)) return FA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pl.total || !aligned(workspace, 256)) return FA_ERR_WORKSPACE;
    if (scale <= 0.f) scale = 1.0f / std::sqrt(static_cast<float>(d));

    unsigned *err = nullptr;
    fa_status s = error_word(&err);
    if (s != FA_OK) return s;
    HostStreams *hs = nullptr;
    if (host_streams(&hs) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> serial(hs->enqueue);
    const cudaStream_t caller = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *kl_dev = key_len_host ? reinterpret_cast<int32_t *>(ws + pl.slots * pl.slot) : nullptr;

    const cudaStream_t up = hs->up;
    bool ok = cudaEventRecord(hs->start, caller) == cudaSuccess && cudaStreamWaitEvent(up, hs->start, 0) == cudaSuccess;
    for (int i = 0; ok && i < pl.slots; ++i) ok = cudaStreamWaitEvent(hs->st[i], hs->start, 0) == cudaSuccess;
    // the kernels read key_len after the first group's inputs, which follow it on `up`
    if (ok && kl_dev)
        ok = cudaMemcpyAsync(kl_dev, key_len_host, static_cast<size_t>(B) * sizeof(int32_t), cudaMemcpyHostToDevice,
                             up) == cudaSuccess;
    const size_t head_elems = static_cast<size_t>(N) * d;
    const size_t bytes = static_cast<size_t>(pl.hg) * head_elems * 2;
    for (int g = 0; ok && g < pl.groups; ++g) {
        // slot g % slots; each event is waited on before its next record (host order)
        const int i = g % pl.slots;
        uint8_t *slot = ws + i * pl.slot;
        uint8_t *q = slot, *k = slot + pl.tile, *v = slot + 2 * pl.tile, *o = slot + 3 * pl.tile;
        float *l = reinterpret_cast<float *>(slot + 4 * pl.tile);
        const size_t bh0 = static_cast<size_t>(g) * pl.hg;   // first (batch, head) of the group
        const int b = static_cast<int>(bh0 / H);
        const size_t off = bh0 * head_elems * 2;
        // inputs: after the slot's previous outputs have left
        if (g >= pl.slots) ok = cudaStreamWaitEvent(up, hs->d2h[i], 0) == cudaSuccess;
        ok = ok &&
             cudaMemcpyAsync(q, static_cast<const uint8_t *>(Qh) + off, bytes, cudaMemcpyHostToDevice, up) ==
                 cudaSuccess &&
             cudaMemcpyAsync(k, static_cast<const uint8_t *>(Kh) + off, bytes, cudaMemcpyHostToDevice, up) ==
                 cudaSuccess &&
             cudaMemcpyAsync(v, static_cast<const uint8_t *>(Vh) + off, bytes, cudaMemcpyHostToDevice, up) ==
                 cudaSuccess &&
             cudaEventRecord(hs->h2d[i], up) == cudaSuccess;
        if (!ok) break;
        PrefillParams p;
        std::memset(&p, 0, sizeof p);
        p.Q = q;
        p.K = k;
        p.V = v;
        p.O = o;
        p.L = Lh ? l : nullptr;
        p.key_len = kl_dev ? kl_dev + b : nullptr;
        p.B = 1;
        p.H = pl.hg;
        p.N = N;
        p.causal = causal;
        p.scale_log2 = scale * 1.4426950408889634f;
        p.err = err;
        const cudaStream_t st = hs->st[i];
        ok = cudaStreamWaitEvent(st, hs->h2d[i], 0) == cudaSuccess && launch_prefill(p, d, st) == cudaSuccess &&
             cudaMemcpyAsync(static_cast<uint8_t *>(Oh) + off, o, bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess;
        if (ok && Lh)
            ok = cudaMemcpyAsync(Lh + bh0 * N, l, static_cast<size_t>(pl.hg) * N * sizeof(float),
                                 cudaMemcpyDeviceToHost, st) == cudaSuccess;
        if (ok) ok = cudaEventRecord(hs->d2h[i], st) == cudaSuccess;
    }
    // the caller's stream waits for every internal stream, also after a failure
    bool joined = cudaEventRecord(hs->h2d[0], up) == cudaSuccess &&
                  cudaStreamWaitEvent(caller, hs->h2d[0], 0) == cudaSuccess;
    for (int i = 0; i < pl.slots; ++i)
        joined = cudaEventRecord(hs->d2h[i], hs->st[i]) == cudaSuccess &&
                 cudaStreamWaitEvent(caller, hs->d2h[i], 0) == cudaSuccess && joined;
    return ok && joined ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

extern "C" fa_status fa_shutdown(void) {
    fa_status st = FA_OK;
    {
        std::lock_guard<std::mutex> lock(g_host_mu);
        int cur = -1;
        bool have_cur = false;
        for (int dev = 0; dev < kMaxDevices; ++dev) {
            HostStreams *h = g_host[dev];
            if (!h) continue;
            if (!have_cur) have_cur = cudaGetDevice(&cur) == cudaSuccess;
            // the calls that used these streams are complete before they go away
            if (cudaSetDevice(dev) != cudaSuccess) {
                st = FA_ERR_CUDA;
            } else {
                cudaError_t e = cudaStreamSynchronize(h->up);
                for (int i = 0; i < kHostSlots; ++i) {
                    const cudaError_t ei = cudaStreamSynchronize(h->st[i]);
                    if (e == cudaSuccess) e = ei;
                }
                if (e != cudaSuccess) st = FA_ERR_CUDA;
                destroy_host_streams(h);
            }
            g_host[dev] = nullptr;
        }
        if (have_cur && cur >= 0) cudaSetDevice(cur);
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int dev = 0; dev < kMaxDevices; ++dev) {
            g_err_ptr[dev] = nullptr;
            g_sm_count[dev] = 0;
            g_decode_ctas[dev][0] = g_decode_ctas[dev][1] = 0;
        }
    }
    fa::reset_noalloc_addresses();
    return st;
}
