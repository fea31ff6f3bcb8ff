// fa_decode_noalloc.cu -- fa_decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they decode:
// a serving runtime that hands the whole GPU to its own pool at start-up and
// forbids any later driver allocation, a plugin hosted by an application that
// owns the memory budget, or a latency-critical token loop where cudaMalloc /
// cudaFree could synchronise the device.  For them this entry point keeps the
// split partials in one fixed array that lives in the library's own device
// memory (every GPU that loads the library holds it until the process exits).
// It allocates nothing, and the arithmetic is exactly fa_decode's: the call
// forwards to fa_decode with that array as the workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// The shared scratch: FA_DECODE_NOALLOC_MAX_BYTES, 256-byte aligned like any
// fa_decode workspace.  The name is a host-side stand-in in host code; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_DECODE_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
fa_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return FA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return FA_OK;
}

}  // namespace

namespace fa {
void reset_noalloc_addresses() {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < kMaxDevices; ++i) g_scratch_addr[i] = nullptr;
}
}  // namespace fa

extern "C" FA_API fa_status fa_decode_noalloc(const void *q, const void *Kcache, const void *Vcache,
                                              const int32_t *seqlens, const int32_t *seqlens_host, void *O,
                                              float *L, int B, int H, int Lmax, int d, float scale,
                                              int num_splits, fa_stream_t stream) {
    const size_t need = fa_decode_workspace_bytes_for_lengths(B, H, Lmax, d, num_splits, seqlens_host);
    if (need == 0) {
        // arguments fa_decode rejects: let it report which one
        return fa_decode(q, Kcache, Vcache, seqlens, seqlens_host, O, L, B, H, Lmax, d, scale, num_splits,
                         nullptr, 0, stream);
    }
    if (need > static_cast<size_t>(FA_DECODE_NOALLOC_MAX_BYTES)) return FA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const fa_status s = scratch_address(&scratch);
    if (s != FA_OK) return s;
    return fa_decode(q, Kcache, Vcache, seqlens, seqlens_host, O, L, B, H, Lmax, d, scale, num_splits, scratch,
                     static_cast<size_t>(FA_DECODE_NOALLOC_MAX_BYTES), stream);
}
