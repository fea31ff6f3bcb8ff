// fa_selftest.cu -- exercises the bounded-wait failure path on the GPU.
//
// One thread waits on an mbarrier that nothing will ever arrive at.  The wait
// gives up after the requested time, records kSiteSelfTest in the device
// error word (the same word the attention kernels use) and the kernel returns
// normally: no trap, no fault, no hang, and the context stays usable.
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

__global__ void wait_selftest_kernel(unsigned long long limit_ns, unsigned *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_limit(smem_u32(&bar), 0, limit_ns, err, kSiteSelfTest);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned long long limit_ns, unsigned *err, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace fa
