// Self-test of the bounded device wait used by every kernel of the library:
// one thread waits on an mbarrier that nothing ever completes, gives up after
// the time limit and reports KVDEC_DEVERR_TIMEOUT.  The kernel then returns
// normally, so the CUDA context stays usable.
#include "common.cuh"
#include "kernels.h"

namespace kvdec {

__global__ void selftest_wait_kernel(uint64_t timeout_ns, uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(b, 0, timeout_ns)) report(err, KVDEC_DEVERR_TIMEOUT);
}

cudaError_t launch_selftest_wait(uint64_t timeout_ns, uint32_t* err, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(timeout_ns, err);
    return cudaGetLastError();
}

}  // namespace kvdec
