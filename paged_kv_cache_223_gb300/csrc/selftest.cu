// selftest.cu -- exercises the bounded-wait path of the copy pipelines without a fault:
// one warp waits on an mbarrier that nothing ever completes.
#include "pa_device.cuh"

namespace pa {

__global__ void wait_selftest_kernel(int *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncwarp();
    // no arrival and no copy is ever issued on this barrier: the bounded wait must give up
    if (!mbar_wait_bounded(b, 0u, limit_ns) && threadIdx.x == 0) set_status(status, STATUS_TIMEOUT);
}

cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace pa
