// selftest.cu -- device-side failure detection check: one thread waits on an
// mbarrier that nothing ever completes, then on a hand-off counter that
// nothing ever increments, through the same bounded waits the layer's kernels
// use; both waits must give up, the kernel records MOE_ERR_DEVICE_TIMEOUT
// (only when both did) and returns normally.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

__device__ int32_t g_never_counted = 0;  // no kernel ever adds to it

__global__ void wait_timeout_probe(int32_t *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_ns(&bar, 0, &abort_flag, limit_ns) &&
        !wait_count_ns(&g_never_counted, 1, &abort_flag, limit_ns))
        record_status(status, MOE_ERR_DEVICE_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout_probe(int32_t *status, uint64_t limit_ns, cudaStream_t s) {
    wait_timeout_probe<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace moe
