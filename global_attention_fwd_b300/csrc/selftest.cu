// selftest.cu -- a kernel whose only job is a bounded wait on an mbarrier that
// nothing ever completes: it exercises the timeout path every real kernel
// uses (record in the device error word, return) without faulting the GPU.
#include "zg_kernels.cuh"

namespace zg {
namespace {
__global__ void wait_selftest_kernel(DevCtl ctl) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, ctl, 99);  // no arrival is ever made
    __syncthreads();
}
}  // namespace

cudaError_t launch_wait_selftest(DevCtl ctl, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(ctl);
    return cudaGetLastError();
}
}  // namespace zg
