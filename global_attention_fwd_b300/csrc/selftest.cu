// selftest.cu -- kernels that exercise the error paths of the library without
// faulting the GPU: a bounded wait on an mbarrier that nothing ever completes
// (the timeout path every real kernel uses: record in the device error word,
// return), and the index check of the debug build.
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

// The index check of the debug build, exercised without an out-of-range access: the kernel asks
// idx_ok() about index n of an n-element range, but the store it guards always goes to element 0
// of a valid one-word buffer.  Debug build: the check fails, is recorded, the store is skipped.
// Normal build: idx_ok() is the constant true and the valid store happens.
__device__ uint32_t g_index_selftest_word;
__global__ void index_selftest_kernel(DevCtl ctl) {
    if (threadIdx.x == 0 && idx_ok(ctl, 1, 1, 98)) g_index_selftest_word = 1u;
}
}  // namespace

cudaError_t launch_wait_selftest(DevCtl ctl, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(ctl);
    return cudaGetLastError();
}

cudaError_t launch_index_selftest(DevCtl ctl, cudaStream_t s) {
    index_selftest_kernel<<<1, 32, 0, s>>>(ctl);
    return cudaGetLastError();
}
}  // namespace zg
