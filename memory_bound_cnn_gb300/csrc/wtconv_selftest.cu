// Diagnostic: exercises the bounded-wait failure path of the layer's kernels on purpose, without
// any fault: one thread waits on a shared-memory barrier that no thread and no copy ever
// completes; the wait gives up after its bounded number of tries (about half a second), raises
// the sticky device flag and the kernel returns normally.
#include "wtconv_device.cuh"
#include "wtconv_selftest.h"

namespace wtconv {

namespace {

__global__ void __launch_bounds__(32) wtconv_wait_selftest_kernel(int *flag) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // expects one arrival, which never comes
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, flag);
}

}  // namespace

cudaError_t launch_wait_selftest(int *flag, cudaStream_t st) {
    wtconv_wait_selftest_kernel<<<1, 32, 0, st>>>(flag);
    return cudaGetLastError();
}

}  // namespace wtconv
