// Diagnostics of the library (no part of the layer's computation):
//   * the bounded-wait failure path of the layer's kernels, exercised on purpose without any
//     fault: one thread waits on a shared-memory barrier that no thread and no copy ever
//     completes; the wait gives up after half a second, raises the sticky device flag and the
//     kernel returns normally;
//   * the FP32 packed-FMA throughput of the device: the peak the layer's conv arithmetic (packed
//     fma.rn.f32x2) can reach, the denominator of its ALU roofline.
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

// Independent chains of packed FMAs: each thread runs kChains chains of `iters` dependent
// fma.rn.f32x2 (2 lanes x 2 FLOP each).  The result goes to a sink only when it equals a value it
// never reaches, so the chains cannot be removed.
constexpr int kChains = 8;
__device__ float g_fma_sink;

__global__ void __launch_bounds__(256) wtconv_fma_probe_kernel(int iters, float seed) {
    f2_t acc[kChains];
    const f2_t m = pk2(0.999f, 0.998f), c = pk2(1e-7f, 2e-7f);
#pragma unroll
    for (int i = 0; i < kChains; ++i) acc[i] = pk2(seed + threadIdx.x * 1e-3f + i, seed - i);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[i]) : "l"(m), "l"(c));
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += lo2(acc[i]) + hi2(acc[i]);
    if (s == 1234.5678f) g_fma_sink = s;
}

}  // namespace

cudaError_t measure_fma_peak(int iters, double *tflops) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = sms * 8, threads = 256;  // 8 resident CTAs of 8 warps per SM
    cudaEvent_t a = nullptr, b = nullptr;
    if ((e = cudaEventCreate(&a)) != cudaSuccess) return e;
    if ((e = cudaEventCreate(&b)) != cudaSuccess) { cudaEventDestroy(a); return e; }
    float ms = 0.f;
    wtconv_fma_probe_kernel<<<grid, threads>>>(iters / 4 + 1, 0.5f);  // warm-up (clocks, code load)
    e = cudaEventRecord(a);
    if (e == cudaSuccess) {
        wtconv_fma_probe_kernel<<<grid, threads>>>(iters, 0.25f);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(b);
    if (e == cudaSuccess) e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (e != cudaSuccess) return e;
    const double flop = (double)grid * threads * iters * kChains * 4.0;
    *tflops = ms > 0.f ? flop / (ms * 1e-3) / 1e12 : 0.0;
    return cudaSuccess;
}

cudaError_t launch_wait_selftest(int *flag, cudaStream_t st) {
    wtconv_wait_selftest_kernel<<<1, 32, 0, st>>>(flag);
    return cudaGetLastError();
}

}  // namespace wtconv
