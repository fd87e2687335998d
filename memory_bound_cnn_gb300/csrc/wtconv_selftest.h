// Diagnostic kernels of the library (no part of the layer's computation).
#pragma once

#include <cuda_runtime.h>

namespace wtconv {

// One bounded shared-memory barrier wait that nothing completes: it gives up after half a second
// and raises *flag, exactly as a kernel wait of the layer would.
cudaError_t launch_wait_selftest(int *flag, cudaStream_t st);

// Packed-FMA throughput of the current device in TFLOP/s: chains of fma.rn.f32x2 on every SM
// (iters per chain), timed with CUDA events on the legacy default stream; synchronises.
cudaError_t measure_fma_peak(int iters, double *tflops);

}  // namespace wtconv
