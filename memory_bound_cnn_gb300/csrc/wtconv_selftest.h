// Diagnostic kernels of the library (no part of the layer's computation).
#pragma once

#include <cuda_runtime.h>

namespace wtconv {

// One bounded shared-memory barrier wait that nothing completes: it gives up after its bounded
// number of tries and raises *flag, exactly as a kernel wait of the layer would.
cudaError_t launch_wait_selftest(int *flag, cudaStream_t st);

}  // namespace wtconv
