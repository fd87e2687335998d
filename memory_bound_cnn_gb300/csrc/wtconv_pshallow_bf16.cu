// Tiled batch-pair shallow kernel instantiations for __nv_bfloat16 activations.
#include "wtconv_pshallow.cuh"

namespace wtconv {

cudaError_t launch_pshallow_bf16(const PsArgs &a, size_t smem, cudaStream_t st) {
    return launch_pshallow_typed<__nv_bfloat16>(a, smem, st);
}
int occupancy_pshallow_bf16(int K, size_t smem, int nthreads, int s) {
    return occupancy_pshallow_typed<__nv_bfloat16>(K, smem, nthreads, s);
}

}  // namespace wtconv
