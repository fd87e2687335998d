// Tiled batch-pair weight-gradient kernel instantiations for __half activations.
#include "wtconv_ptile_dw.cuh"

namespace wtconv {

cudaError_t launch_ptile_dw_f16(const PtileArgs &a, size_t smem, cudaStream_t st) {
    return launch_ptile_dw_typed<__half>(a, smem, st);
}
int occupancy_ptile_dw_f16(int K, int LT, int base, size_t smem, int nthreads, int iq) {
    return occupancy_ptile_dw_typed<__half>(K, LT, base, smem, nthreads, iq);
}

}  // namespace wtconv
