// Batch-pair weight-gradient kernels instantiated for float activations (one translation unit
// per activation type, apart from the forward's, so they compile in parallel).
#include "wtconv_pair_dw.cuh"

namespace wtconv {

template <>
cudaError_t launch_pair_dw_typed<float>(const PairArgs &a, size_t smem, cudaStream_t st) {
    switch (a.K) {
    case 3: return launch_pair_dw_t<3, float>(a, smem, st);
    case 5: return launch_pair_dw_t<5, float>(a, smem, st);
    case 7: return launch_pair_dw_t<7, float>(a, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

template <>
int occupancy_pair_dw_typed<float>(int K, size_t smem, int nthreads) {
    switch (K) {
    case 3: return occ_pair_dw_t<3, float>(smem, nthreads);
    case 5: return occ_pair_dw_t<5, float>(smem, nthreads);
    case 7: return occ_pair_dw_t<7, float>(smem, nthreads);
    default: return 0;
    }
}

}  // namespace wtconv
