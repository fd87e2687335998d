// Host side of the batch-pair kernels: shared-memory sizes, and the dispatch on the activation
// type to the per-type translation units.
#include "wtconv_pair_dw.cuh"
#include "wtconv_pair_fwd.cuh"

namespace wtconv {

size_t pair_fwd_smem_bytes(const PairArgs &a, int elem_bytes) {
    (void)elem_bytes;
    return pair_fwd_layout(a).total;
}

size_t pair_dw_smem_bytes(const PairArgs &a, int elem_bytes) {
    (void)elem_bytes;
    return pair_dw_layout(a).total;
}

cudaError_t launch_pair_fwd(const PairArgs &a, int dtype, size_t smem, cudaStream_t st) {
    switch (dtype) {
    case 0: return launch_pair_fwd_typed<float>(a, smem, st);
    case 1: return launch_pair_fwd_typed<__nv_bfloat16>(a, smem, st);
    case 2: return launch_pair_fwd_typed<__half>(a, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

int occupancy_pair_fwd(int dtype, int K, size_t smem, int nthreads) {
    switch (dtype) {
    case 0: return occupancy_pair_fwd_typed<float>(K, smem, nthreads);
    case 1: return occupancy_pair_fwd_typed<__nv_bfloat16>(K, smem, nthreads);
    case 2: return occupancy_pair_fwd_typed<__half>(K, smem, nthreads);
    default: return 0;
    }
}

cudaError_t launch_pair_dw(const PairArgs &a, int dtype, size_t smem, cudaStream_t st) {
    switch (dtype) {
    case 0: return launch_pair_dw_typed<float>(a, smem, st);
    case 1: return launch_pair_dw_typed<__nv_bfloat16>(a, smem, st);
    case 2: return launch_pair_dw_typed<__half>(a, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

int occupancy_pair_dw(int dtype, int K, size_t smem, int nthreads) {
    switch (dtype) {
    case 0: return occupancy_pair_dw_typed<float>(K, smem, nthreads);
    case 1: return occupancy_pair_dw_typed<__nv_bfloat16>(K, smem, nthreads);
    case 2: return occupancy_pair_dw_typed<__half>(K, smem, nthreads);
    default: return 0;
    }
}

}  // namespace wtconv
