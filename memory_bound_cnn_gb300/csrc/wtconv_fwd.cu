// Forward kernel of the WTConv layer (also serves the input gradient, which is the same operator
// on dy with every kernel rotated by 180 degrees and no bias).
//
// One CTA owns channel c and a run of batch entries; it holds G whole planes in shared memory
// (fp32, zero-padded) and for each plane group:
//   1. reads the planes once from HBM (16-byte vector loads) -- the only activation read;
//   2. builds the unnormalised Haar pyramid on chip, level by level (butterflies);
//   3. convolves every subband of every level with its folded kernel into Z^l;
//   4. writes each output pixel once: bias + base conv + closed-form synthesis gather.
#include "wtconv_device.cuh"

namespace wtconv {

size_t fwd_smem_bytes(const Geo &geo, int G, int L, int K) {
    size_t floats = (size_t)G * geo.slot_floats + (size_t)(1 + 4 * L) * wslot_stride(K) + 4;
    return floats * sizeof(float);
}

template <int K, typename T>
__global__ void __launch_bounds__(kThreads) wtconv_fwd_kernel(const LayerArgs a) {
    extern __shared__ __align__(16) float smem[];
    __shared__ Geo geo;
    if (threadIdx.x == 0) geo = a.geo;
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = a.G;
    float *slots = smem;
    float *wts = smem + (size_t)G * a.geo.slot_floats;
    float *bias_s = wts + (1 + 4 * a.L) * wslot_stride(K);

    // zero every slot once: borders and ragged margins stay zero from here on
    {
        float4 *s4 = reinterpret_cast<float4 *>(slots);
        const int n4 = G * a.geo.slot_floats / 4;
        for (int i = threadIdx.x; i < n4; i += blockDim.x) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    stage_weights<K>(a, c, wts, bias_s);
    __syncthreads();
    const float bias = *bias_s;
    const T *x = static_cast<const T *>(a.x);
    T *y = static_cast<T *>(a.out);
    const size_t HW = (size_t)a.H * a.W;

    for (int grp = 0; grp < a.groups_per_cta; ++grp) {
        const int b0 = (nbi * a.groups_per_cta + grp) * G;
        if (b0 >= a.B) break;
        for (int g = 0; g < G; ++g) {
            const int b = b0 + g;
            const bool valid = b < a.B;
            load_plane<T, K / 2>(x + ((size_t)(valid ? b : 0) * a.C + c) * HW, valid,
                                 slots + (size_t)g * geo.slot_floats + geo.off_x, a.H, a.W, geo.pitch[0]);
        }
        __syncthreads();
        for (int l = 1; l <= a.L; ++l) {
            analysis_level<K / 2>(geo, slots, G, l, geo.off_x, geo.off_y);
            __syncthreads();
        }
        conv_levels<K>(geo, slots, G, geo.off_y, wts);
        __syncthreads();
        output_phase<K, T>(a, geo, slots, G, geo.off_x, wts, bias, y, c, b0);
        __syncthreads();
    }
}

template <int K, typename T>
static cudaError_t launch_fwd_t(const LayerArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_fwd_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(a.nb * a.C));
    kern<<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_fwd_t(size_t smem) {
    auto kern = wtconv_fwd_kernel<K, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess) return 0;
    return n;
}

#define WTCONV_DISPATCH(K_, DT_, FN, ...)                                                 \
    switch ((K_) * 4 + (DT_)) {                                                           \
    case 3 * 4 + 0: return FN<3, float>(__VA_ARGS__);                                     \
    case 3 * 4 + 1: return FN<3, __nv_bfloat16>(__VA_ARGS__);                             \
    case 3 * 4 + 2: return FN<3, __half>(__VA_ARGS__);                                    \
    case 5 * 4 + 0: return FN<5, float>(__VA_ARGS__);                                     \
    case 5 * 4 + 1: return FN<5, __nv_bfloat16>(__VA_ARGS__);                             \
    case 5 * 4 + 2: return FN<5, __half>(__VA_ARGS__);                                    \
    case 7 * 4 + 0: return FN<7, float>(__VA_ARGS__);                                     \
    case 7 * 4 + 1: return FN<7, __nv_bfloat16>(__VA_ARGS__);                             \
    case 7 * 4 + 2: return FN<7, __half>(__VA_ARGS__);                                    \
    default: break;                                                                       \
    }

cudaError_t launch_forward(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_fwd_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_forward(int dtype, int K, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_fwd_t, smem);
    return 0;
}

}  // namespace wtconv
