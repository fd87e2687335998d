// Backward kernels of the WTConv layer.
//
// wtconv_bwd_kernel: one CTA owns channel c and a run of batch entries.  Per plane group it reads
// x and dy once, builds both Haar pyramids on chip (Yhat from x, Ghat from dy) and
//   * (input gradient) convolves Ghat with the 180-degree-rotated folded kernels and writes dx
//     through the same closed-form synthesis as the forward: dx = sum_l A_l^T K_l^T A_l dy + K_b^T dy;
//   * (weight gradients) correlates Ghat^l_s with Yhat^l_s for every tap:
//     dW'^l_s[u,v] = 4^-l sum_{i,j} Ghat[i,j] Yhat[i+u-P, j+v-P], and dy with x for the base kernel,
//     accumulating in registers per lane, reducing across the warp with shuffles (fixed-order
//     butterfly) and across warps and plane groups in shared memory.  Each CTA writes one
//     partial per (channel, tap); no atomics, so the result is deterministic.
// wtconv_dw_finalize_kernel sums the partials over the CTAs of a channel in a fixed order and
// unfolds the scales by the chain rule: dw = s dW', ds = sum_t w dW' (+ b db' for the base), db = s_b db'.
#include "wtconv_device.cuh"

namespace wtconv {

static inline int n_sig(int L) { return 1 + 4 * L; }

size_t bwd_smem_bytes(const Geo &geo, int G, int L, int K) {
    size_t floats = (size_t)G * geo.slot_floats + (size_t)n_sig(L) * wslot_stride(K) + 4 +
                    (size_t)n_sig(L) * kWarps * dw_na(K) + round_up(n_sig(L) + 1, 4);
    return floats * sizeof(float);
}

// Tiles (4x4) of subband sig in one slot, and their column count.
__device__ __forceinline__ void dw_sig_tiles(const Geo &geo, int sig, int &nt, int &tcols, int &lvl) {
    lvl = sig == 0 ? 0 : (sig - 1) / 4 + 1;
    const int h = geo.H >> lvl, w = geo.W >> lvl;
    tcols = round_up(w, 4) / 4;
    nt = (round_up(h, 4) / 4) * tcols;
}

template <int K>
__device__ __forceinline__ void dw_phase(const Geo &geo, const float *slots, int G, const int *cstart,
                                         int nsig, float *dwacc) {
    constexpr int NA = dw_na(K), NA32 = dw_na32(K);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nchunks = cstart[nsig];
    const int c_begin = (warp * nchunks) / kWarps, c_end = ((warp + 1) * nchunks) / kWarps;
    float acc[NA32];
#pragma unroll
    for (int i = 0; i < NA32; ++i) acc[i] = 0.f;
    int cur = -1;
    for (int ch = c_begin; ch < c_end; ++ch) {
        int sig = 0;
        while (ch >= cstart[sig + 1]) ++sig;
        if (sig != cur && cur >= 0) {
            float res[NA32 / 32];
            warp_reduce_scatter<NA32>(acc, res);
#pragma unroll
            for (int blk = 0; blk < NA32 / 32; ++blk) {
                const int t = blk * 32 + lane;
                if (t < NA) dwacc[(cur * kWarps + warp) * NA + t] += res[blk];
            }
#pragma unroll
            for (int i = 0; i < NA32; ++i) acc[i] = 0.f;
        }
        cur = sig;
        int nt, tcols, lvl;
        dw_sig_tiles(geo, sig, nt, tcols, lvl);
        const int item = (ch - cstart[sig]) * 32 + lane;
        if (item < G * nt) {
            const int g = item / nt, e = item - g * nt;
            const int ti = e / tcols, tj = e - ti * tcols;
            const float *slot = slots + (size_t)g * geo.slot_floats;
            const float *ysrc, *gsrc;
            if (lvl == 0) {
                ysrc = slot + geo.off_x;
                gsrc = slot + geo.off_dy;
            } else {
                const int s = (sig - 1) & 3, sub = s * geo.rows[lvl] * geo.pitch[lvl];
                ysrc = slot + geo.off_y[lvl] + sub;
                gsrc = slot + geo.off_g[lvl] + sub;
            }
            dw_tile_4x4<K>(ysrc, gsrc, geo.pitch[lvl], 4 * ti, 4 * tj, acc);
        }
    }
    if (cur >= 0) {
        float res[NA32 / 32];
        warp_reduce_scatter<NA32>(acc, res);
#pragma unroll
        for (int blk = 0; blk < NA32 / 32; ++blk) {
            const int t = blk * 32 + lane;
            if (t < NA) dwacc[(cur * kWarps + warp) * NA + t] += res[blk];
        }
    }
}

template <int K, typename T>
__global__ void __launch_bounds__(kThreads) wtconv_bwd_kernel(const LayerArgs a) {
    extern __shared__ __align__(16) float smem[];
    __shared__ Geo geo;
    if (threadIdx.x == 0) geo = a.geo;
    constexpr int NA = dw_na(K);
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = a.G;
    const int nsig = 1 + 4 * a.L;
    float *slots = smem;
    float *wts = smem + (size_t)G * a.geo.slot_floats;
    float *bias_s = wts + nsig * wslot_stride(K);
    float *dwacc = bias_s + 4;
    int *cstart = reinterpret_cast<int *>(dwacc + nsig * kWarps * NA);

    {
        float4 *s4 = reinterpret_cast<float4 *>(slots);
        const int n4 = G * a.geo.slot_floats / 4;
        for (int i = threadIdx.x; i < n4; i += blockDim.x) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = threadIdx.x; i < nsig * kWarps * NA; i += blockDim.x) dwacc[i] = 0.f;
    }
    if (a.want_dx) stage_weights<K>(a, c, wts, bias_s);
    __syncthreads();
    if (threadIdx.x == 0) {  // chunk table: 32 tiles per chunk, subband-major
        int tot = 0;
        for (int sig = 0; sig < nsig; ++sig) {
            int nt, tcols, lvl;
            dw_sig_tiles(geo, sig, nt, tcols, lvl);
            cstart[sig] = tot;
            tot += (G * nt + 31) / 32;
        }
        cstart[nsig] = tot;
    }
    __syncthreads();

    const T *x = static_cast<const T *>(a.x);
    const T *dy = static_cast<const T *>(a.dy);
    T *dx = static_cast<T *>(a.out);
    const size_t HW = (size_t)a.H * a.W;

    for (int grp = 0; grp < a.groups_per_cta; ++grp) {
        const int b0 = (nbi * a.groups_per_cta + grp) * G;
        if (b0 >= a.B) break;
        for (int g = 0; g < G; ++g) {
            const int b = b0 + g;
            const bool valid = b < a.B;
            const size_t off = ((size_t)(valid ? b : 0) * a.C + c) * HW;
            float *slot = slots + (size_t)g * geo.slot_floats;
            load_plane<T, K / 2>(x + off, valid, slot + geo.off_x, a.H, a.W, geo.pitch[0]);
            load_plane<T, K / 2>(dy + off, valid, slot + geo.off_dy, a.H, a.W, geo.pitch[0]);
        }
        __syncthreads();
        for (int l = 1; l <= a.L; ++l) {
            analysis_level<K / 2>(geo, slots, G, l, geo.off_x, geo.off_y);
            analysis_level<K / 2>(geo, slots, G, l, geo.off_dy, geo.off_g);
            __syncthreads();
        }
        if (a.want_dx) conv_levels<K>(geo, slots, G, geo.off_g, wts);
        dw_phase<K>(geo, slots, G, cstart, nsig, dwacc);
        __syncthreads();
        if (a.want_dx) {
            output_phase<K, T>(a, geo, slots, G, geo.off_dy, wts, 0.f, dx, c, b0);
            __syncthreads();
        }
    }

    // one partial per (channel, subband, tap) for this CTA: sum over warps in a fixed order
    float *part = a.partials + ((size_t)nbi * a.C + c) * nsig * NA;
    for (int i = threadIdx.x; i < nsig * NA; i += blockDim.x) {
        const int sig = i / NA, t = i - sig * NA;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += dwacc[(sig * kWarps + w) * NA + t];
        part[i] = s;
    }
}

// Sum the per-CTA partials of each (channel, subband) in order of CTA index and unfold the
// scales (chain rule through the folding W' = s w, b' = s_b b).  One 64-thread block per
// (channel, subband); thread t owns tap t (thread K*K: the gradient sum of the base bias).
__global__ void __launch_bounds__(64) wtconv_dw_finalize_kernel(const LayerArgs a, float *d_base_w,
                                                                float *d_base_bias, float *d_base_scale,
                                                                float *d_wavelet_w, float *d_wavelet_scale) {
    __shared__ float prod[64];
    const int K = a.K, KK = K * K, NA = KK + 1, nsig = 1 + 4 * a.L;
    const int c = blockIdx.x / nsig, sig = blockIdx.x - c * nsig;
    const int t = threadIdx.x;
    const size_t stride = (size_t)a.C * nsig * NA;
    const float *p = a.partials + ((size_t)c * nsig + sig) * NA;
    float v = 0.f;
    if (t < NA)
        for (int n = 0; n < a.nb; ++n) v += p[n * stride + t];
    const int l = sig == 0 ? 0 : (sig - 1) / 4 + 1;
    size_t ch = 0;
    float scale, wt = 0.f;
    if (sig == 0) {
        scale = a.base_scale[c];
        if (t < KK) wt = a.base_w[(size_t)c * KK + t];
        else if (t == KK) wt = a.base_bias[c];
    } else {
        ch = (size_t)(l - 1) * 4 * a.C + 4 * c + ((sig - 1) & 3);
        scale = a.wavelet_scale[ch];
        v = ldexpf(v, -2 * l);  // the pyramid is unnormalised by 2^l on both operands
        if (t < KK) wt = a.wavelet_w[ch * KK + t];
    }
    if (t < KK) {
        if (sig == 0) d_base_w[(size_t)c * KK + t] = scale * v;
        else d_wavelet_w[ch * KK + t] = scale * v;
    }
    if (sig == 0 && t == KK) d_base_bias[c] = scale * v;
    const bool use = (t < KK) || (sig == 0 && t == KK);
    prod[t] = use ? wt * v : 0.f;
    __syncthreads();
    if (t == 0) {
        float ds = 0.f;
        for (int i = 0; i < NA; ++i) ds += prod[i];
        if (sig == 0) d_base_scale[c] = ds;
        else d_wavelet_scale[ch] = ds;
    }
}

template <int K, typename T>
static cudaError_t launch_bwd_t(const LayerArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_bwd_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_bwd_t(size_t smem) {
    auto kern = wtconv_bwd_kernel<K, T>;
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

cudaError_t launch_backward(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_bwd_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_backward(int dtype, int K, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_bwd_t, smem);
    return 0;
}

cudaError_t launch_dw_finalize(const LayerArgs &a, float *d_base_w, float *d_base_bias, float *d_base_scale,
                               float *d_wavelet_w, float *d_wavelet_scale, cudaStream_t st) {
    const int n = a.C * (1 + 4 * a.L);
    wtconv_dw_finalize_kernel<<<n, 64, 0, st>>>(a, d_base_w, d_base_bias, d_base_scale, d_wavelet_w,
                                                d_wavelet_scale);
    return cudaGetLastError();
}

}  // namespace wtconv
