// Weight-gradient kernels of the WTConv layer.
//
// wtconv_dw_kernel: each CTA owns channel c and a run of batch entries, walked in groups of G
// planes.  Per group it reads x and dy once, builds both Haar pyramids on chip (Yhat from x,
// Ghat from dy) and correlates them tap by tap:
//     dW'^l_s[u, v] = 4^-l sum_{i,j} Ghat^l_s[i, j] Yhat^l_s[i+u-P, j+v-P]      (level l, subband s)
//     dw'_b[u, v]   =      sum_{h,w} dy[h, w] x[h+u-P, w+v-P],   db' = sum dy  (base path)
// Every thread is pinned to one of these 1+4L correlations for the whole CTA and owns a fixed
// share of its sliding-window items, so its k*k tap sums stay in registers (packed f32x2 pairs)
// across all planes; they are reduced once, at the end, in a fixed order -- no atomics, so the
// result is deterministic.  With L >= 3, when the items of levels >= 3 fit on one warp at the same
// items per thread, that warp is the CTA's last: it builds levels >= 3 of both pyramids while the
// other threads already correlate levels 0 .. 2.  Each CTA writes one partial per (channel, subband, tap).
// wtconv_dw_finalize_kernel sums the partials of a channel in CTA order and unfolds the scales
// by the chain rule through the folding W' = s w, b' = s_b b: dw = s dW', ds = sum_t w dW'
// (+ b db' for the base path), db = s_b db'.
#include "wtconv_analysis.cuh"

namespace wtconv {

static inline int n_sig(int L) { return 1 + 4 * L; }

size_t dw_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off) {
    (void)L;
    size_t slots = (size_t)G * geo.slot_floats * sizeof(float);
    if (stage_off) *stage_off = (int)slots;
    if (stage) slots += 2 * (size_t)G * geo.H * geo.W * elem_bytes;
    const size_t red = (size_t)kMaxThreads * (2 * K * K + 1) * sizeof(float);
    const size_t bytes = slots > red ? slots : red;
    return (bytes + 15) / 16 * 16;
}

// Correlation images: ci = 0 the base path (dy with the padded x, column-pair items of kRows x
// kCols pixels, the two halves of each accumulator pair are partial sums of the same tap);
// ci = 1 + 2(l-1) + pp the level-l subband pair pp (Ghat with Yhat, items of kRows x kColsL
// positions, the halves are the two subbands).
template <int K, typename T>
__global__ void __launch_bounds__(kMaxThreads, (K <= 5 ? 2 : 1)) wtconv_dw_kernel(const LayerArgs a) {
    constexpr int P = K / 2, KK = K * K, NA = KK + 1, NR = 2 * KK + 1;
    constexpr int kMaxImg = 1 + 2 * kMaxLevels;
    extern __shared__ __align__(16) float smem[];
    __shared__ Geo geo;
    __shared__ int tstart[kMaxImg + 1], tend[kMaxImg];
    __shared__ int per_thread, per_thread_deep, split;
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = a.G, nimg = 1 + 2 * a.L, nsig = 1 + 4 * a.L;
    float *slots = smem;

    if (threadIdx.x == 0) {
        geo = a.geo;
        const int nt = blockDim.x;
        auto items = [&](int ci) {
            const int l = ci == 0 ? 0 : (ci - 1) / 2 + 1;
            return G * a.geo.rseg[l] * a.geo.cstr[l];
        };
        int tot = 0;
        for (int ci = 0; ci < nimg; ++ci) tot += items(ci);
        // items per thread d: the smallest d for which every image's items fit on whole threads
        int d = (tot + nt - 1) / nt;
        if (d < 1) d = 1;
        for (;; ++d) {
            int need = 0;
            for (int ci = 0; ci < nimg; ++ci) need += (items(ci) + d - 1) / d;
            if (need <= nt) break;
        }
        // the split layout at the same d: levels 0 .. 2 (images 0 .. 4) on threads [0, nt - 32),
        // levels >= 3 on the last warp with the fewest items per thread dd that fit it (the warp
        // builds those levels first, so fewer items keep it off the critical path)
        const int cdeep = 5;
        int lo = 0;
        for (int ci = 0; ci < cdeep && ci < nimg; ++ci) lo += (items(ci) + d - 1) / d;
        int dd = 1;
        for (;; ++dd) {
            int hi = 0;
            for (int ci = cdeep; ci < nimg; ++ci) hi += (items(ci) + dd - 1) / dd;
            if (hi <= 32 || dd >= d) break;
        }
        int hi = 0;
        for (int ci = cdeep; ci < nimg; ++ci) hi += (items(ci) + dd - 1) / dd;
        split = (a.L >= 3 && nt >= 128 && lo <= nt - 32 && hi <= 32) ? 1 : 0;
        int t0 = 0;
        for (int ci = 0; ci < nimg; ++ci) {
            if (split && ci == cdeep) t0 = nt - 32;
            tstart[ci] = t0;
            t0 += (items(ci) + (split && ci >= cdeep ? dd : d) - 1) / (split && ci >= cdeep ? dd : d);
            tend[ci] = t0;
        }
        tstart[nimg] = t0;
        per_thread = d;
        per_thread_deep = split ? dd : d;
    }
    {
        float4 *s4 = reinterpret_cast<float4 *>(slots);
        const int n4 = G * a.geo.slot_floats / 4;
        for (int i = threadIdx.x; i < n4; i += blockDim.x) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();

    // this thread's image and item range
    int my = -1, item_begin = 0, item_end = 0;
    for (int ci = 0; ci < nimg; ++ci)
        if ((int)threadIdx.x >= tstart[ci] && (int)threadIdx.x < tend[ci]) my = ci;
    const bool deep_warp = split && (int)threadIdx.x >= (int)blockDim.x - 32;
    const int lvl = my <= 0 ? 0 : (my - 1) / 2 + 1;
    const int pp = my <= 0 ? 0 : (my - 1) & 1;
    if (my >= 0) {
        const int items = G * geo.rseg[lvl] * geo.cstr[lvl];
        const int pt = my >= 5 ? per_thread_deep : per_thread;
        item_begin = (threadIdx.x - tstart[my]) * pt;
        item_end = min(items, item_begin + pt);
    }
    const int pitch = geo.pitch[lvl];
    const int y_off = lvl == 0 ? geo.off_x : geo.off_y[lvl] + pp * geo.pimg[lvl];
    const int g_off = lvl == 0 ? geo.off_dy : geo.off_g[lvl] + pp * geo.pimg[lvl];
    const int ncols = geo.cstr[lvl], per_plane = geo.rseg[lvl] * ncols;

    f2_t acc[KK];
#pragma unroll
    for (int i = 0; i < KK; ++i) acc[i] = 0ull;
    float dysum = 0.f;

    const T *x = static_cast<const T *>(a.x);
    const T *dy = static_cast<const T *>(a.dy);
    const size_t HW = (size_t)a.H * a.W;
    T *stg_x = a.stage ? reinterpret_cast<T *>(reinterpret_cast<char *>(smem) + a.stage_off) : nullptr;
    T *stg_dy = a.stage ? stg_x + (size_t)G * HW : nullptr;
    const int first = nbi * a.groups_per_cta * G;
    int ngrp = 0;
    while (ngrp < a.groups_per_cta && first + ngrp * G < a.B) ++ngrp;

    for (int grp = 0; grp < ngrp; ++grp) {
        const int b0 = first + grp * G;
        if (stg_x) {
            if (grp == 0) {
                stage_planes<T>(x, stg_x, a.B, a.C, c, b0, G, HW, a.dv.stage_chunks);
                stage_planes<T>(dy, stg_dy, a.B, a.C, c, b0, G, HW, a.dv.stage_chunks);
                cp_async_commit();
            }
            cp_async_wait_all();
            __syncthreads();
        }
        // A. both planes -> padded fp32 copies + both Haar pyramids; then the next group streams in
        analysis_from_global<T, P>(a, geo, x, stg_x, c, b0, slots, geo.off_x, geo.off_y);
        dysum += analysis_from_global<T, P>(a, geo, dy, stg_dy, c, b0, slots, geo.off_dy, geo.off_g);
        __syncthreads();
        if (stg_x && grp + 1 < ngrp) {
            stage_planes<T>(x, stg_x, a.B, a.C, c, b0 + G, G, HW, a.dv.stage_chunks);
            stage_planes<T>(dy, stg_dy, a.B, a.C, c, b0 + G, G, HW, a.dv.stage_chunks);
            cp_async_commit();
        }
        if (split) {
            if (deep_warp) {
                for (int l = 3; l <= geo.L; l += 2) {
                    analysis_from_shared<P>(a, geo, slots, G, geo.off_y, l, blockDim.x - 32, 32);
                    analysis_from_shared<P>(a, geo, slots, G, geo.off_g, l, blockDim.x - 32, 32);
                    __syncwarp();
                }
            }
        } else {
            for (int l = 3; l <= geo.L; l += 2) {
                analysis_from_shared<P>(a, geo, slots, G, geo.off_y, l);
                analysis_from_shared<P>(a, geo, slots, G, geo.off_g, l);
                __syncthreads();
            }
        }
        if (!stg_x && grp + 1 < ngrp && ((HW * sizeof(T)) & 15) == 0 && (int)threadIdx.x < 2 * G) {
            const int bn = b0 + G + (threadIdx.x >> 1);
            if (bn < a.B) prefetch_l2(((threadIdx.x & 1) ? dy : x) + ((size_t)bn * a.C + c) * HW, (uint32_t)(HW * sizeof(T)));
        }
        // C. this thread's share of its correlation
        for (int it = item_begin; it < item_end; ++it) {
            const int g = fdiv(a.dv.item_plane[lvl], it), e = it - g * per_plane;
            const int rs = fdiv(a.dv.item_cols[lvl], e), cs = e - rs * ncols;
            const float *slot = slots + (size_t)g * geo.slot_floats;
            if (lvl == 0) {
                dw_item<K>(slot + y_off + (rs * kRows) * pitch + cs * kCols,
                           slot + g_off + (rs * kRows + P) * pitch + cs * kCols + P, pitch, acc);
            } else {
                dw_item_pair<K>(slot + y_off + 2 * ((rs * kRows) * pitch + cs * kColsL),
                                slot + g_off + 2 * ((rs * kRows + P) * pitch + cs * kColsL + P), pitch, acc);
            }
        }
        __syncthreads();
    }

    // reduce: per-thread tap sums -> one partial per (subband, tap), in thread order
    cp_async_wait_all();
    __syncthreads();
    float *red = smem;
#pragma unroll
    for (int i = 0; i < KK; ++i) {
        const float lo = lo2(acc[i]), hi = hi2(acc[i]);
        red[threadIdx.x * NR + i] = lvl == 0 ? lo + hi : lo;
        red[threadIdx.x * NR + KK + i] = lvl == 0 ? 0.f : hi;
    }
    red[threadIdx.x * NR + 2 * KK] = dysum;
    __syncthreads();
    float *part = a.partials + ((size_t)nbi * a.C + c) * nsig * NA;
    for (int i = threadIdx.x; i < nsig * NA; i += blockDim.x) {
        const int sig = i / NA, t = i - sig * NA;
        float s = 0.f;
        if (t < KK) {
            int ci = 0, half = 0;
            if (sig > 0) {
                const int l = (sig - 1) / 4 + 1, sb = (sig - 1) & 3;
                ci = 1 + 2 * (l - 1) + (sb >> 1);
                half = sb & 1;
            }
            for (int th = tstart[ci]; th < tend[ci]; ++th) s += red[th * NR + half * KK + t];
        } else if (sig == 0) {
            for (int th = 0; th < (int)blockDim.x; ++th) s += red[th * NR + 2 * KK];
        }
        part[i] = s;
    }
}

// Sum the per-CTA partials of each (channel, subband) in order of CTA index and unfold the
// scales.  One 64-thread block per (channel, subband); thread t owns tap t (thread K*K: the
// gradient sum of the base bias).
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
static cudaError_t launch_dw_t(const LayerArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_dw_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), a.threads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_dw_t(int threads, size_t smem) {
    auto kern = wtconv_dw_kernel<K, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) return 0;
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

cudaError_t launch_dw(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_dw_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_dw(int dtype, int K, int threads, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_dw_t, threads, smem);
    return 0;
}

cudaError_t launch_dw_finalize(const LayerArgs &a, float *d_base_w, float *d_base_bias, float *d_base_scale,
                               float *d_wavelet_w, float *d_wavelet_scale, cudaStream_t st) {
    const int n = a.C * n_sig(a.L);
    wtconv_dw_finalize_kernel<<<n, 64, 0, st>>>(a, d_base_w, d_base_bias, d_base_scale, d_wavelet_w,
                                                d_wavelet_scale);
    return cudaGetLastError();
}

}  // namespace wtconv
