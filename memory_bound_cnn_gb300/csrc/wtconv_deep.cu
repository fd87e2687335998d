// Deep kernel of the WTConv layer: Haar levels >= 2 of every plane and their closed-form
// synthesis down to level-1 resolution (forward on x, or the input gradient on dy with rotated
// kernels).  The shallow kernel adds this "deep contribution" to each output pixel.
//
// For output pixel (h, w) the closed form sums sum_l sum_s sigma_s(bit_{l-1} h, bit_{l-1} w) *
// Z^l_s[h >> l, w >> l]; for l >= 2 the row and column bits used are bits >= 1, so the deep part is
// constant over 2 x 2 pixel blocks and is computed once per level-1 position (i, j) = (h>>1, w>>1):
//     D[i][j] = sum_{l>=2} sum_s sigma_s(bit_{l-2} i, bit_{l-2} j) * Z^l_s[i >> (l-1), j >> (l-1)].
// Each CTA owns channel c and a run of batch entries in groups of G planes.  Per group: one read
// of each plane builds level 2 (from 4 x 4 pixel blocks) and the deeper levels on chip; every
// level's subband-pair convs run as sliding-window items; D is written once.
#include "wtconv_items.cuh"

namespace wtconv {

size_t deep_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off) {
    size_t bytes = (size_t)G * geo.slot_floats * sizeof(float) + (size_t)(1 + 2 * L) * wpairs(K) * sizeof(f2_t);
    bytes = (bytes + 15) / 16 * 16;
    if (stage_off) *stage_off = (int)bytes;
    if (stage) bytes += (size_t)G * geo.H * geo.W * elem_bytes;
    return (bytes + 15) / 16 * 16;
}

// Level 2 of G planes straight from the input (4 x 4 pixel blocks; level 1 is not kept).
template <typename T>
__device__ __forceinline__ void deep_analysis_from_global(const LayerArgs &a, const Geo &geo, const T *x,
                                                          const T *stg, int c, int b0, float *slots) {
    const int G = a.G, W = geo.W;
    const size_t HW = (size_t)geo.H * W;
    const FastDiv &dn = a.dv.a_n[1], &dw = a.dv.a_w[1];
    const int bw = (int)dw.d, n = (int)dn.d;
    for (int it = threadIdx.x; it < G * n; it += blockDim.x) {
        const int g = fdiv(dn, it), e = it - g * n;
        const int bi = fdiv(dw, e), bj = e - bi * bw;
        const int b = b0 + g;
        float v[4][4];
        if (b < a.B) {
            const T *plane = stg ? stg + (size_t)g * HW : x + ((size_t)b * a.C + c) * HW;
            const T *src = plane + (size_t)(4 * bi) * W + 4 * bj;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (a.vec_ld) {
                    const float4 t = Act<T>::ld4(src + r * W);
                    v[r][0] = t.x; v[r][1] = t.y; v[r][2] = t.z; v[r][3] = t.w;
                } else {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) v[r][cc] = Act<T>::ld(src + r * W + cc);
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) v[r][cc] = 0.f;
        }
        // level-1 low band of the four 2x2 blocks (unnormalised), then the level-2 butterfly
        float ll[2][2];
#pragma unroll
        for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2)
                ll[a2][b2] = (v[2 * a2][2 * b2] + v[2 * a2][2 * b2 + 1]) + (v[2 * a2 + 1][2 * b2] + v[2 * a2 + 1][2 * b2 + 1]);
        float *slot = slots + (size_t)g * geo.slot_floats;
        put_quad_pairs(slot, geo, geo.off_y, 2, bi, bj, butterfly(ll[0][0], ll[0][1], ll[1][0], ll[1][1]));
    }
}

template <int K, typename T>
__global__ void __launch_bounds__(kMaxThreads, (K <= 5 ? 2 : 1)) wtconv_deep_kernel(const LayerArgs a, float *dout) {
    constexpr int P = K / 2, WP = wpairs(K);
    constexpr int kMaxImg = 1 + 2 * kMaxLevels;
    extern __shared__ __align__(16) float smem[];
    __shared__ Geo geo;
    __shared__ int cstart[kMaxImg + 1], in_off[kMaxImg], out_off[kMaxImg], img_lvl[kMaxImg];
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = a.G;
    const int ci0 = 3, ci1 = 1 + 2 * a.L;  // conv images of levels 2 .. L
    float *slots = smem;
    f2_t *wts = reinterpret_cast<f2_t *>(smem + (size_t)G * a.geo.slot_floats);

    if (threadIdx.x == 0) {
        geo = a.geo;
        int tot = 0;
        for (int ci = ci0; ci < ci1; ++ci) {
            const int l = (ci - 1) / 2 + 1, pp = (ci - 1) & 1;
            cstart[ci] = tot;
            img_lvl[ci] = l;
            in_off[ci] = a.geo.off_y[l] + pp * a.geo.pimg[l];
            out_off[ci] = a.geo.off_z[l] + pp * a.geo.zimg[l];
            tot += G * a.geo.rseg[l] * a.geo.cstr[l];
        }
        cstart[ci1] = tot;
    }
    const T *x = static_cast<const T *>(a.x);
    const size_t HW = (size_t)a.H * a.W;
    // the first group's planes start towards L2 now, while the slots are cleared and the kernels
    // staged (the later groups' planes are prefetched one group ahead in the loop below)
    if (!a.stage && ((HW * sizeof(T)) & 15) == 0 && (int)threadIdx.x < G) {
        const int b = nbi * a.groups_per_cta * G + (int)threadIdx.x;
        if (b < a.B) prefetch_l2(x + ((size_t)b * a.C + c) * HW, (uint32_t)(HW * sizeof(T)));
    }
    {
        float4 *s4 = reinterpret_cast<float4 *>(slots);
        const int n4 = G * a.geo.slot_floats / 4;
        for (int i = threadIdx.x; i < n4; i += blockDim.x) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    stage_weights<K>(a, c, wts);
    __syncthreads();

    const int H1 = a.H >> 1, W1 = a.W >> 1;
    T *stg = a.stage ? reinterpret_cast<T *>(reinterpret_cast<char *>(smem) + a.stage_off) : nullptr;
    const int nitems = cstart[ci1];
    const int nws = (int)a.dv.out_w.d, nd = (int)a.dv.out_n.d;  // D row segments of 8 and per plane
    const int slot_floats = geo.slot_floats;
    const int first = nbi * a.groups_per_cta * G;
    int ngrp = 0;
    while (ngrp < a.groups_per_cta && first + ngrp * G < a.B) ++ngrp;
    const bool l2_prefetch = !stg && ((HW * sizeof(T)) & 15) == 0;

    if (stg && ngrp > 0) {
        stage_planes<T>(x, stg, a.B, a.C, c, first, G, HW, a.dv.stage_chunks);
        cp_async_commit();
    }
    for (int grp = 0; grp < ngrp; ++grp) {
        const int b0 = first + grp * G;
        const bool has_next = grp + 1 < ngrp;
        if (stg) {
            cp_async_wait_all();
            __syncthreads();
        } else if (l2_prefetch && has_next && (int)threadIdx.x < G && b0 + G + (int)threadIdx.x < a.B) {
            prefetch_l2(x + ((size_t)(b0 + G + threadIdx.x) * a.C + c) * HW, (uint32_t)(HW * sizeof(T)));
        }
        deep_analysis_from_global<T>(a, geo, x, stg, c, b0, slots);
        __syncthreads();
        if (stg && has_next) {
            stage_planes<T>(x, stg, a.B, a.C, c, b0 + G, G, HW, a.dv.stage_chunks);
            cp_async_commit();
        }
        for (int l = 3; l <= geo.L; l += 2) {
            analysis_from_shared<P>(a, geo, slots, G, geo.off_y, l);
            __syncthreads();
        }
        for (int it = threadIdx.x; it < nitems; it += blockDim.x) {
            int ci = ci0;
            while (it >= cstart[ci + 1]) ++ci;
            const int l = img_lvl[ci];
            const int local = it - cstart[ci];
            const int g = fdiv(a.dv.item_plane[l], local), e = local - g * (int)a.dv.item_plane[l].d;
            const int rs = fdiv(a.dv.item_cols[l], e), cs = e - rs * (int)a.dv.item_cols[l].d;
            float *slot = slots + g * slot_floats;
            f2_t w[K * K];
            load_weights<K>(wts + ci * WP, w);
            const int pitch = geo.pitch[l], opitch = geo.zpitch[l];
            conv_item_pair<K>(slot + in_off[ci] + 2 * ((rs * kRows) * pitch + cs * kColsL), pitch, w,
                              slot + out_off[ci] + 2 * ((rs * kRows) * opitch + cs * kColsL), opitch);
        }
        __syncthreads();
        for (int it = threadIdx.x; it < G * nd; it += blockDim.x) {
            const int g = fdiv(a.dv.out_n, it), e = it - g * nd;
            const int i = fdiv(a.dv.out_w, e), ws = e - i * nws;
            const int b = b0 + g;
            if (b >= a.B) continue;
            const int j0 = ws * 8;
            float d[8];
            deep_gather8(geo, slots + g * slot_floats, i, j0, d);
            float *dst = dout + ((size_t)b * a.C + c) * H1 * W1 + (size_t)i * W1 + j0;
            const int nv = min(8, W1 - j0);
            if (nv == 8 && (W1 & 3) == 0) {
                reinterpret_cast<float4 *>(dst)[0] = make_float4(d[0], d[1], d[2], d[3]);
                reinterpret_cast<float4 *>(dst)[1] = make_float4(d[4], d[5], d[6], d[7]);
            } else {
                for (int q = 0; q < nv; ++q) dst[q] = d[q];
            }
        }
        __syncthreads();
    }
}

template <int K, typename T>
static cudaError_t launch_deep_t(const LayerArgs &a, float *dout, size_t smem, cudaStream_t st) {
    auto kern = wtconv_deep_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), a.threads, smem, st>>>(a, dout);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_deep_t(int threads, size_t smem) {
    auto kern = wtconv_deep_kernel<K, T>;
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

cudaError_t launch_deep(const LayerArgs &a, float *dout, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_deep_t, a, dout, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_deep(int dtype, int K, int threads, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_deep_t, threads, smem);
    return 0;
}

}  // namespace wtconv
