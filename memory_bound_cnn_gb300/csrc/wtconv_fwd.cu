// Forward kernel of the WTConv layer (also serves the input gradient: the same operator on dy
// with every kernel rotated by 180 degrees and no bias).
//
// Each CTA owns channel c and a run of batch entries and walks through them in groups of G
// planes.  Per group:
//   A. one read of each plane from HBM builds the padded fp32 plane and the Haar pyramid in
//      shared memory (two levels per pass); the next group is prefetched into L2 meanwhile;
//   C. every k x k conv of the layer -- the base conv of the plane and the conv of every subband
//      of every level, with the folded kernels -- runs as sliding-window items (8 x 4 outputs,
//      packed f32x2 FMAs) spread over all threads; results stay in shared memory;
//   D. each output pixel is written once: base conv + bias + closed-form synthesis gather.
#include "wtconv_analysis.cuh"

namespace wtconv {

size_t fwd_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off) {
    size_t bytes = (size_t)G * geo.slot_floats * sizeof(float) + (size_t)(1 + 2 * L) * wpairs(K) * sizeof(f2_t);
    bytes = (bytes + 15) / 16 * 16;
    if (stage_off) *stage_off = (int)bytes;
    if (stage) bytes += (size_t)G * geo.H * geo.W * elem_bytes;
    return (bytes + 15) / 16 * 16;
}

// Closed-form synthesis of the 8 output pixels (h, w0 .. w0+7), w0 % 8 == 0, added to out[]:
//   out[c] += sum_l sum_s sigma_s(bit_{l-1}(h), bit_{l-1}(w0+c)) * Z^l_s[h >> l][(w0+c) >> l]
// (Z carries the 2^-l synthesis factor through the folded kernels).  With Z^l stored as the pair
// images (Z_LL, Z_LH) and (Z_HL, Z_HH), one packed op gives (p, r) = (Z_LL +- Z_HL, Z_LH +- Z_HH)
// (sign by the row bit); the pixel with column bit b then gets p + r (b = 0) or p - r (b = 1).
__device__ __forceinline__ void synth_gather8(const Geo &geo, const float *slot, int h, int w0, float (&out)[8]) {
    {   // level 1: four positions; row bit a = bit 0 of h, column bit b = c & 1
        const float *z = slot + geo.off_z[1] + 2 * ((h >> 1) * geo.zpitch[1] + (w0 >> 1));
        const float4 a01 = *reinterpret_cast<const float4 *>(z), b01 = *reinterpret_cast<const float4 *>(z + 4);
        const float *z2 = z + geo.zimg[1];
        const float4 a23 = *reinterpret_cast<const float4 *>(z2), b23 = *reinterpret_cast<const float4 *>(z2 + 4);
        const float ll[4] = {a01.x, a01.z, b01.x, b01.z}, lh[4] = {a01.y, a01.w, b01.y, b01.w};
        const float hl[4] = {a23.x, a23.z, b23.x, b23.z}, hh[4] = {a23.y, a23.w, b23.y, b23.w};
        const bool ra = h & 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float p = ra ? ll[q] - hl[q] : ll[q] + hl[q];
            const float r = ra ? lh[q] - hh[q] : lh[q] + hh[q];
            out[2 * q] += p + r;
            out[2 * q + 1] += p - r;
        }
    }
    if (geo.L >= 2) {  // level 2: two positions, column bit b = bit 1 of c
        const float *z = slot + geo.off_z[2] + 2 * ((h >> 2) * geo.zpitch[2] + (w0 >> 2));
        const float4 a01 = *reinterpret_cast<const float4 *>(z);
        const float4 a23 = *reinterpret_cast<const float4 *>(z + geo.zimg[2]);
        const bool ra = (h >> 1) & 1;
        const float p0 = ra ? a01.x - a23.x : a01.x + a23.x, r0 = ra ? a01.y - a23.y : a01.y + a23.y;
        const float p1 = ra ? a01.z - a23.z : a01.z + a23.z, r1 = ra ? a01.w - a23.w : a01.w + a23.w;
        const float s0 = p0 + r0, d0 = p0 - r0, s1 = p1 + r1, d1 = p1 - r1;
        out[0] += s0; out[1] += s0; out[2] += d0; out[3] += d0;
        out[4] += s1; out[5] += s1; out[6] += d1; out[7] += d1;
    }
    float lo = 0.f, hi = 0.f;  // levels >= 3: one position, constant over each half (level 3) or all 8
    for (int l = 3; l <= geo.L; ++l) {
        const float *z = slot + geo.off_z[l] + 2 * ((h >> l) * geo.zpitch[l] + (w0 >> l));
        const float2 a01 = *reinterpret_cast<const float2 *>(z);
        const float2 a23 = *reinterpret_cast<const float2 *>(z + geo.zimg[l]);
        const bool ra = (h >> (l - 1)) & 1;
        const float p = ra ? a01.x - a23.x : a01.x + a23.x, r = ra ? a01.y - a23.y : a01.y + a23.y;
        if (l == 3) {
            lo += p + r;
            hi += p - r;
        } else {
            const float v = ((w0 >> (l - 1)) & 1) ? p - r : p + r;
            lo += v;
            hi += v;
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        out[c] += lo;
        out[c + 4] += hi;
    }
}

// Conv images of a slot: ci = 0 the base conv (X -> base buffer, column-pair items of kRows x
// kCols pixels), ci = 1 + 2(l-1) + pp the level-l subband pair pp (Y^l pair image -> Z^l pair
// image, items of kRows x kColsL positions).
template <int K, typename T>
__global__ void __launch_bounds__(kMaxThreads, (K <= 5 ? 2 : 1)) wtconv_fwd_kernel(const LayerArgs a) {
    constexpr int P = K / 2, WP = wpairs(K);
    constexpr int kMaxImg = 1 + 2 * kMaxLevels;
    extern __shared__ __align__(16) float smem[];
    __shared__ Geo geo;
    __shared__ int cstart[kMaxImg + 1], in_off[kMaxImg], out_off[kMaxImg], img_lvl[kMaxImg];
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = a.G, nimg = 1 + 2 * a.L;
    float *slots = smem;
    f2_t *wts = reinterpret_cast<f2_t *>(smem + (size_t)G * a.geo.slot_floats);

    if (threadIdx.x == 0) {
        geo = a.geo;
        int tot = 0;
        for (int ci = 0; ci < nimg; ++ci) {
            const int l = ci == 0 ? 0 : (ci - 1) / 2 + 1, pp = ci == 0 ? 0 : (ci - 1) & 1;
            cstart[ci] = tot;
            img_lvl[ci] = l;
            in_off[ci] = ci == 0 ? a.geo.off_x : a.geo.off_y[l] + pp * a.geo.pimg[l];
            out_off[ci] = ci == 0 ? a.geo.off_base : a.geo.off_z[l] + pp * a.geo.zimg[l];
            tot += G * a.geo.rseg[l] * a.geo.cstr[l];
        }
        cstart[nimg] = tot;
    }
    {
        float4 *s4 = reinterpret_cast<float4 *>(slots);
        const int n4 = G * a.geo.slot_floats / 4;
        for (int i = threadIdx.x; i < n4; i += blockDim.x) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    stage_weights<K>(a, c, wts);
    const float bias = a.with_bias ? a.base_scale[c] * a.base_bias[c] : 0.f;
    const f2_t bias2 = pk2(bias, bias);
    __syncthreads();

    const T *x = static_cast<const T *>(a.x);
    T *y = static_cast<T *>(a.out);
    const size_t HW = (size_t)a.H * a.W;
    T *stg = a.stage ? reinterpret_cast<T *>(reinterpret_cast<char *>(smem) + a.stage_off) : nullptr;
    const int nitems = cstart[nimg];
    const int nws = (int)a.dv.out_w.d, nd = (int)a.dv.out_n.d;
    const int slot_floats = geo.slot_floats;
    const int first = nbi * a.groups_per_cta * G;
    int ngrp = 0;  // groups this CTA owns
    while (ngrp < a.groups_per_cta && first + ngrp * G < a.B) ++ngrp;

    // whole planes of 16-byte multiples can be bulk-prefetched into L2 when they are not staged
    const bool l2_prefetch = !stg && ((HW * sizeof(T)) & 15) == 0;
    // prologue: pyramid of the first group, staging of the second
    if (stg) {
        stage_planes<T>(x, stg, a.B, a.C, c, first, G, HW, a.dv.stage_chunks);
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
    }
    if (ngrp > 0) analysis_from_global<T, P>(a, geo, x, stg, c, first, slots, geo.off_x, geo.off_y);
    __syncthreads();
    if (stg && ngrp > 1) {
        stage_planes<T>(x, stg, a.B, a.C, c, first + G, G, HW, a.dv.stage_chunks);
        cp_async_commit();
    }
    for (int l = 3; l <= geo.L && ngrp > 0; l += 2) {
        analysis_from_shared<P>(a, geo, slots, G, geo.off_y, l);
        __syncthreads();
    }

    for (int grp = 0; grp < ngrp; ++grp) {
        const int b0 = first + grp * G;
        const bool has_next = grp + 1 < ngrp;

        if (l2_prefetch && has_next && (int)threadIdx.x < G && b0 + G + (int)threadIdx.x < a.B)
            prefetch_l2(x + ((size_t)(b0 + G + threadIdx.x) * a.C + c) * HW, (uint32_t)(HW * sizeof(T)));
        // C. every conv of the layer, as sliding-window items
        for (int it = threadIdx.x; it < nitems; it += blockDim.x) {
            int ci = 0;
            while (it >= cstart[ci + 1]) ++ci;
            const int l = img_lvl[ci];
            const int local = it - cstart[ci];
            const int g = fdiv(a.dv.item_plane[l], local), e = local - g * (int)a.dv.item_plane[l].d;
            const int rs = fdiv(a.dv.item_cols[l], e), cs = e - rs * (int)a.dv.item_cols[l].d;
            float *slot = slots + g * slot_floats;
            f2_t w[K * K];
            load_weights<K>(wts + ci * WP, w);
            const int pitch = geo.pitch[l], opitch = geo.zpitch[l];
            if (ci == 0) {
                conv_item<K>(slot + in_off[0] + (rs * kRows) * pitch + cs * kCols, pitch, w,
                             slot + out_off[0] + (rs * kRows) * opitch + cs * kCols, opitch, bias2);
            } else {
                conv_item_pair<K>(slot + in_off[ci] + 2 * ((rs * kRows) * pitch + cs * kColsL), pitch, w,
                                  slot + out_off[ci] + 2 * ((rs * kRows) * opitch + cs * kColsL), opitch);
            }
        }
        if (stg && has_next) cp_async_wait_all();
        __syncthreads();

        // D. outputs of this group (base conv + bias + closed-form synthesis), and A. the next
        // group's planes -> padded copy + first Haar levels (disjoint shared buffers)
        for (int it = threadIdx.x; it < G * nd; it += blockDim.x) {
            const int g = fdiv(a.dv.out_n, it), e = it - g * nd;
            const int h = fdiv(a.dv.out_w, e), ws = e - h * nws;
            const int b = b0 + g;
            if (b >= a.B) continue;
            const int w0 = ws * 8;
            const float *slot = slots + g * slot_floats;
            const float *bb = slot + geo.off_base + h * geo.zpitch[0] + w0;
            const float4 b0v = *reinterpret_cast<const float4 *>(bb);
            const float4 b1v = *reinterpret_cast<const float4 *>(bb + 4);
            float out[8] = {b0v.x, b0v.y, b0v.z, b0v.w, b1v.x, b1v.y, b1v.z, b1v.w};
            synth_gather8(geo, slot, h, w0, out);
            T *dst = y + ((size_t)b * a.C + c) * HW + (size_t)h * geo.W + w0;
            const int nv = min(8, geo.W - w0);
            if (a.st_mode == 2 && nv == 8) {
                Act<T>::st8(dst, out);
            } else if (a.st_mode >= 1) {
                Act<T>::st4(dst, out);
                if (nv == 8) Act<T>::st4(dst + 4, out + 4);
            } else {
                for (int i = 0; i < nv; ++i) Act<T>::st(dst + i, out[i]);
            }
        }
        if (has_next) analysis_from_global<T, P>(a, geo, x, stg, c, b0 + G, slots, geo.off_x, geo.off_y);
        __syncthreads();
        if (has_next) {
            if (stg && grp + 2 < ngrp) {
                stage_planes<T>(x, stg, a.B, a.C, c, b0 + 2 * G, G, HW, a.dv.stage_chunks);
                cp_async_commit();
            }
            for (int l = 3; l <= geo.L; l += 2) {
                analysis_from_shared<P>(a, geo, slots, G, geo.off_y, l);
                __syncthreads();
            }
        }
    }
}

template <int K, typename T>
static cudaError_t launch_fwd_t(const LayerArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_fwd_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), a.threads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_fwd_t(int threads, size_t smem) {
    auto kern = wtconv_fwd_kernel<K, T>;
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

cudaError_t launch_forward(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_fwd_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_forward(int dtype, int K, int threads, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_fwd_t, threads, smem);
    return 0;
}

}  // namespace wtconv
