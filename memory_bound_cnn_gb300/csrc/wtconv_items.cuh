// Output items shared by the forward kernels of the WTConv layer: the fused 8 x 4 pixel item
// (level-1 subband-pair convs, their closed-form synthesis and the base conv on top), and the
// gather of the deep levels' contribution at level-1 resolution.
#pragma once

#include "wtconv_analysis.cuh"

namespace wtconv {

// cp.async of `N` bytes (4, 8 or 16); src_bytes = 0 zero-fills the destination without reading.
template <int N>
__device__ __forceinline__ void cp_async_n(void *smem_dst, const void *gmem_src, int src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    if constexpr (N == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gmem_src), "r"(src_bytes) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(d), "l"(gmem_src), "n"(N), "r"(src_bytes)
                     : "memory");
}

// Level-1 conv of one subband-pair image for 4 coefficient rows x 2 positions, kept in registers.
template <int K>
__device__ __forceinline__ void level1_item(const float *__restrict__ in, int pitch, const f2_t *wsm,
                                            f2_t (&z)[4][kColsL]) {
    constexpr int NV = (kColsL + K - 1 + 1) / 2;
    f2_t w[K * K];
    load_weights<K>(wsm, w);
#pragma unroll
    for (int i = 0; i < 4 + K - 1; ++i) {
        f2_t x[2 * NV];
        load_pair_row<NV>(in + 2 * i * pitch, x);
#pragma unroll
        for (int v = 0; v < K; ++v) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < 4) {
#pragma unroll
                    for (int q = 0; q < kColsL; ++q) {
                        if (u == 0 && v == 0) z[j][q] = fmul2(w[0], x[q]);
                        else ffma2_acc(z[j][q], w[u * K + v], x[q + v]);
                    }
                }
            }
        }
    }
}

// Base conv of one 8 x 4 pixel block on top of `init`, each finished row rounded and stored:
// out[r][c] = init[r][c] + sum_{u,v} w[u][v] * X[r + u][c + v - P].  `in` points at the 16-byte
// aligned X position 4 - P columns left of the window origin (window row r, column 0); three
// 16-byte loads per window row cover columns 0 .. 11 of that, the window is columns
// 4 - P .. 4 - P + 3 + K - 1.
template <int K, typename T>
__device__ __forceinline__ void base_item_store(const float *__restrict__ in, int pitch, const f2_t *wsm,
                                                const f2_t (&init)[kRows][2], T *dst, int ld, int nrows,
                                                int ncols, bool vec) {
    constexpr int P = K / 2, O = 4 - P;
    f2_t w[K * K];
    load_weights<K>(wsm, w);
    f2_t acc[kRows][2];
#pragma unroll
    for (int i = 0; i < kRows + K - 1; ++i) {
        f2_t e[6], o[5];
        load_row<3>(in + i * pitch, e, o);
#pragma unroll
        for (int v = 0; v < K; ++v) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < kRows) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int s0 = O + v + 2 * q;  // first column of the pair
                        const f2_t xv = (s0 & 1) ? o[(s0 - 1) / 2] : e[s0 / 2];
                        if (u == 0 && v == 0) acc[j][q] = ffma2(w[0], xv, init[j][q]);
                        else ffma2_acc(acc[j][q], w[u * K + v], xv);
                    }
                }
            }
        }
        const int jd = i - (K - 1);
        if (jd >= 0 && jd < nrows) {
            const float vals[4] = {lo2(acc[jd][0]), hi2(acc[jd][0]), lo2(acc[jd][1]), hi2(acc[jd][1])};
            T *d = dst + (size_t)jd * ld;
            if (vec && ncols == 4) {
                Act<T>::st4(d, vals);
            } else {
                for (int c = 0; c < ncols; ++c) Act<T>::st(d + c, vals[c]);
            }
        }
    }
}

// Four narrow activations (8 bytes) to fp32.
template <typename T>
__device__ __forceinline__ float4 cvt4(const T *p) {
    return Act<T>::ld4(p);
}

// D[i][j0 .. j0+7] (level-1 positions, j0 % 8 == 0) from the deep levels' conv outputs.
__device__ __forceinline__ void deep_gather8(const Geo &geo, const float *slot, int i, int j0, float (&out)[8]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) out[c] = 0.f;
    {   // level 2 (relative level 1): four positions; row bit = bit 0 of i, column bit = c & 1
        const float *z = slot + geo.off_z[2] + 2 * ((i >> 1) * geo.zpitch[2] + (j0 >> 1));
        const float4 a01 = *reinterpret_cast<const float4 *>(z), b01 = *reinterpret_cast<const float4 *>(z + 4);
        const float *z2 = z + geo.zimg[2];
        const float4 a23 = *reinterpret_cast<const float4 *>(z2), b23 = *reinterpret_cast<const float4 *>(z2 + 4);
        const float ll[4] = {a01.x, a01.z, b01.x, b01.z}, lh[4] = {a01.y, a01.w, b01.y, b01.w};
        const float hl[4] = {a23.x, a23.z, b23.x, b23.z}, hh[4] = {a23.y, a23.w, b23.y, b23.w};
        const bool ra = i & 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float p = ra ? ll[q] - hl[q] : ll[q] + hl[q];
            const float r = ra ? lh[q] - hh[q] : lh[q] + hh[q];
            out[2 * q] += p + r;
            out[2 * q + 1] += p - r;
        }
    }
    if (geo.L >= 3) {  // level 3: two positions, column bit = bit 1 of c
        const float *z = slot + geo.off_z[3] + 2 * ((i >> 2) * geo.zpitch[3] + (j0 >> 2));
        const float4 a01 = *reinterpret_cast<const float4 *>(z);
        const float4 a23 = *reinterpret_cast<const float4 *>(z + geo.zimg[3]);
        const bool ra = (i >> 1) & 1;
        const float p0 = ra ? a01.x - a23.x : a01.x + a23.x, r0 = ra ? a01.y - a23.y : a01.y + a23.y;
        const float p1 = ra ? a01.z - a23.z : a01.z + a23.z, r1 = ra ? a01.w - a23.w : a01.w + a23.w;
        const float s0 = p0 + r0, d0 = p0 - r0, s1 = p1 + r1, d1 = p1 - r1;
        out[0] += s0; out[1] += s0; out[2] += d0; out[3] += d0;
        out[4] += s1; out[5] += s1; out[6] += d1; out[7] += d1;
    }
    float lo = 0.f, hi = 0.f;  // levels >= 4: one position, constant over each half (level 4) or all 8
    for (int l = 4; l <= geo.L; ++l) {
        const int t = l - 1;  // level relative to the level-1 grid
        const float *z = slot + geo.off_z[l] + 2 * ((i >> t) * geo.zpitch[l] + (j0 >> t));
        const float2 a01 = *reinterpret_cast<const float2 *>(z);
        const float2 a23 = *reinterpret_cast<const float2 *>(z + geo.zimg[l]);
        const bool ra = (i >> (t - 1)) & 1;
        const float p = ra ? a01.x - a23.x : a01.x + a23.x, r = ra ? a01.y - a23.y : a01.y + a23.y;
        if (t == 3) {
            lo += p + r;
            hi += p - r;
        } else {
            const float v = ((j0 >> (t - 1)) & 1) ? p - r : p + r;
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

}  // namespace wtconv
