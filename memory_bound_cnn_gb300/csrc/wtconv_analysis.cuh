// On-chip Haar analysis passes: one read of each input plane (from the shared staging area or
// from global memory) builds the padded fp32 copy of the plane and the first Haar levels; later
// passes build deeper levels from the low band in shared memory.  Each pass computes two levels
// per item where it can (a 4x4 block of the finer low band gives four level-l positions and one
// level-(l+1) position), so an L-level pyramid needs ceil(L/2) passes (and barriers).
// Levels are written as subband-pair images: pair 0 = (LL, LH), pair 1 = (HL, HH).
#pragma once

#include "wtconv_device.cuh"

namespace wtconv {

// Write the quad of level l at interior position (i, j) of the slot's pair images.
__device__ __forceinline__ void put_quad_pairs(float *slot, const Geo &geo, const int *off, int l, int i, int j,
                                               const Quad &q) {
    const int P = geo.P;
    float *p0 = slot + off[l] + 2 * ((i + P) * geo.pitch[l] + j + P);
    *reinterpret_cast<float2 *>(p0) = make_float2(q.ll, q.lh);
    *reinterpret_cast<float2 *>(p0 + geo.pimg[l]) = make_float2(q.hl, q.hh);
}

// LL value of level l at interior position (i, j).
__device__ __forceinline__ float get_ll(const float *slot, const Geo &geo, const int *off, int l, int i, int j) {
    const int P = geo.P;
    return slot[off[l] + 2 * ((i + P) * geo.pitch[l] + j + P)];
}

// Pass 1: read G planes of x (type T; from the shared staging area when `stg` is not null, else
// from global memory), write the padded fp32 copy X and Haar level 1 (and level 2 when L >= 2).
// Returns the sum of the values read (used for the bias gradient).
template <typename T, int P>
__device__ __forceinline__ float analysis_from_global(const LayerArgs &a, const Geo &geo, const T *x, const T *stg,
                                                      int c, int b0, float *slots, int x_off, const int *pyr_off) {
    const int G = a.G, W = geo.W;
    const size_t HW = (size_t)geo.H * W;
    float sum = 0.f;
    const FastDiv &dn = a.dv.a_n[1], &dw = a.dv.a_w[1];
    const int bw = (int)dw.d, n = (int)dn.d;
    const int xp = geo.pitch[0];
    if (geo.L >= 2) {
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
            float *slot = slots + (size_t)g * geo.slot_floats;
            float *X = slot + x_off + (4 * bi + P) * xp + 4 * bj + P;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if constexpr ((P & 1) == 0) {  // 8-byte aligned: two wide stores (fewer bank conflicts)
                    *reinterpret_cast<float2 *>(X + r * xp) = make_float2(v[r][0], v[r][1]);
                    *reinterpret_cast<float2 *>(X + r * xp + 2) = make_float2(v[r][2], v[r][3]);
                } else {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) X[r * xp + cc] = v[r][cc];
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) sum += v[r][cc];
            }
            Quad q[2][2];
#pragma unroll
            for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2) {
                    q[a2][b2] = butterfly(v[2 * a2][2 * b2], v[2 * a2][2 * b2 + 1], v[2 * a2 + 1][2 * b2],
                                          v[2 * a2 + 1][2 * b2 + 1]);
                    put_quad_pairs(slot, geo, pyr_off, 1, 2 * bi + a2, 2 * bj + b2, q[a2][b2]);
                }
            put_quad_pairs(slot, geo, pyr_off, 2, bi, bj, butterfly(q[0][0].ll, q[0][1].ll, q[1][0].ll, q[1][1].ll));
        }
    } else {
        for (int it = threadIdx.x; it < G * n; it += blockDim.x) {
            const int g = fdiv(dn, it), e = it - g * n;
            const int bi = fdiv(dw, e), bj = e - bi * bw;
            const int b = b0 + g;
            float v00 = 0.f, v01 = 0.f, v10 = 0.f, v11 = 0.f;
            if (b < a.B) {
                const T *plane = stg ? stg + (size_t)g * HW : x + ((size_t)b * a.C + c) * HW;
                const T *src = plane + (size_t)(2 * bi) * W + 2 * bj;
                v00 = Act<T>::ld(src); v01 = Act<T>::ld(src + 1);
                v10 = Act<T>::ld(src + W); v11 = Act<T>::ld(src + W + 1);
            }
            float *slot = slots + (size_t)g * geo.slot_floats;
            float *X = slot + x_off + (2 * bi + P) * xp + 2 * bj + P;
            X[0] = v00; X[1] = v01; X[xp] = v10; X[xp + 1] = v11;
            sum += (v00 + v01) + (v10 + v11);
            put_quad_pairs(slot, geo, pyr_off, 1, bi, bj, butterfly(v00, v01, v10, v11));
        }
    }
    return sum;
}

// Later passes: levels l (and l+1 when l+1 <= L) from the low band of level l-1 in shared memory,
// on threads t0 .. t0+nt-1 (nt = 0: the whole CTA).
template <int P>
__device__ __forceinline__ void analysis_from_shared(const LayerArgs &a, const Geo &geo, float *slots, int G,
                                                     const int *pyr_off, int l, int t0 = 0, int nt = 0) {
    const bool two = (l + 1 <= geo.L);
    const FastDiv &dn = a.dv.a_n[l], &dw = a.dv.a_w[l];
    const int bw = (int)dw.d, n = (int)dn.d;
    if (nt == 0) nt = blockDim.x;
    for (int it = (int)threadIdx.x - t0; it < G * n; it += nt) {
        const int g = fdiv(dn, it), e = it - g * n;
        const int bi = fdiv(dw, e), bj = e - bi * bw;
        float *slot = slots + (size_t)g * geo.slot_floats;
        if (two) {
            float v[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) v[r][cc] = get_ll(slot, geo, pyr_off, l - 1, 4 * bi + r, 4 * bj + cc);
            Quad q[2][2];
#pragma unroll
            for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2) {
                    q[a2][b2] = butterfly(v[2 * a2][2 * b2], v[2 * a2][2 * b2 + 1], v[2 * a2 + 1][2 * b2],
                                          v[2 * a2 + 1][2 * b2 + 1]);
                    put_quad_pairs(slot, geo, pyr_off, l, 2 * bi + a2, 2 * bj + b2, q[a2][b2]);
                }
            put_quad_pairs(slot, geo, pyr_off, l + 1, bi, bj,
                           butterfly(q[0][0].ll, q[0][1].ll, q[1][0].ll, q[1][1].ll));
        } else {
            const float v00 = get_ll(slot, geo, pyr_off, l - 1, 2 * bi, 2 * bj);
            const float v01 = get_ll(slot, geo, pyr_off, l - 1, 2 * bi, 2 * bj + 1);
            const float v10 = get_ll(slot, geo, pyr_off, l - 1, 2 * bi + 1, 2 * bj);
            const float v11 = get_ll(slot, geo, pyr_off, l - 1, 2 * bi + 1, 2 * bj + 1);
            put_quad_pairs(slot, geo, pyr_off, l, bi, bj, butterfly(v00, v01, v10, v11));
        }
    }
}

}  // namespace wtconv
