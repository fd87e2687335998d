// On-chip Haar analysis passes: one read of each input plane from global memory builds the
// padded fp32 copy of the plane and the first Haar levels; later passes build deeper levels from
// the low band in shared memory.  Each pass computes two levels per item where it can (a 4x4
// block of the finer low band gives four level-l positions and one level-(l+1) position), so an
// L-level pyramid needs ceil(L/2) passes (and barriers).
#pragma once

#include "wtconv_device.cuh"

namespace wtconv {

// Level-l subband images of one slot: padded, interior origin (P, P).
struct LevelView {
    float *base;  // subband 0
    int sub;      // floats between subbands
    int pitch;
};

__device__ __forceinline__ LevelView level_view(float *slot, const Geo &geo, const int *off, int l) {
    return {slot + off[l], geo.rows[l] * geo.pitch[l], geo.pitch[l]};
}

// Pass 1: read G planes of x (type T; from the shared staging area when `stg` is not null, else
// from global memory), write the padded fp32 copy X and Haar level 1 (and level 2 when L >= 2).
// Returns the sum of the values read (used for the bias gradient).
template <typename T, int P>
__device__ __forceinline__ float analysis_from_global(const LayerArgs &a, const Geo &geo, const T *x, const T *stg,
                                                      int c, int b0, float *slots, int x_off, const int *pyr_off) {
    const int G = a.G, H = geo.H, W = geo.W;
    const size_t HW = (size_t)H * W;
    float sum = 0.f;
    if (geo.L >= 2) {
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
                        float4 t = Act<T>::ld4(src + r * W);
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
            float *X = slot + x_off + (4 * bi + P) * geo.pitch[0] + 4 * bj + P;
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    X[r * geo.pitch[0] + cc] = v[r][cc];
                    sum += v[r][cc];
                }
            const LevelView l1 = level_view(slot, geo, pyr_off, 1);
            Quad q[2][2];
#pragma unroll
            for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2) {
                    q[a2][b2] = butterfly(v[2 * a2][2 * b2], v[2 * a2][2 * b2 + 1], v[2 * a2 + 1][2 * b2],
                                          v[2 * a2 + 1][2 * b2 + 1]);
                    put_quad(l1.base, l1.sub, (2 * bi + a2 + P) * l1.pitch + 2 * bj + b2 + P, q[a2][b2]);
                }
            const LevelView l2 = level_view(slot, geo, pyr_off, 2);
            put_quad(l2.base, l2.sub, (bi + P) * l2.pitch + bj + P,
                     butterfly(q[0][0].ll, q[0][1].ll, q[1][0].ll, q[1][1].ll));
        }
    } else {
        const FastDiv &dn = a.dv.a_n[1], &dw = a.dv.a_w[1];
        const int bw = (int)dw.d, n = (int)dn.d;
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
            float *X = slot + x_off + (2 * bi + P) * geo.pitch[0] + 2 * bj + P;
            X[0] = v00; X[1] = v01; X[geo.pitch[0]] = v10; X[geo.pitch[0] + 1] = v11;
            sum += (v00 + v01) + (v10 + v11);
            const LevelView l1 = level_view(slot, geo, pyr_off, 1);
            put_quad(l1.base, l1.sub, (bi + P) * l1.pitch + bj + P, butterfly(v00, v01, v10, v11));
        }
    }
    return sum;
}

// Later passes: levels l (and l+1 when l+1 <= L) from the low band of level l-1 in shared memory.
template <int P>
__device__ __forceinline__ void analysis_from_shared(const LayerArgs &a, const Geo &geo, float *slots, int G,
                                                     const int *pyr_off, int l) {
    const int two = (l + 1 <= geo.L);
    const FastDiv &dn = a.dv.a_n[l], &dw = a.dv.a_w[l];
    const int bw = (int)dw.d, n = (int)dn.d;
    if (two) {
        for (int it = threadIdx.x; it < G * n; it += blockDim.x) {
            const int g = fdiv(dn, it), e = it - g * n;
            const int bi = fdiv(dw, e), bj = e - bi * bw;
            float *slot = slots + (size_t)g * geo.slot_floats;
            const LevelView s = level_view(slot, geo, pyr_off, l - 1);
            const float *ll = s.base + (4 * bi + P) * s.pitch + 4 * bj + P;
            float v[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) v[r][cc] = ll[r * s.pitch + cc];
            const LevelView d1 = level_view(slot, geo, pyr_off, l);
            Quad q[2][2];
#pragma unroll
            for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2) {
                    q[a2][b2] = butterfly(v[2 * a2][2 * b2], v[2 * a2][2 * b2 + 1], v[2 * a2 + 1][2 * b2],
                                          v[2 * a2 + 1][2 * b2 + 1]);
                    put_quad(d1.base, d1.sub, (2 * bi + a2 + P) * d1.pitch + 2 * bj + b2 + P, q[a2][b2]);
                }
            const LevelView d2 = level_view(slot, geo, pyr_off, l + 1);
            put_quad(d2.base, d2.sub, (bi + P) * d2.pitch + bj + P,
                     butterfly(q[0][0].ll, q[0][1].ll, q[1][0].ll, q[1][1].ll));
        }
    } else {
        for (int it = threadIdx.x; it < G * n; it += blockDim.x) {
            const int g = fdiv(dn, it), e = it - g * n;
            const int bi = fdiv(dw, e), bj = e - bi * bw;
            float *slot = slots + (size_t)g * geo.slot_floats;
            const LevelView s = level_view(slot, geo, pyr_off, l - 1);
            const float *ll = s.base + (2 * bi + P) * s.pitch + 2 * bj + P;
            const LevelView d1 = level_view(slot, geo, pyr_off, l);
            put_quad(d1.base, d1.sub, (bi + P) * d1.pitch + bj + P,
                     butterfly(ll[0], ll[1], ll[s.pitch], ll[s.pitch + 1]));
        }
    }
}

}  // namespace wtconv
