// Device code of the WTConv layer for sm_103a (GB300): shared-memory geometry, the on-chip Haar
// analysis, the k x k micro-tile convolutions, the closed-form synthesis gather and the weight
// gradient correlations.  Host code sees only the argument structs and the launchers declared
// in wtconv_internal.h.
//
// The method (paper "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation", Resumo Tecnico / Metodologia):
//   * on-chip Haar analysis: the 2x2 butterflies of every level are recomputed from one read of
//     the input plane and kept in shared memory; no coefficient tensor reaches HBM;
//   * weight folding: each learned scale is multiplied into its conv kernel (and the base scale
//     into the base bias) when the kernel is staged, so no separate scale pass exists;
//   * closed-form synthesis: output pixel (h, w) gathers sum_l 2^-l sum_s sigma_s Z^l_s[h>>l, w>>l]
//     with sigma_s set by bit l-1 of h (row) and w (column) -- one pass, no cascade buffers.
// Power-of-two factors are moved out of the butterflies: the pyramid is kept unnormalised
// (Yhat^l = 2^l Y^l, exact), so the level-l kernels carry 4^-l.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wtconv_internal.h"

namespace wtconv {

// ------------------------------------------------------------------ activation element types

template <typename T> struct Act;
template <> struct Act<float> {
    static __device__ __forceinline__ float ld(const float *p) { return *p; }
    static __device__ __forceinline__ void st(float *p, float v) { *p = v; }
};
template <> struct Act<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
};
template <> struct Act<__half> {
    static __device__ __forceinline__ float ld(const __half *p) { return __half2float(*p); }
    static __device__ __forceinline__ void st(__half *p, float v) { *p = __float2half_rn(v); }
};

// 16-byte vector of activations <-> floats
template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    static __device__ __forceinline__ void unpack(const uint4 &u, float *f);
};
template <> __device__ __forceinline__ void Vec16<float>::unpack(const uint4 &u, float *f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <> __device__ __forceinline__ void Vec16<__nv_bfloat16>::unpack(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
template <> __device__ __forceinline__ void Vec16<__half>::unpack(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
        float2 t = __half22float2(h);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// Four consecutive outputs of one row, rounded to T and stored (vectorised when `vec`).
template <typename T>
__device__ __forceinline__ void store4(T *dst, const float *v, int n_valid, bool vec) {
    if (vec && n_valid == 4) {
        if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            T t[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) Act<T>::st(&t[i], v[i]);
            *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(t);
        }
    } else {
        for (int i = 0; i < n_valid; ++i) Act<T>::st(dst + i, v[i]);
    }
}

// ---------------------------------------------------------------------------- plane loading

// Copy one H x W plane from global memory into the interior of a zero-padded shared buffer
// (interior origin (P, P), row pitch `pitch`), converting to fp32.  A missing plane (b >= B)
// is written as zeros.
template <typename T, int P>
__device__ __forceinline__ void load_plane(const T *__restrict__ g, bool valid, float *dst, int H, int W,
                                           int pitch) {
    const int HW = H * W;
    float *base = dst + P * pitch + P;
    if (!valid) {
        for (int e = threadIdx.x; e < HW; e += blockDim.x) {
            int r = e / W, c = e - r * W;
            base[r * pitch + c] = 0.f;
        }
        return;
    }
    constexpr int N = Vec16<T>::N;
    if ((HW % N) == 0 && (reinterpret_cast<uintptr_t>(g) & 15) == 0) {
        const uint4 *g4 = reinterpret_cast<const uint4 *>(g);
        const int nv = HW / N;
        for (int q = threadIdx.x; q < nv; q += blockDim.x) {
            uint4 u = g4[q];
            float f[N];
            Vec16<T>::unpack(u, f);
            int e = q * N;
            int r = e / W, c = e - r * W;
#pragma unroll
            for (int i = 0; i < N; ++i) {
                base[r * pitch + c] = f[i];
                if (++c == W) { c = 0; ++r; }
            }
        }
    } else {
        for (int e = threadIdx.x; e < HW; e += blockDim.x) {
            int r = e / W, c = e - r * W;
            base[r * pitch + c] = Act<T>::ld(g + e);
        }
    }
}

// ------------------------------------------------------------------------- Haar analysis

// One level of the unnormalised Haar butterfly for every slot: level l's four subbands (interior
// (i, j) of the padded level-l buffer) from the 2x2 blocks of the level l-1 low band.
// LL = a+b+c+d, LH = a-b+c-d, HL = a+b-c-d, HH = a-b-c+d for the block [[a, b], [c, d]].
template <int P>
__device__ __forceinline__ void analysis_level(const Geo &geo, float *slots, int nslots, int l,
                                               int src_off0, const int *dst_off) {
    const int h = geo.H >> l, w = geo.W >> l;
    const int sp = geo.pitch[l - 1], dp = geo.pitch[l];
    const int sub = geo.rows[l] * dp;
    const int n = h * w;
    for (int it = threadIdx.x; it < nslots * n; it += blockDim.x) {
        int g = it / n, e = it - g * n;
        int i = e / w, j = e - i * w;
        float *slot = slots + (size_t)g * geo.slot_floats;
        const float *src = slot + (l == 1 ? src_off0 : dst_off[l - 1]);
        const float *s0 = src + (2 * i + P) * sp + (2 * j + P);
        float a, b, c, d;
        if constexpr ((P & 1) == 0) {
            float2 t0 = *reinterpret_cast<const float2 *>(s0);
            float2 t1 = *reinterpret_cast<const float2 *>(s0 + sp);
            a = t0.x; b = t0.y; c = t1.x; d = t1.y;
        } else {
            a = s0[0]; b = s0[1]; c = s0[sp]; d = s0[sp + 1];
        }
        float s_top = a + b, d_top = a - b, s_bot = c + d, d_bot = c - d;
        float *o = slot + dst_off[l] + (i + P) * dp + (j + P);
        o[0] = s_top + s_bot;        // LL
        o[sub] = d_top + d_bot;      // LH
        o[2 * sub] = s_top - s_bot;  // HL
        o[3 * sub] = d_top - d_bot;  // HH
    }
}

// -------------------------------------------------------------------- k x k micro-tile conv

// acc[r][c] += sum_{u,v} wk[u*K+v] * src[(r0+r+u) * pitch + c0+c+v] for a 2 x 4 output tile whose
// zero-padded input window starts at (r0, c0); wk in shared memory (broadcast reads).
template <int K>
__device__ __forceinline__ void conv_tile_2x4(const float *__restrict__ src, int pitch, int r0, int c0,
                                              const float *__restrict__ wk, float (&acc)[2][4]) {
    constexpr int NW = (4 + K - 1 + 3) / 4;  // float4 loads per window row
    float w[K * K];
#pragma unroll
    for (int i = 0; i < K * K; ++i) w[i] = wk[i];
#pragma unroll
    for (int ir = 0; ir < K + 1; ++ir) {
        float row[4 * NW];
        const float4 *p4 = reinterpret_cast<const float4 *>(src + (r0 + ir) * pitch + c0);
#pragma unroll
        for (int q = 0; q < NW; ++q) {
            float4 t = p4[q];
            row[4 * q] = t.x; row[4 * q + 1] = t.y; row[4 * q + 2] = t.z; row[4 * q + 3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int u = ir - r;
            if (u >= 0 && u < K) {
#pragma unroll
                for (int v = 0; v < K; ++v)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(w[u * K + v], row[c + v], acc[r][c]);
            }
        }
    }
}

// ------------------------------------------------------------------ weight staging (folding)

// Stage channel c's kernels into shared memory with the scales folded in:
//   slot 0            : s_b[c] * w_b[c]
//   slot 1 + 4(l-1)+s : 4^-l * s_l[4c+s] * w_l[4c+s]     (4^-l: unnormalised pyramid, see top)
// `flip` rotates every kernel by 180 degrees (the transposed conv of the input gradient).
// bias_out receives s_b[c] * b_b[c] (or 0 when !with_bias).
template <int K>
__device__ __forceinline__ void stage_weights(const LayerArgs &a, int c, float *wts, float *bias_out) {
    constexpr int KK = K * K, KS = wslot_stride(K);
    const int nsig = 1 + 4 * a.L;
    for (int it = threadIdx.x; it < nsig * KK; it += blockDim.x) {
        int sig = it / KK, t = it - sig * KK;
        int tu = t / K, tv = t - tu * K;
        int src_t = a.flip ? (K - 1 - tu) * K + (K - 1 - tv) : t;
        float v;
        if (sig == 0) {
            v = a.base_scale[c] * a.base_w[(size_t)c * KK + src_t];
        } else {
            int l = (sig - 1) / 4 + 1, s = (sig - 1) & 3;
            size_t ch = (size_t)(l - 1) * 4 * a.C + 4 * c + s;
            v = ldexpf(a.wavelet_scale[ch] * a.wavelet_w[ch * KK + src_t], -2 * l);
        }
        wts[sig * KS + t] = v;
    }
    if (threadIdx.x == 0) *bias_out = a.with_bias ? a.base_scale[c] * a.base_bias[c] : 0.f;
}

// ------------------------------------------------------------------ conv phase (levels 1..L)

// Z^l_s = Wfold^l_s (*) Yhat^l_s for every slot, level and subband, flattened over 2x4 tiles.
template <int K>
__device__ __forceinline__ void conv_levels(const Geo &geo, float *slots, int nslots, const int *pyr_off,
                                            const float *wts) {
    constexpr int KS = wslot_stride(K);
    int lvl_start[kMaxLevels + 2];
    int tot = 0;
    for (int l = 1; l <= geo.L; ++l) {
        lvl_start[l] = tot;
        tot += 4 * ((geo.zrows[l] / 2) * (geo.zpitch[l] / 4));
    }
    lvl_start[geo.L + 1] = tot;
    for (int it = threadIdx.x; it < nslots * tot; it += blockDim.x) {
        int g = it / tot, e = it - g * tot;
        int l = 1;
        while (e >= lvl_start[l + 1]) ++l;
        e -= lvl_start[l];
        const int tc = geo.zpitch[l] / 4, nt = (geo.zrows[l] / 2) * tc;
        int s = e / nt;
        e -= s * nt;
        int tr = e / tc, tcc = e - tr * tc;
        float *slot = slots + (size_t)g * geo.slot_floats;
        const float *src = slot + pyr_off[l] + s * geo.rows[l] * geo.pitch[l];
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        conv_tile_2x4<K>(src, geo.pitch[l], 2 * tr, 4 * tcc, wts + (1 + 4 * (l - 1) + s) * KS, acc);
        float *z = slot + geo.off_z[l] + s * geo.zrows[l] * geo.zpitch[l] + (2 * tr) * geo.zpitch[l] + 4 * tcc;
        *reinterpret_cast<float4 *>(z) = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        *reinterpret_cast<float4 *>(z + geo.zpitch[l]) = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
    }
}

// ------------------------------------------------------- output phase: base conv + synthesis

// Closed-form synthesis for the 2x4 output tile at (h0, w0) (h0 even, w0 % 4 == 0):
//   out[r][c] += sum_l sum_s sigma_s(bit_{l-1}(h0+r), bit_{l-1}(w0+c)) * Z^l_s[(h0+r)>>l][(w0+c)>>l]
// Level 1: the tile covers two coefficients (columns), row bit a = r, column bit b = c & 1.
// Level 2: one coefficient; a is tile-uniform, b = c >> 1.  Levels >= 3: one coefficient with
// tile-uniform signs, summed into a scalar first.
__device__ __forceinline__ void synth_gather(const Geo &geo, const float *slot, int h0, int w0,
                                             float (&out)[2][4]) {
    {   // level 1
        const int zp = geo.zpitch[1], zs = geo.zrows[1] * zp;
        const float *z = slot + geo.off_z[1] + (h0 >> 1) * zp + (w0 >> 1);
        float2 z0 = *reinterpret_cast<const float2 *>(z);
        float2 z1 = *reinterpret_cast<const float2 *>(z + zs);
        float2 z2 = *reinterpret_cast<const float2 *>(z + 2 * zs);
        float2 z3 = *reinterpret_cast<const float2 *>(z + 3 * zs);
        const float zz0[2] = {z0.x, z0.y}, zz1[2] = {z1.x, z1.y}, zz2[2] = {z2.x, z2.y}, zz3[2] = {z3.x, z3.y};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float p0 = zz0[q] + zz2[q], p1 = zz0[q] - zz2[q];
            float q0 = zz1[q] + zz3[q], q1 = zz1[q] - zz3[q];
            out[0][2 * q] += p0 + q0;
            out[0][2 * q + 1] += p0 - q0;
            out[1][2 * q] += p1 + q1;
            out[1][2 * q + 1] += p1 - q1;
        }
    }
    if (geo.L >= 2) {  // level 2
        const int zp = geo.zpitch[2], zs = geo.zrows[2] * zp;
        const float *z = slot + geo.off_z[2] + (h0 >> 2) * zp + (w0 >> 2);
        const bool a = (h0 >> 1) & 1;
        float z0 = z[0], z1 = z[zs], z2 = z[2 * zs], z3 = z[3 * zs];
        float p = a ? z0 - z2 : z0 + z2;
        float q = a ? z1 - z3 : z1 + z3;
        float v0 = p + q, v1 = p - q;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            out[r][0] += v0; out[r][1] += v0; out[r][2] += v1; out[r][3] += v1;
        }
    }
    float deep = 0.f;
    for (int l = 3; l <= geo.L; ++l) {
        const int zp = geo.zpitch[l], zs = geo.zrows[l] * zp;
        const float *z = slot + geo.off_z[l] + (h0 >> l) * zp + (w0 >> l);
        const bool a = (h0 >> (l - 1)) & 1, b = (w0 >> (l - 1)) & 1;
        float z0 = z[0], z1 = z[zs], z2 = z[2 * zs], z3 = z[3 * zs];
        float p = a ? z0 - z2 : z0 + z2;
        float q = a ? z1 - z3 : z1 + z3;
        deep += b ? p - q : p + q;
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) out[r][c] += deep;
}

// y (or dx) tiles: bias + base conv over the padded full-resolution input + closed-form
// synthesis of the per-level conv outputs; rounded to T and written to global memory.
template <int K, typename T>
__device__ __forceinline__ void output_phase(const LayerArgs &a, const Geo &geo, float *slots, int nslots,
                                             int in_off, const float *wts, float bias, T *out, int c,
                                             int b0) {
    const int tc = (geo.W + 3) / 4, tr = geo.H / 2, nt = tr * tc;
    const bool vec = (geo.W % 4) == 0;
    for (int it = threadIdx.x; it < nslots * nt; it += blockDim.x) {
        int g = it / nt, e = it - g * nt;
        const int b = b0 + g;
        if (b >= a.B) continue;
        int trr = e / tc, tcc = e - trr * tc;
        const int h0 = 2 * trr, w0 = 4 * tcc;
        const float *slot = slots + (size_t)g * geo.slot_floats;
        float acc[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) acc[r][cc] = bias;
        conv_tile_2x4<K>(slot + in_off, geo.pitch[0], h0, w0, wts, acc);
        synth_gather(geo, slot, h0, w0, acc);
        T *dst = out + ((size_t)b * a.C + c) * geo.H * geo.W + (size_t)h0 * geo.W + w0;
        const int nv = min(4, geo.W - w0);
        store4<T>(dst, acc[0], nv, vec);
        store4<T>(dst + geo.W, acc[1], nv, vec);
    }
}

// --------------------------------------------------------------- weight-gradient correlation

// acc[u*K+v] += sum over the 4x4 pixel tile at interior (i0, j0) of G[i][j] * Y[i+u-P][j+v-P]
// (Y zero-padded, origin of the window = padded (i0, j0)); acc[K*K] += sum of G (used for the
// base path's bias gradient).
template <int K>
__device__ __forceinline__ void dw_tile_4x4(const float *__restrict__ ysrc, const float *__restrict__ gsrc,
                                            int pitch, int i0, int j0, float *acc) {
    constexpr int P = K / 2, NW = (4 + K - 1 + 3) / 4;
    float gv[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const float *gp = gsrc + (i0 + r + P) * pitch + (j0 + P);
        if constexpr ((P & 1) == 0) {
            float2 t0 = *reinterpret_cast<const float2 *>(gp);
            float2 t1 = *reinterpret_cast<const float2 *>(gp + 2);
            gv[r][0] = t0.x; gv[r][1] = t0.y; gv[r][2] = t1.x; gv[r][3] = t1.y;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) gv[r][c] = gp[c];
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[K * K] += gv[r][c];
    }
#pragma unroll
    for (int ir = 0; ir < K + 3; ++ir) {
        float row[4 * NW];
        const float4 *p4 = reinterpret_cast<const float4 *>(ysrc + (i0 + ir) * pitch + j0);
#pragma unroll
        for (int q = 0; q < NW; ++q) {
            float4 t = p4[q];
            row[4 * q] = t.x; row[4 * q + 1] = t.y; row[4 * q + 2] = t.z; row[4 * q + 3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int u = ir - r;
            if (u >= 0 && u < K) {
#pragma unroll
                for (int v = 0; v < K; ++v)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[u * K + v] = fmaf(gv[r][c], row[c + v], acc[u * K + v]);
            }
        }
    }
}

// Sum NA (<= 32 * NB32) per-lane accumulators across the warp so that lane t ends up holding
// total[t + 32 * blk] for each 32-wide block (butterfly reduce-scatter; fixed order).
template <int NA32>
__device__ __forceinline__ void warp_reduce_scatter(float *v /* [NA32] */, float *res /* [NA32/32] */) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int blk = 0; blk < NA32 / 32; ++blk) {
        float *x = v + 32 * blk;
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            const bool upper = lane & m;
#pragma unroll
            for (int i = 0; i < m; ++i) {
                float send = upper ? x[i] : x[i + m];
                float keep = upper ? x[i + m] : x[i];
                x[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
        }
        res[blk] = x[0];
    }
}

}  // namespace wtconv
