// Weight gradient of the WTConv layer for planes too large for the whole-plane kernel.
//
// The two Haar pyramids (Yhat of x, Ghat of dy; unnormalised butterflies) are written level by
// level to the workspace as one float4 (LL, LH, HL, HH) per position, then each level is
// correlated tile by tile:
//     dW'^l_s[u, v] = sum_{b,i,j} Ghat^l_s[b, i, j] Yhat^l_s[b, i+u-P, j+v-P]      (level l, subband s)
//     dw'_b[u, v]   = sum_{b,h,w} dy[b, h, w] x[b, h+u-P, w+v-P],   db' = sum dy   (base path)
// with zero padding outside each plane.  CTA n of a channel takes the units n, n + nb, ... of a
// level (unit = one batch entry's tile), keeps its tap sums in registers and reduces them in a
// fixed order, so every (channel, signal, tap) gets nb partials that the shared finalize kernel
// sums and unfolds (the 4^-l of the unnormalised pyramids included).  No atomics: deterministic.
#include "wtconv_device.cuh"

namespace wtconv {

namespace {

constexpr int kTH = 16, kTW = 64;  // correlation tile (positions of the level)
constexpr int kCorrThreads = 256;

template <typename S> struct PyrSrc;
template <> struct PyrSrc<float4> {  // a finer pyramid level: its LL band
    static __device__ __forceinline__ float ll(const float4 *p, size_t i) { return p[i].x; }
};
template <typename T> struct PyrSrc {  // the input planes themselves
    static __device__ __forceinline__ float ll(const T *p, size_t i) { return Act<T>::ld(p + i); }
};

// One Haar level of both tensors (blockIdx.y selects x or dy): position (i, j) of level l from
// the 2x2 block at (2i, 2j) of the finer level's LL band (the input plane for l = 1).
template <typename S>
__global__ void __launch_bounds__(256) wtconv_haar_level_kernel(const S *src_x, const S *src_dy, float4 *dst_x,
                                                                  float4 *dst_dy, long long planes, int Hl, int Wl) {
    const S *src = blockIdx.y ? src_dy : src_x;
    float4 *dst = blockIdx.y ? dst_dy : dst_x;
    const long long n = planes * Hl * Wl;
    const size_t W0 = 2 * (size_t)Wl;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
         idx += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(idx % Wl);
        const long long rest = idx / Wl;
        const int i = (int)(rest % Hl);
        const long long p = rest / Hl;
        const size_t o = ((size_t)p * 2 * Hl + 2 * (size_t)i) * W0 + 2 * (size_t)j;
        const Quad q = butterfly(PyrSrc<S>::ll(src, o), PyrSrc<S>::ll(src, o + 1), PyrSrc<S>::ll(src, o + W0),
                                 PyrSrc<S>::ll(src, o + W0 + 1));
        dst[idx] = make_float4(q.ll, q.lh, q.hl, q.hh);
    }
}

// Level 2 of every plane straight from the input: one thread per level-2 position reads its
// 4 x 4 pixel block, forms the four level-1 low bands (unnormalised 2 x 2 sums) and their
// butterfly, and writes the quad (LL, LH, HL, HH) to q2 [B*C][H/4][W/4].  Two positions per
// iteration keep eight row loads in flight.  W % 4 == 0 (L >= 2), so rows load as vectors.
// blockIdx.y selects the tensor (x or dy).
template <typename T>
__global__ void __launch_bounds__(256) wtconv_level2_kernel(const T *__restrict__ x0, const T *__restrict__ x1,
                                                            float4 *__restrict__ q0, float4 *__restrict__ q1,
                                                            long long n, int W4, int W) {
    const T *__restrict__ x = blockIdx.y ? x1 : x0;
    float4 *__restrict__ q2 = blockIdx.y ? q1 : q0;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; i0 < n; i0 += 2 * stride) {
        float4 v[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long i = i0 + h * stride;
            const long long ii = i < n ? i : i0;
            const long long prow = ii / W4;  // plane * (H/4) + block row
            const int bj = (int)(ii - prow * W4);
            const T *src = x + (size_t)prow * 4 * W + 4 * (size_t)bj;
#pragma unroll
            for (int r = 0; r < 4; ++r) v[h][r] = Act<T>::ld4(src + (size_t)r * W);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long i = i0 + h * stride;
            if (i >= n) break;
            const float ll00 = (v[h][0].x + v[h][0].y) + (v[h][1].x + v[h][1].y);
            const float ll01 = (v[h][0].z + v[h][0].w) + (v[h][1].z + v[h][1].w);
            const float ll10 = (v[h][2].x + v[h][2].y) + (v[h][3].x + v[h][3].y);
            const float ll11 = (v[h][2].z + v[h][2].w) + (v[h][3].z + v[h][3].w);
            const Quad q = butterfly(ll00, ll01, ll10, ll11);
            q2[i] = make_float4(q.ll, q.lh, q.hl, q.hh);
        }
    }
}

template <typename S, int NSUB>
__device__ __forceinline__ void load_sub(const S *p, size_t i, bool in, float (&v)[NSUB]) {
    if constexpr (NSUB == 4) {
        const float4 t = in ? p[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
        v[0] = in ? Act<S>::ld(p + i) : 0.f;
    }
}

// Correlation of one level.  NSUB = 1: the base path on the input planes (type S = T);
// NSUB = 4: a pyramid level (S = float4), one subband per quarter of the CTA.
template <int K, int NSUB, typename S>
__global__ void __launch_bounds__(kCorrThreads) wtconv_dw_corr_kernel(const S *ysrc, const S *gsrc, int B, int C,
                                                                        int Hl, int Wl, int nb, int nsig, int sig0,
                                                                        float *partials) {
    constexpr int P = K / 2, KK = K * K, NA = KK + 1, RP = NA + 1;
    constexpr int YH = kTH + 2 * P, YW = kTW + 2 * P;
    constexpr int TPS = kCorrThreads / NSUB;  // threads per subband
    constexpr int IPR = kTW / 4;              // 1 x 4 items per tile row
    __shared__ float ys[NSUB][YH][YW];
    __shared__ float gs[NSUB][kTH][kTW];
    extern __shared__ float red[];            // kCorrThreads x RP
    const int c = blockIdx.x % C, n = blockIdx.x / C;
    const int s = threadIdx.x / TPS, ts = threadIdx.x - s * TPS;
    const int tiles_c = (Wl + kTW - 1) / kTW;
    const int tiles = ((Hl + kTH - 1) / kTH) * tiles_c;
    const long long units = (long long)B * tiles;
    float acc[KK];
#pragma unroll
    for (int t = 0; t < KK; ++t) acc[t] = 0.f;
    float gsum = 0.f;

    for (long long u = n; u < units; u += nb) {
        const int b = (int)(u / tiles), t = (int)(u - (long long)b * tiles);
        const int tr = t / tiles_c, tc = t - tr * tiles_c;
        const int r0 = tr * kTH, c0 = tc * kTW;
        const S *yp = ysrc + ((size_t)b * C + c) * Hl * Wl;
        const S *gp = gsrc + ((size_t)b * C + c) * Hl * Wl;
        __syncthreads();  // the previous tile is consumed
        for (int e = threadIdx.x; e < YH * YW; e += kCorrThreads) {
            const int i = e / YW, j = e - i * YW;
            const int r = r0 - P + i, col = c0 - P + j;
            const bool in = r >= 0 && r < Hl && col >= 0 && col < Wl;
            float v[NSUB];
            load_sub<S, NSUB>(yp, in ? (size_t)r * Wl + col : 0, in, v);
#pragma unroll
            for (int q = 0; q < NSUB; ++q) ys[q][i][j] = v[q];
        }
        for (int e = threadIdx.x; e < kTH * kTW; e += kCorrThreads) {
            const int i = e / kTW, j = e - i * kTW;
            const int r = r0 + i, col = c0 + j;
            const bool in = r < Hl && col < Wl;
            float v[NSUB];
            load_sub<S, NSUB>(gp, in ? (size_t)r * Wl + col : 0, in, v);
#pragma unroll
            for (int q = 0; q < NSUB; ++q) gs[q][i][j] = v[q];
        }
        __syncthreads();
        for (int it = ts; it < kTH * IPR; it += TPS) {
            const int i = it / IPR, j0 = 4 * (it - i * IPR);
            float g[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                g[q] = gs[s][i][j0 + q];
                gsum += g[q];
            }
#pragma unroll
            for (int uu = 0; uu < K; ++uu) {
                float yv[4 + K - 1];
#pragma unroll
                for (int m = 0; m < 4 + K - 1; ++m) yv[m] = ys[s][i + uu][j0 + m];
#pragma unroll
                for (int v = 0; v < K; ++v)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[uu * K + v] = fmaf(g[q], yv[q + v], acc[uu * K + v]);
            }
        }
    }
    // fixed-order reduction over the threads of each subband
    float *mine = red + threadIdx.x * RP;
#pragma unroll
    for (int t = 0; t < KK; ++t) mine[t] = acc[t];
    mine[KK] = NSUB == 1 ? gsum : 0.f;
    __syncthreads();
    for (int j = threadIdx.x; j < NSUB * NA; j += kCorrThreads) {
        const int ss = j / NA, tap = j - ss * NA;
        float v = 0.f;
        for (int th = 0; th < TPS; ++th) v += red[(ss * TPS + th) * RP + tap];
        partials[(((size_t)n * C + c) * nsig + sig0 + ss) * NA + tap] = v;
    }
}

template <int K, typename T>
cudaError_t launch_dw_pyramid_t(const DwPyramidArgs &a, cudaStream_t st) {
    const long long planes = (long long)a.B * a.C;
    const int nsig = 1 + 4 * a.L;
    constexpr int RP = K * K + 2;
    const size_t red_bytes = (size_t)kCorrThreads * RP * sizeof(float);
    // 1. pyramids, level by level (from level 2 on when the tiled kernel covers base and level 1:
    //    level 2 then comes straight from 4 x 4 pixel blocks)
    if (a.from_level == 2) {
        const long long n = planes * (a.H >> 2) * (a.W >> 2);
        long long blocks = (n + 2 * 256 - 1) / (2 * 256);
        if (blocks > (1LL << 20)) blocks = 1LL << 20;
        wtconv_level2_kernel<T><<<dim3((unsigned)blocks, 2), 256, 0, st>>>(
            static_cast<const T *>(a.x), static_cast<const T *>(a.dy), a.pyr_x[2], a.pyr_dy[2], n, a.W >> 2, a.W);
    }
    for (int l = a.from_level == 2 ? 3 : 1; l <= a.L; ++l) {
        const int Hl = a.H >> l, Wl = a.W >> l;
        const long long n = planes * Hl * Wl;
        long long blocks = (n + 255) / 256;
        if (blocks > 65535LL * 16) blocks = 65535LL * 16;
        const dim3 grid((unsigned)blocks, 2);
        if (l == 1)
            wtconv_haar_level_kernel<T><<<grid, 256, 0, st>>>(static_cast<const T *>(a.x),
                                                              static_cast<const T *>(a.dy), a.pyr_x[1],
                                                              a.pyr_dy[1], planes, Hl, Wl);
        else
            wtconv_haar_level_kernel<float4><<<grid, 256, 0, st>>>(a.pyr_x[l - 1], a.pyr_dy[l - 1], a.pyr_x[l],
                                                                   a.pyr_dy[l], planes, Hl, Wl);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 2. correlations: base path, then every level (static + dynamic shared memory exceeds the
    //    default 48 KB window, so the dynamic part is opted in explicitly)
    e = cudaFuncSetAttribute(wtconv_dw_corr_kernel<K, 1, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)red_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(wtconv_dw_corr_kernel<K, 4, float4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)red_bytes);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(a.nb * a.C));
    if (a.from_level == 1)
        wtconv_dw_corr_kernel<K, 1, T><<<grid, kCorrThreads, red_bytes, st>>>(
            static_cast<const T *>(a.x), static_cast<const T *>(a.dy), a.B, a.C, a.H, a.W, a.nb, nsig, 0, a.partials);
    for (int l = a.from_level; l <= a.L; ++l)
        wtconv_dw_corr_kernel<K, 4, float4><<<grid, kCorrThreads, red_bytes, st>>>(
            a.pyr_x[l], a.pyr_dy[l], a.B, a.C, a.H >> l, a.W >> l, a.nb, nsig, 1 + 4 * (l - 1), a.partials);
    return cudaGetLastError();
}

}  // namespace

size_t dw_pyramid_bytes(int B, int C, int H, int W, int L, int from_level) {
    size_t bytes = 0;
    for (int l = from_level; l <= L; ++l) bytes += 2 * (((size_t)B * C * (H >> l) * (W >> l) * sizeof(float4) + 255) / 256 * 256);
    return bytes;
}

cudaError_t launch_dw_pyramid(const DwPyramidArgs &a, int dtype, cudaStream_t st) {
    switch (a.K * 4 + dtype) {
    case 3 * 4 + 0: return launch_dw_pyramid_t<3, float>(a, st);
    case 3 * 4 + 1: return launch_dw_pyramid_t<3, __nv_bfloat16>(a, st);
    case 3 * 4 + 2: return launch_dw_pyramid_t<3, __half>(a, st);
    case 5 * 4 + 0: return launch_dw_pyramid_t<5, float>(a, st);
    case 5 * 4 + 1: return launch_dw_pyramid_t<5, __nv_bfloat16>(a, st);
    case 5 * 4 + 2: return launch_dw_pyramid_t<5, __half>(a, st);
    case 7 * 4 + 0: return launch_dw_pyramid_t<7, float>(a, st);
    case 7 * 4 + 1: return launch_dw_pyramid_t<7, __nv_bfloat16>(a, st);
    case 7 * 4 + 2: return launch_dw_pyramid_t<7, __half>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace wtconv
