// Tiled weight-gradient kernel of the WTConv layer: the base-path and level-1 correlations,
//     dw'_b[u, v]   = sum_{b,h,w} dy[b, h, w] x[b, h+u-P, w+v-P],   db' = sum dy
//     dW'^1_s[u, v] = sum_{b,i,j} Ghat^1_s[b, i, j] Yhat^1_s[b, i+u-P, j+v-P]     (s = LL, LH, HL, HH)
// with Yhat^1 / Ghat^1 the unnormalised level-1 Haar subbands of x / dy and zero padding outside
// each plane.  (Levels >= 2 are correlated on their pyramids by the level kernels.)
//
// A CTA is one warp that owns channel c and walks a run of units (output tiles of G planes, the
// shallow kernel's tiling).  Per unit one lane loads, with one bulk tensor copy each, the x tile
// with its 2P halo and the dy tile (zero outside the plane); the warp builds both level-1
// pyramids on chip as subband-pair images.  Every lane is pinned to one correlation for the
// whole CTA -- lanes 0-15 the base path (8 x 4 pixel items), lanes 16-23 the subband pair LL|LH
// and lanes 24-31 the pair HL|HH (8 x 2 coefficient items) -- and keeps its k*k tap sums in
// registers (packed f32x2) across all units.  At the end a fixed-order warp-shuffle tree
// reduces each correlation and one lane writes the CTA's partials, so the result is
// deterministic.
#include "wtconv_device.cuh"

namespace wtconv {

namespace {

constexpr int kBaseLanes = 16;  // lanes 0 .. 15: base path; 16 .. 23: pair 0; 24 .. 31: pair 1
constexpr int kPairLanes = 8;

__host__ __device__ inline size_t round128(size_t b) { return (b + 127) / 128 * 128; }

}  // namespace

// Shared memory: raw x tile, raw dy tile (each 128-byte aligned; for fp32 they are the fp32
// tiles X / DY themselves), the fp32 X / DY tiles (narrow types only), the level-1 pair images of
// x (with halo) and of dy (interior).
size_t dw_tile_smem_bytes(const ShallowGeo &sg, int elem_bytes) {
    const size_t dyn = (size_t)sg.G * sg.TH * sg.TW;
    size_t b = round128((size_t)sg.raw_bytes) + round128(dyn * elem_bytes);
    if (elem_bytes != 4) b += (size_t)sg.xbuf * sizeof(float) + dyn * sizeof(float);
    b += (size_t)sg.G * sg.pslot * sizeof(float);  // Yhat^1 pairs
    b += dyn * sizeof(float);                        // Ghat^1 pairs: 2 images of (TH/2) x (TW/2) x 2
    return b + 128;                                  // room to align the base to 128 bytes
}

template <int K, typename T>
__global__ void __launch_bounds__(32, (K <= 5 ? 12 : 8)) wtconv_dw_tile_kernel(const __grid_constant__ DwTileArgs a) {
    constexpr int P = K / 2, KK = K * K, O = 4 - P;
    constexpr int NVP = (kColsL + K - 1 + 1) / 2;  // 16-byte loads per level-1 window row
    constexpr bool kConvert = sizeof(T) != 4;
    extern __shared__ __align__(128) float smem[];
    __shared__ __align__(8) uint64_t bar;
    const ShallowGeo sg = a.sg;
    const int lane = threadIdx.x;
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = sg.G, TH = sg.TH, TW = sg.TW;
    const int dyn = G * TH * TW;
    // bulk tensor copies need 128-byte aligned destinations: align the base by hand
    const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(smem);
    char *raw_x = reinterpret_cast<char *>(smem) + (((s0 + 127u) & ~127u) - s0);
    char *raw_dy = raw_x + round128((size_t)sg.raw_bytes);
    float *X = kConvert ? reinterpret_cast<float *>(raw_dy + round128((size_t)dyn * sizeof(T)))
                        : reinterpret_cast<float *>(raw_x);
    float *DY = kConvert ? X + sg.xbuf : reinterpret_cast<float *>(raw_dy);
    float *ypairs = kConvert ? DY + dyn : reinterpret_cast<float *>(raw_dy + round128((size_t)dyn * sizeof(T)));
    float *gpairs = ypairs + G * sg.pslot;
    const int gw = TW / 2, gimg = G * (TH / 2) * gw * 2;  // Ghat^1 pair image: positions per row, floats
    if (lane == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();

    const FastDiv fd_tiles = a.tiles, fd_tiles_c = a.tiles_c;
    const int u_begin = nbi * a.units_per_cta;
    const int u_end = min(a.units, u_begin + a.units_per_cta);
    const uint32_t bytes = (uint32_t)(G * sg.xrows * sg.xw * (int)sizeof(T) + dyn * (int)sizeof(T));
    auto issue = [&](int u) {
        if (lane == 0) {
            const int bg = (int)fdiv(fd_tiles, (uint32_t)u), t = u - bg * (int)fd_tiles.d;
            const int tr = (int)fdiv(fd_tiles_c, (uint32_t)t), tc = t - tr * sg.tiles_c;
            mbar_arrive_expect_tx(&bar, bytes);
            tma_load_4d(raw_x, &a.tmap_x, tc * TW - sg.padx, tr * TH - 2 * P, c, bg * G, &bar);
            tma_load_4d(raw_dy, &a.tmap_dy, tc * TW, tr * TH, c, bg * G, &bar);
        }
    };

    // lane role and its items per unit
    const int role = lane < kBaseLanes ? 0 : (lane < kBaseLanes + kPairLanes ? 1 : 2);
    const int rl = role == 0 ? lane : (role == 1 ? lane - kBaseLanes : lane - kBaseLanes - kPairLanes);
    const int rstride = role == 0 ? kBaseLanes : kPairLanes;
    const int base_per_plane = sg.items_r * sg.items_c;          // 8 x 4 pixel items
    const int pcols = TW / 4, pair_per_plane = (TH / 16) * pcols;  // 8 x 2 coefficient items
    const int n_items = G * (role == 0 ? base_per_plane : pair_per_plane);
    // level-1 analysis lane layout (positions of the halo'd x pyramid; interior of the dy pyramid)
    const int ycols = sg.ycols;
    const int a_rstep = ycols >= 32 ? 1 : 32 / ycols, a_lanes = ycols >= 32 ? 32 : a_rstep * ycols;
    const int a_row0 = ycols >= 32 ? 0 : lane / ycols, a_col0 = ycols >= 32 ? lane : lane - a_row0 * ycols;
    const int g_rstep = gw >= 32 ? 1 : 32 / gw, g_lanes = gw >= 32 ? 32 : g_rstep * gw;
    const int g_row0 = gw >= 32 ? 0 : lane / gw, g_col0 = gw >= 32 ? lane : lane - g_row0 * gw;

    f2_t acc[KK];
#pragma unroll
    for (int t = 0; t < KK; ++t) acc[t] = 0;
    float gsum = 0.f;

    if (u_begin < u_end) issue(u_begin);
    for (int u = u_begin; u < u_end; ++u) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bar, (uint32_t)(u - u_begin) & 1, a.timeout))) {
            // the flag is raised: this CTA's partials become NaN (the gradients show it), and the
            // CTA leaves without touching the buffers a copy may still target
            const int ns = 1 + 4 * a.L;
            float *part = a.partials + ((size_t)nbi * a.C + c) * ns * (KK + 1);
            for (int i = lane; i < ns * (KK + 1); i += 32) part[i] = __int_as_float(0x7fc00000);
            return;
        }
        __syncwarp();
        if constexpr (kConvert) {
            // raw tiles -> fp32, loads first, then the stores
            const uint2 *rx = reinterpret_cast<const uint2 *>(raw_x);
            const uint2 *rd = reinterpret_cast<const uint2 *>(raw_dy);
            float4 *x4 = reinterpret_cast<float4 *>(X), *d4 = reinterpret_cast<float4 *>(DY);
            const int nx = sg.xbuf / 4, nd = dyn / 4;
            for (int i = lane; i < nx + nd; i += 2 * 32) {
                uint2 v[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int k = i + q * 32 < nx + nd ? i + q * 32 : i;
                    v[q] = k < nx ? rx[k] : rd[k - nx];
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int k = i + q * 32;
                    if (k < nx + nd) {
                        const float4 f = Act<T>::ld4(reinterpret_cast<const T *>(&v[q]));
                        if (k < nx) x4[k] = f;
                        else d4[k - nx] = f;
                    }
                }
            }
            __syncwarp();
            if (u + 1 < u_end) issue(u + 1);  // the raw buffers are free again
        }
        // level-1 pyramids: Yhat^1 of the halo'd x tile, Ghat^1 of the dy tile (both unnormalised)
        if (lane < a_lanes) {
            for (int col = a_col0; col < ycols; col += 32) {
                const float *xs = X + sg.padx - 2 * P + 2 * col + (2 * a_row0) * sg.xw;
                float *y0 = ypairs + 2 * (a_row0 * sg.ypitch + col);
                for (int ya = a_row0; ya < G * sg.yrows; ya += 4 * a_rstep) {
                    f2_t t0[4], t1[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const bool in = ya + q * a_rstep < G * sg.yrows;
                        const float *xq = xs + (in ? 2 * q * a_rstep * sg.xw : 0);
                        t0[q] = *reinterpret_cast<const f2_t *>(xq);
                        t1[q] = *reinterpret_cast<const f2_t *>(xq + sg.xw);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (ya + q * a_rstep < G * sg.yrows) {
                            const f2_t sv = fadd2(t0[q], t1[q]), dv = fsub2(t0[q], t1[q]);
                            const float s0 = lo2(sv), s1 = hi2(sv), d0 = lo2(dv), d1 = hi2(dv);
                            float *yq = y0 + 2 * q * a_rstep * sg.ypitch;
                            *reinterpret_cast<float2 *>(yq) = make_float2(s0 + s1, s0 - s1);
                            *reinterpret_cast<float2 *>(yq + G * sg.yimg) = make_float2(d0 + d1, d0 - d1);
                        }
                    }
                    xs += 8 * a_rstep * sg.xw;
                    y0 += 8 * a_rstep * sg.ypitch;
                }
            }
        }
        if (lane < g_lanes) {
            for (int col = g_col0; col < gw; col += 32) {
                const float *ds = DY + 2 * col + (2 * g_row0) * TW;
                float *g0 = gpairs + 2 * (g_row0 * gw + col);
                for (int ga = g_row0; ga < G * (TH / 2); ga += 4 * g_rstep) {
                    f2_t t0[4], t1[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const bool in = ga + q * g_rstep < G * (TH / 2);
                        const float *dq = ds + (in ? 2 * q * g_rstep * TW : 0);
                        t0[q] = *reinterpret_cast<const f2_t *>(dq);
                        t1[q] = *reinterpret_cast<const f2_t *>(dq + TW);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (ga + q * g_rstep < G * (TH / 2)) {
                            const f2_t sv = fadd2(t0[q], t1[q]), dv = fsub2(t0[q], t1[q]);
                            const float s0 = lo2(sv), s1 = hi2(sv), d0 = lo2(dv), d1 = hi2(dv);
                            float *gq = g0 + 2 * q * g_rstep * gw;
                            *reinterpret_cast<float2 *>(gq) = make_float2(s0 + s1, s0 - s1);
                            *reinterpret_cast<float2 *>(gq + gimg) = make_float2(d0 + d1, d0 - d1);
                        }
                    }
                    ds += 8 * g_rstep * TW;
                    g0 += 8 * g_rstep * gw;
                }
            }
        }
        __syncwarp();

        // this lane's correlation items for the unit
        for (int it = rl; it < n_items; it += rstride) {
            if (role == 0) {
                const int ig = it / base_per_plane, ie = it - ig * base_per_plane;
                const int irs = ie / sg.items_c, ics = ie - irs * sg.items_c;
                const float *xw = X + (ig * sg.xrows + kRows * irs + P) * sg.xw + kCols * ics + sg.padx - 4;
                const float *dw = DY + (ig * TH + kRows * irs) * TW + kCols * ics;
                f2_t gr[kRows][2];
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    const float4 d4v = *reinterpret_cast<const float4 *>(dw + j * TW);
                    gr[j][0] = pk2(d4v.x, d4v.y);
                    gr[j][1] = pk2(d4v.z, d4v.w);
                    gsum += (d4v.x + d4v.y) + (d4v.z + d4v.w);
                }
#pragma unroll
                for (int i = 0; i < kRows + K - 1; ++i) {
                    f2_t e[6], o[5];
                    load_row<3>(xw + i * sg.xw, e, o);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
#pragma unroll
                        for (int u2 = 0; u2 < K; ++u2) {
                            const int j = i - u2;
                            if (j >= 0 && j < kRows) {
#pragma unroll
                                for (int v = 0; v < K; ++v) {
                                    const int s0 = O + v + 2 * q;
                                    const f2_t xv = (s0 & 1) ? o[(s0 - 1) / 2] : e[s0 / 2];
                                    ffma2_acc(acc[u2 * K + v], gr[j][q], xv);
                                }
                            }
                        }
                    }
                }
            } else {
                const int pp = role - 1;
                const int ig = it / pair_per_plane, ie = it - ig * pair_per_plane;
                const int irs = ie / pcols, ics = ie - irs * pcols;
                const float *yw = ypairs + pp * G * sg.yimg + 2 * ((ig * sg.yrows + kRows * irs) * sg.ypitch + 2 * ics);
                const float *gp = gpairs + pp * gimg + 2 * ((ig * (TH / 2) + kRows * irs) * gw + 2 * ics);
                f2_t gr[kRows][kColsL];
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    const ulonglong2 t2 = *reinterpret_cast<const ulonglong2 *>(gp + 2 * j * gw);
                    gr[j][0] = t2.x;
                    gr[j][1] = t2.y;
                }
#pragma unroll
                for (int i = 0; i < kRows + K - 1; ++i) {
                    f2_t xr[2 * NVP];
                    load_pair_row<NVP>(yw + 2 * i * sg.ypitch, xr);
#pragma unroll
                    for (int q = 0; q < kColsL; ++q) {
#pragma unroll
                        for (int u2 = 0; u2 < K; ++u2) {
                            const int j = i - u2;
                            if (j >= 0 && j < kRows) {
#pragma unroll
                                for (int v = 0; v < K; ++v) ffma2_acc(acc[u2 * K + v], gr[j][q], xr[q + v]);
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if constexpr (!kConvert) {
            if (u + 1 < u_end) issue(u + 1);
        }
    }

    // fixed-order warp-shuffle reduction: within 8-lane groups, then the two base groups
    const size_t stride_sig = (size_t)(KK + 1);
    float *out = a.partials + ((size_t)nbi * a.C + c) * (1 + 4 * a.L) * stride_sig;
#pragma unroll
    for (int t = 0; t <= KK; ++t) {
        float lo, hi;
        if (t < KK) {
            lo = lo2(acc[t]);
            hi = hi2(acc[t]);
        } else {
            lo = gsum;
            hi = 0.f;
        }
        if (role == 0) {  // the two halves of a base accumulator are partial sums of one tap
            lo += hi;
            hi = 0.f;
        }
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1) {
            lo += __shfl_xor_sync(0xffffffffu, lo, off);
            hi += __shfl_xor_sync(0xffffffffu, hi, off);
        }
        const float lo8 = __shfl_xor_sync(0xffffffffu, lo, 8);
        if (lane == 0) out[t] = lo + lo8;  // base: signal 0 (tap t, or db' at t == KK)
        if (lane == kBaseLanes || lane == kBaseLanes + kPairLanes) {
            const int s0 = 1 + 2 * (role - 1);  // level-1 subbands 2pp and 2pp+1 are signals 1 + 2pp, 2 + 2pp
            out[s0 * stride_sig + t] = t < KK ? lo : 0.f;
            out[(s0 + 1) * stride_sig + t] = t < KK ? hi : 0.f;
        }
    }
}

template <int K, typename T>
static cudaError_t launch_dw_tile_t(const DwTileArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_dw_tile_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), 32, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_dw_tile_t(size_t smem) {
    auto kern = wtconv_dw_tile_kernel<K, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32, smem) != cudaSuccess) return 0;
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

cudaError_t launch_dw_tile(const DwTileArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_dw_tile_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_dw_tile(int dtype, int K, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_dw_tile_t, smem);
    return 0;
}

}  // namespace wtconv
