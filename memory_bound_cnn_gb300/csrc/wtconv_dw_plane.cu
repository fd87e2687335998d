// Fused whole-plane weight-gradient kernel of the WTConv layer:
//     dw'_b[u, v]   = sum_{b,h,w} dy[b, h, w] x[b, h+u-P, w+v-P],   db' = sum dy      (base path)
//     dW'^l_s[u, v] = sum_{b,i,j} Ghat^l_s[b, i, j] Yhat^l_s[b, i+u-P, j+v-P]        (level l, subband s)
// with Yhat / Ghat the unnormalised Haar pyramids of x / dy and zero padding outside each plane.
//
// A CTA of up to kDwPlaneMaxThreads threads owns channel c and a run of batch entries, one plane at a time:
//   1. one bulk tensor copy each brings x with a 2P halo and dy (zero outside the plane);
//   2. level 1 of both is computed as padded subband-pair images, levels >= 2 of both from the
//      level-1 low bands, all on chip;
//   3. every thread is pinned, for the whole CTA, to a share of one correlation's items (the
//      base path on 8 x 4 pixel items, or one subband pair of one level on 8 x 2 coefficient
//      items) and keeps its k*k tap sums in registers (packed f32x2) across all planes.  The base
//      threads fill whole warps, and every level's items run the same code on its own images, so
//      no warp splits between two item codes.
// At the end the tap sums are reduced in a fixed thread order into one partial per
// (channel, signal, tap): deterministic, no atomics.
#include "wtconv_items.cuh"

namespace wtconv {

namespace {

__host__ __device__ inline size_t r128(size_t b) { return (b + 127) / 128 * 128; }

// Shared-memory layout (bytes from a 128-byte aligned base).  fp32: nbuf copy buffers of x (+ halo)
// and dy, where the bulk copies land and the analysis and base items read.  Narrow types: one fp32
// X and DY, and nbuf buffers of the raw copies.  Then the level-1 pair images of x and dy (same
// padded layout) and the slot of levels >= 2.  With nbuf = 2 the next plane's copies run while
// the CTA works on the current one.
struct DwPlaneLayout {
    size_t x[2], dy[2], rx[2], rdy[2], y1, g1, deep, end, total;
};

__host__ __device__ inline DwPlaneLayout dw_plane_layout(const DwPlaneArgs &a, int eb) {
    DwPlaneLayout p;
    const ShallowGeo &sg = a.sg;
    const size_t dyn = (size_t)sg.TH * sg.TW;
    const size_t l1 = (size_t)2 * 2 * a.y1rows * sg.ypitch * sizeof(float);  // both pairs of one signal
    const int nbuf = a.nbuf == 2 ? 2 : 1;
    size_t o = 0;
    if (eb == 4) {
        for (int i = 0; i < nbuf; ++i) {
            p.x[i] = o;
            o += r128((size_t)sg.xbuf * sizeof(float));
            p.dy[i] = o;
            o += r128(dyn * sizeof(float));
        }
        if (nbuf == 1) { p.x[1] = p.x[0]; p.dy[1] = p.dy[0]; }
        for (int i = 0; i < 2; ++i) { p.rx[i] = p.x[i]; p.rdy[i] = p.dy[i]; }
    } else {
        p.x[0] = p.x[1] = o;
        o += r128((size_t)sg.xbuf * sizeof(float));
        p.dy[0] = p.dy[1] = o;
        o += r128(dyn * sizeof(float));
        for (int i = 0; i < nbuf; ++i) {
            p.rx[i] = o;
            o += r128((size_t)sg.xrows * sg.xw * eb);
            p.rdy[i] = o;
            o += r128(dyn * eb);
        }
        if (nbuf == 1) { p.rx[1] = p.rx[0]; p.rdy[1] = p.rdy[0]; }
    }
    p.y1 = o;
    o += r128(l1);
    p.g1 = o;
    o += r128(l1);
    p.deep = o;
    o += r128((a.L >= 2 ? (size_t)a.dg.slot_floats : 0) * sizeof(float));
    p.end = o;
    // the end-of-CTA reduction reuses the space from offset 0 on
    const size_t red = (size_t)a.nthreads * (2 * a.K * a.K + 1) * sizeof(float);
    if (o < red) o = red;
    p.total = o + 128;  // room to align the base
    return p;
}

}  // namespace

size_t dw_plane_smem_bytes(const DwPlaneArgs &a, int elem_bytes) { return dw_plane_layout(a, elem_bytes).total; }

template <int K, typename T>
__global__ void __launch_bounds__(kDwPlaneMaxThreads, (K <= 5 ? 2 : 1))
    wtconv_dw_plane_kernel(const __grid_constant__ DwPlaneArgs a) {
    constexpr int P = K / 2, KK = K * K, O = 4 - P, NR = 2 * KK + 1, NA = KK + 1;
    constexpr bool kConvert = sizeof(T) != 4;
    extern __shared__ __align__(128) float smem_raw[];
    __shared__ __align__(8) uint64_t bar[2];
    const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(smem_raw);
    char *base = reinterpret_cast<char *>(smem_raw) + (((s0 + 127u) & ~127u) - s0);
    const DwPlaneLayout lay = dw_plane_layout(a, (int)sizeof(T));
    float *Y1 = reinterpret_cast<float *>(base + lay.y1);
    float *G1 = reinterpret_cast<float *>(base + lay.g1);
    float *dslot = reinterpret_cast<float *>(base + lay.deep);
    const ShallowGeo &sg = a.sg;
    const Geo &dg = a.dg;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int L = a.L, TH = sg.TH, TW = sg.TW;
    const int yp = sg.ypitch;             // level-1 pitch (positions) of x's and dy's images
    const int l1img = 2 * a.y1rows * yp;  // floats per level-1 pair image

    // zero the level-1 and deeper images once: halos and rows no analysis writes read as zero
    {
        float4 *z = reinterpret_cast<float4 *>(Y1);
        const int nz = (int)((lay.end - lay.y1) / sizeof(float4));
        for (int i = tid; i < nz; i += nt) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_fence_init();
    }
    __syncthreads();

    // this thread's correlation image, item range per plane, and image pointers
    const int nimg = 1 + 2 * L;
    int ci = -1;
    for (int k = 0; k < nimg; ++k)
        if (tid >= a.tstart[k] && tid < a.tstart[k + 1]) ci = k;
    // items by slot: every item row has a multiple of 8 slots (those past the row's items idle),
    // so that the 8 threads of each quarter warp read neighbouring 16-byte columns of one item row
    // and never share banks across a row boundary
    int n_img = 0, icols = 8, ncols = 0, pitch = yp, pt = a.per_thread;
    const float *ybase = nullptr, *gbase = nullptr;
    if (ci == 0) {
        ncols = sg.items_c;
        icols = (ncols + 7) & ~7;
        n_img = sg.items_r * icols;
        pt = a.per_thread_base;
    } else if (ci > 0) {
        const int lvl = (ci - 1) / 2 + 1, pp = (ci - 1) & 1;
        ncols = dg.cstr[lvl];
        icols = (ncols + 7) & ~7;
        n_img = dg.rseg[lvl] * icols;
        if (lvl == 1) {
            ybase = Y1 + pp * l1img;
            gbase = G1 + pp * l1img + 2 * (P * yp + P);
        } else {
            pitch = dg.pitch[lvl];
            ybase = dslot + dg.off_y[lvl] + pp * dg.pimg[lvl];
            gbase = dslot + dg.off_g[lvl] + pp * dg.pimg[lvl] + 2 * (P * pitch + P);
        }
    }
    // items it_first, it_first + it_step, ... (< n_img): neighbouring threads take neighbouring
    // items at every step, so their window loads fall on neighbouring banks
    const int it_first = ci < 0 ? 0 : tid - a.tstart[ci];
    const int it_step = ci < 0 ? 1 : a.tstart[ci + 1] - a.tstart[ci];
    const int it_end = ci < 0 ? 0 : min(n_img, it_first + pt * it_step);

    // per-thread coordinates of the level-1 analysis loops (no division per element)
    const int ycols = sg.ycols, gw = TW / 2;
    const int a_rstep = ycols >= nt ? 1 : nt / ycols, a_thr = ycols >= nt ? nt : a_rstep * ycols;
    const int a_row0 = ycols >= nt ? 0 : tid / ycols, a_col0 = ycols >= nt ? tid : tid - a_row0 * ycols;
    const int g_rstep = gw >= nt ? 1 : nt / gw, g_thr = gw >= nt ? nt : g_rstep * gw;
    const int g_row0 = gw >= nt ? 0 : tid / gw, g_col0 = gw >= nt ? tid : tid - g_row0 * gw;
    const int y1_valid = TH / 2 + 2 * P;  // level-1 rows of x (with halo) the analysis writes

    f2_t acc[KK];
#pragma unroll
    for (int t = 0; t < KK; ++t) acc[t] = 0;
    float dysum = 0.f;

    const int b_begin = nbi * a.planes_per_cta;
    const int n_planes = min(a.B, b_begin + a.planes_per_cta) - b_begin;
    const int nbuf = a.nbuf == 2 ? 2 : 1;
    const uint32_t bytes = (uint32_t)((sg.xrows * sg.xw + TH * TW) * (int)sizeof(T));
    // plane k of this CTA goes to buffer k % nbuf; its barrier completes once per use of that buffer
    auto issue = [&](int k) {
        const int bf = k & (nbuf - 1);
        mbar_arrive_expect_tx(&bar[bf], bytes);
        tma_load_4d(base + (bf ? lay.rx[1] : lay.rx[0]), &a.tmap_x, -sg.padx, -2 * P, c, b_begin + k, &bar[bf]);
        tma_load_4d(base + (bf ? lay.rdy[1] : lay.rdy[0]), &a.tmap_dy, 0, 0, c, b_begin + k, &bar[bf]);
    };
    if (tid == 0 && n_planes > 0) issue(0);

    for (int k = 0; k < n_planes; ++k) {
        const int bf = k & (nbuf - 1);
        const uint32_t parity = (uint32_t)(nbuf == 2 ? k >> 1 : k) & 1u;
        // warp 0 waits for the copies, the others at the barrier; all leave together if the wait gave up
        const bool gave_up = tid < 32 && !mbar_wait(&bar[bf], parity, a.timeout);
        if (__syncthreads_or(gave_up)) {
            // the flag is raised: this CTA's partials become NaN (the gradients show it), and the
            // CTA leaves without touching the buffers a copy may still target
            const int ns = 1 + 4 * L;
            float *part = a.partials + ((size_t)nbi * a.C + c) * ns * NA;
            for (int i = tid; i < ns * NA; i += nt) part[i] = __int_as_float(0x7fc00000);
            return;
        }
        // the other buffer was last read before the barrier that ended the previous plane
        if (nbuf == 2 && tid == 0 && k + 1 < n_planes) issue(k + 1);
        float *X = reinterpret_cast<float *>(base + (bf ? lay.x[1] : lay.x[0]));
        float *DY = reinterpret_cast<float *>(base + (bf ? lay.dy[1] : lay.dy[0]));
        if constexpr (kConvert) {
            const T *rx = reinterpret_cast<const T *>(base + (bf ? lay.rx[1] : lay.rx[0]));
            const T *rdy = reinterpret_cast<const T *>(base + (bf ? lay.rdy[1] : lay.rdy[0]));
            // raw copies -> fp32 (loads first, then the stores)
            const int nx = sg.xbuf / 4, nd = TH * TW / 4;
            const uint2 *r2x = reinterpret_cast<const uint2 *>(rx), *r2d = reinterpret_cast<const uint2 *>(rdy);
            float4 *x4 = reinterpret_cast<float4 *>(X), *d4 = reinterpret_cast<float4 *>(DY);
            for (int i = tid; i < nx + nd; i += 2 * nt) {
                uint2 v[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int e = i + q * nt < nx + nd ? i + q * nt : i;
                    v[q] = e < nx ? r2x[e] : r2d[e - nx];
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int e = i + q * nt;
                    if (e < nx + nd) {
                        const float4 f = cvt4<T>(reinterpret_cast<const T *>(&v[q]));
                        if (e < nx) x4[e] = f;
                        else d4[e - nx] = f;
                    }
                }
            }
            __syncthreads();
        }
        // level 1 of x (interior + P positions of halo; X row 0 is image row -2P, X column padx
        // is image column 0) and of dy (interior) as padded subband-pair images
        if (tid < a_thr) {
            for (int col = a_col0; col < ycols; col += nt) {
                const float *xs = X + sg.padx - 2 * P + 2 * col + (2 * a_row0) * sg.xw;
                float *y0 = Y1 + 2 * (a_row0 * yp + col);
                for (int ya = a_row0; ya < y1_valid; ya += 4 * a_rstep) {
                    f2_t t0[4], t1[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float *xq = xs + (ya + q * a_rstep < y1_valid ? 2 * q * a_rstep * sg.xw : 0);
                        t0[q] = *reinterpret_cast<const f2_t *>(xq);
                        t1[q] = *reinterpret_cast<const f2_t *>(xq + sg.xw);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (ya + q * a_rstep < y1_valid) {
                            const f2_t sv = fadd2(t0[q], t1[q]), dv = fsub2(t0[q], t1[q]);
                            const float a0 = lo2(sv), a1 = hi2(sv), d0 = lo2(dv), d1 = hi2(dv);
                            float *yq = y0 + 2 * q * a_rstep * yp;
                            *reinterpret_cast<float2 *>(yq) = make_float2(a0 + a1, a0 - a1);
                            *reinterpret_cast<float2 *>(yq + l1img) = make_float2(d0 + d1, d0 - d1);
                        }
                    }
                    xs += 8 * a_rstep * sg.xw;
                    y0 += 8 * a_rstep * yp;
                }
            }
        }
        if (tid < g_thr) {
            for (int col = g_col0; col < gw; col += nt) {
                const float *ds = DY + 2 * col + (2 * g_row0) * TW;
                float *g0 = G1 + 2 * ((g_row0 + P) * yp + col + P);
                for (int ga = g_row0; ga < TH / 2; ga += 4 * g_rstep) {
                    f2_t t0[4], t1[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float *dq = ds + (ga + q * g_rstep < TH / 2 ? 2 * q * g_rstep * TW : 0);
                        t0[q] = *reinterpret_cast<const f2_t *>(dq);
                        t1[q] = *reinterpret_cast<const f2_t *>(dq + TW);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (ga + q * g_rstep < TH / 2) {
                            const f2_t sv = fadd2(t0[q], t1[q]), dv = fsub2(t0[q], t1[q]);
                            const float a0 = lo2(sv), a1 = hi2(sv), d0 = lo2(dv), d1 = hi2(dv);
                            float *gq = g0 + 2 * q * g_rstep * yp;
                            *reinterpret_cast<float2 *>(gq) = make_float2(a0 + a1, a0 - a1);
                            *reinterpret_cast<float2 *>(gq + l1img) = make_float2(d0 + d1, d0 - d1);
                        }
                    }
                    ds += 8 * g_rstep * TW;
                    g0 += 8 * g_rstep * yp;
                }
            }
        }
        __syncthreads();
        // levels >= 2 of both, two levels per pass: a thread reads a 4 x 4 block of level l-1's low
        // band (level 1: interior (i, j) at (i + P, j + P) of Y1 / G1) and writes four level-l quads
        // and one level-(l+1) quad; a last odd level takes a pass of its own on 2 x 2 blocks
        for (int l = 2; l <= L; l += 2) {
            const bool two = l + 1 <= L;
            const int ho = two ? dg.h[l + 1] : dg.h[l], wo = two ? dg.w[l + 1] : dg.w[l];
            for (int i = tid; i < 2 * ho * wo; i += nt) {
                const bool of_dy = i >= ho * wo;
                const int e = of_dy ? i - ho * wo : i;
                const int bi = e / wo, bj = e - bi * wo;
                const int *off = of_dy ? dg.off_g : dg.off_y;
                const float *l1 = of_dy ? G1 : Y1;
                auto ll = [&](int r, int cc) {  // level l-1 low band at interior (r, cc)
                    return l == 2 ? l1[2 * ((r + P) * yp + cc + P)] : get_ll(dslot, dg, off, l - 1, r, cc);
                };
                if (two) {
                    float v[4][4];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) v[r][cc] = ll(4 * bi + r, 4 * bj + cc);
                    Quad q[2][2];
#pragma unroll
                    for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                        for (int b2 = 0; b2 < 2; ++b2) {
                            q[a2][b2] = butterfly(v[2 * a2][2 * b2], v[2 * a2][2 * b2 + 1], v[2 * a2 + 1][2 * b2],
                                                  v[2 * a2 + 1][2 * b2 + 1]);
                            put_quad_pairs(dslot, dg, off, l, 2 * bi + a2, 2 * bj + b2, q[a2][b2]);
                        }
                    put_quad_pairs(dslot, dg, off, l + 1, bi, bj,
                                   butterfly(q[0][0].ll, q[0][1].ll, q[1][0].ll, q[1][1].ll));
                } else {
                    put_quad_pairs(dslot, dg, off, l, bi, bj,
                                   butterfly(ll(2 * bi, 2 * bj), ll(2 * bi, 2 * bj + 1), ll(2 * bi + 1, 2 * bj),
                                             ll(2 * bi + 1, 2 * bj + 1)));
                }
            }
            __syncthreads();
        }

        // this thread's share of its correlation for the plane
        if (ci == 0) {
            for (int it = it_first; it < it_end; it += it_step) {
                const int rs = it / icols, cs = it - rs * icols;
                if (cs >= ncols) continue;
                const float *xw = X + (kRows * rs + P) * sg.xw + kCols * cs + sg.padx - 4;
                const float *dw = DY + (kRows * rs) * TW + kCols * cs;
                f2_t gr[kRows][2];
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    const float4 d4v = *reinterpret_cast<const float4 *>(dw + j * TW);
                    gr[j][0] = pk2(d4v.x, d4v.y);
                    gr[j][1] = pk2(d4v.z, d4v.w);
                    dysum += (d4v.x + d4v.y) + (d4v.z + d4v.w);
                }
#pragma unroll
                for (int i = 0; i < kRows + K - 1; ++i) {
                    f2_t e[6], o[5];
                    load_row<3>(xw + i * sg.xw, e, o);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
#pragma unroll
                        for (int u = 0; u < K; ++u) {
                            const int j = i - u;
                            if (j >= 0 && j < kRows) {
#pragma unroll
                                for (int v = 0; v < K; ++v) {
                                    const int sc = O + v + 2 * q;  // window column of the pair's first x
                                    const f2_t xv = (sc & 1) ? o[(sc - 1) / 2] : e[sc / 2];
                                    ffma2_acc(acc[u * K + v], gr[j][q], xv);
                                }
                            }
                        }
                    }
                }
            }
        } else {
            for (int it = it_first; it < it_end; it += it_step) {
                const int rs = it / icols, cs = it - rs * icols;
                if (cs >= ncols) continue;
                const int off = 2 * ((rs * kRows) * pitch + cs * kColsL);
                dw_item_pair<K>(ybase + off, gbase + off, pitch, acc);
            }
        }
        __syncthreads();
        if (nbuf == 1 && tid == 0 && k + 1 < n_planes) issue(k + 1);  // the one buffer is free again
    }

    // reduce: per-thread tap sums -> one partial per (signal, tap), in thread order
    __syncthreads();
    float *red = reinterpret_cast<float *>(base);
#pragma unroll
    for (int t = 0; t < KK; ++t) {
        const float lo = lo2(acc[t]), hi = hi2(acc[t]);
        red[tid * NR + t] = ci == 0 ? lo + hi : lo;
        red[tid * NR + KK + t] = ci == 0 ? 0.f : hi;
    }
    red[tid * NR + 2 * KK] = dysum;
    __syncthreads();
    const int nsig = 1 + 4 * L;
    float *part = a.partials + ((size_t)nbi * a.C + c) * nsig * NA;
    for (int i = tid; i < nsig * NA; i += nt) {
        const int sig = i / NA, t = i - sig * NA;
        float s = 0.f;
        if (t < KK) {
            int cimg = 0, half = 0;
            if (sig > 0) {
                const int l = (sig - 1) / 4 + 1, sb = (sig - 1) & 3;
                cimg = 1 + 2 * (l - 1) + (sb >> 1);
                half = sb & 1;
            }
            for (int th = a.tstart[cimg]; th < a.tstart[cimg + 1]; ++th) s += red[th * NR + half * KK + t];
        } else if (sig == 0) {
            for (int th = a.tstart[0]; th < a.tstart[1]; ++th) s += red[th * NR + 2 * KK];
        }
        part[i] = s;
    }
}

template <int K, typename T>
static cudaError_t launch_dw_plane_t(const DwPlaneArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_dw_plane_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), (unsigned)a.nthreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_dw_plane_t(size_t smem, int nthreads) {
    auto kern = wtconv_dw_plane_kernel<K, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, nthreads, smem) != cudaSuccess) return 0;
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

cudaError_t launch_dw_plane(const DwPlaneArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_dw_plane_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_dw_plane(int dtype, int K, size_t smem, int nthreads) {
    WTCONV_DISPATCH(K, dtype, occ_dw_plane_t, smem, nthreads);
    return 0;
}

}  // namespace wtconv
