// Fused whole-plane kernel of the WTConv layer (forward y, or the input gradient dx with rotated
// kernels and no bias) for planes whose pyramid fits in shared memory.
//
// A CTA of kPlaneThreads threads owns channel c and a run of batch entries, one plane at a time:
//   1. one bulk tensor copy brings the plane with a 2P halo (zero outside) into the conv layout X;
//   2. Haar level 1 of the plane (+ P coefficients of halo) is computed as two subband-pair
//      images (LL|LH, HL|HH); levels >= 2 are built from the level-1 low band on chip, each
//      level's subbands as pair images with a zero halo;
//   3. the levels >= 2 run their subband-pair conv items (folded kernels, packed f32x2 FMAs,
//      kPlaneDeepRows rows per item);
//   4. their closed-form synthesis is gathered at level-1 resolution into D (shared memory);
//   5. every thread owns 8 x 4 pixel output blocks and computes, in registers, the level-1 convs
//      of its 4 x 2 coefficients, their synthesis onto its pixels, D and the bias, and the base
//      conv on top, and stores each output pixel once.
// x is read once from HBM and y written once; nothing else leaves the chip.
#include "wtconv_items.cuh"

namespace wtconv {

namespace {

__host__ __device__ inline size_t round128(size_t b) { return (b + 127) / 128 * 128; }

// Shared-memory layout (floats from a 128-byte aligned base): X (raw copy for fp32), raw copy
// (narrow types), level-1 pairs, levels >= 2 slot, D, kernels.
struct PlaneLayout {
    size_t x, raw, pairs, deep, d, wts, total_bytes;
};

__host__ __device__ inline PlaneLayout plane_layout(const PlaneArgs &a, int elem_bytes) {
    PlaneLayout p;
    const ShallowGeo &sg = a.sg;
    size_t o = 0;  // bytes
    p.x = o;
    o += round128((size_t)sg.xbuf * sizeof(float));
    p.raw = o;
    if (elem_bytes != 4) o += round128((size_t)sg.raw_bytes);
    p.pairs = o;
    o += (size_t)sg.pslot * sizeof(float);
    p.deep = o;
    o += (a.L >= 2 ? (size_t)a.dg.slot_floats : 0) * sizeof(float);
    p.d = o;
    o += (size_t)(sg.TH / 2) * a.dpitch * sizeof(float);
    p.wts = (o + 15) / 16 * 16;
    o = p.wts + (size_t)(1 + 2 * a.L) * wpairs(a.K) * sizeof(f2_t);
    p.total_bytes = o + 128;  // room to align the base
    return p;
}

// Conv item of kPlaneDeepRows x kColsL positions on a subband-pair image of a level >= 2:
// out[r][c] = sum_{u,v} w[u][v] * in[r + u][c + v] elementwise on the two subbands; `in` points at
// the padded window origin, `out` at the compact pair output; pitches in positions.  Shorter than
// the 8-row items of level 1 so that more threads share the small deep images.
template <int K>
__device__ __forceinline__ void deep_item(const float *__restrict__ in, int pitch, const f2_t (&w)[K * K],
                                          float *__restrict__ out, int opitch) {
    constexpr int R = kPlaneDeepRows, NV = (kColsL + K - 1 + 1) / 2;
    f2_t acc[R][kColsL];
#pragma unroll
    for (int i = 0; i < R + K - 1; ++i) {
        f2_t x[2 * NV];
        load_pair_row<NV>(in + 2 * i * pitch, x);
#pragma unroll
        for (int v = 0; v < K; ++v) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < R) {
#pragma unroll
                    for (int q = 0; q < kColsL; ++q) {
                        if (u == 0 && v == 0) acc[j][q] = fmul2(w[0], x[q]);
                        else ffma2_acc(acc[j][q], w[u * K + v], x[q + v]);
                    }
                }
            }
        }
        const int jd = i - (K - 1);
        if (jd >= 0) {
            ulonglong2 t;
            t.x = acc[jd][0];
            t.y = acc[jd][1];
            *reinterpret_cast<ulonglong2 *>(out + 2 * jd * opitch) = t;
        }
    }
}

}  // namespace

size_t plane_smem_bytes(const PlaneArgs &a, int elem_bytes) { return plane_layout(a, elem_bytes).total_bytes; }

template <int K, typename T>
__global__ void __launch_bounds__(kPlaneThreads, (K <= 5 ? 4 : 2)) wtconv_plane_kernel(const __grid_constant__ PlaneArgs a) {
    constexpr int P = K / 2, WP = wpairs(K), KK = K * K;
    constexpr bool kConvert = sizeof(T) != 4;
    extern __shared__ __align__(128) float smem_raw[];
    __shared__ __align__(8) uint64_t bar;
    const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(smem_raw);
    char *base = reinterpret_cast<char *>(smem_raw) + (((s0 + 127u) & ~127u) - s0);
    const PlaneLayout lay = plane_layout(a, (int)sizeof(T));
    float *X = reinterpret_cast<float *>(base + lay.x);
    T *raw = kConvert ? reinterpret_cast<T *>(base + lay.raw) : reinterpret_cast<T *>(X);
    float *pairs = reinterpret_cast<float *>(base + lay.pairs);
    float *dslot = reinterpret_cast<float *>(base + lay.deep);
    float *D = reinterpret_cast<float *>(base + lay.d);
    f2_t *wts = reinterpret_cast<f2_t *>(base + lay.wts);
    const ShallowGeo &sg = a.sg;
    const Geo &dg = a.dg;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int L = a.L, H = a.H, W = a.W, H1 = H >> 1, W1 = W >> 1;

    // kernels, scales folded in: 0 base {w, w}; 1 + 2(l-1) + pp level l subband pair pp
    for (int it = tid; it < (1 + 2 * L) * KK; it += nt) {
        const int ci = it / KK, t = it - ci * KK;
        const int tu = t / K, tv = t - tu * K;
        const int src_t = a.flip ? (K - 1 - tu) * K + (K - 1 - tv) : t;
        float v0, v1;
        if (ci == 0) {
            v0 = v1 = a.base_scale[c] * a.base_w[(size_t)c * KK + src_t];
        } else {
            const int l = (ci - 1) / 2 + 1, pp = (ci - 1) & 1;
            const size_t ch = (size_t)(l - 1) * 4 * a.C + 4 * c + 2 * pp;
            v0 = ldexpf(a.wavelet_scale[ch] * a.wavelet_w[ch * KK + src_t], -2 * l);
            v1 = ldexpf(a.wavelet_scale[ch + 1] * a.wavelet_w[(ch + 1) * KK + src_t], -2 * l);
        }
        wts[ci * WP + t] = pk2(v0, v1);
    }
    // zero the levels >= 2 slot (its halos must stay zero) and D (rows / columns past the plane)
    {
        float *z0 = dslot;
        const int nz = (int)((lay.wts - lay.deep) / sizeof(float));
        for (int i = tid; i < nz; i += nt) z0[i] = 0.f;
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();

    const int b_begin = nbi * a.planes_per_cta;
    const int b_end = min(a.B, b_begin + a.planes_per_cta);
    const uint32_t bytes = (uint32_t)(sg.xrows * sg.xw * (int)sizeof(T));
    if (tid == 0 && b_begin < b_end) {
        mbar_arrive_expect_tx(&bar, bytes);
        tma_load_4d(raw, &a.tmap_x, -sg.padx, -2 * P, c, b_begin, &bar);
    }
    T *out = static_cast<T *>(a.out);
    const size_t HW = (size_t)H * W;
    const float bias = a.with_bias ? a.base_scale[c] * a.base_bias[c] : 0.f;
    const bool vec_st = a.st_mode >= 1;
    // output items by slot: every item row has a multiple of 8 slots (those past the row's items
    // idle), so that the 8 threads of each quarter warp read neighbouring 16-byte columns of one
    // item row and never share banks across a row boundary
    const int fused_cpad = (sg.items_c + 7) & ~7;
    const int n_fused = sg.items_r * fused_cpad;
    // per-thread coordinates of the analysis loops (computed once: no division per element)
    const int a_rstep = sg.ycols >= nt ? 1 : nt / sg.ycols;
    const int a_threads = sg.ycols >= nt ? nt : a_rstep * sg.ycols;
    const int a_row0 = sg.ycols >= nt ? 0 : tid / sg.ycols, a_col0 = sg.ycols >= nt ? tid : tid - a_row0 * sg.ycols;
    const int w2c = L >= 2 ? a.dg.w[2] : 1;  // level-2 positions: thread tid starts at (tid / w2, tid % w2)
    const int l2_row0 = tid / w2c, l2_col0 = tid - l2_row0 * w2c;
    const int l2_drow = nt / w2c, l2_dcol = nt - l2_drow * w2c;

    for (int b = b_begin; b < b_end; ++b) {
        // thread 0 waits for the copy, the others at the barrier; all leave together if it gave
        // up (the flag is raised and this CTA's remaining outputs stay unwritten)
        const bool gave_up = tid == 0 && !mbar_wait(&bar, (uint32_t)(b - b_begin) & 1, a.timeout);
        if (__syncthreads_or(gave_up)) return;
        if constexpr (kConvert) {
            const uint2 *r2 = reinterpret_cast<const uint2 *>(raw);
            float4 *x4 = reinterpret_cast<float4 *>(X);
            const int n4 = sg.xbuf / 4;
            for (int i = tid; i < n4; i += 4 * nt) {
                uint2 v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = r2[i + q * nt < n4 ? i + q * nt : i];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (i + q * nt < n4) x4[i + q * nt] = cvt4<T>(reinterpret_cast<const T *>(&v[q]));
            }
            __syncthreads();
        }
        // level 1 (+ halo) -> pair images: position (ya, yb) from X rows 2 ya, 2 ya + 1; a thread
        // keeps one column and walks rows (loads of four rows first, then the stores)
        if (tid < a_threads) {
            for (int col = a_col0; col < sg.ycols; col += nt) {
                const float *xs = X + sg.padx - 2 * P + 2 * col + (2 * a_row0) * sg.xw;
                float *y0 = pairs + 2 * (a_row0 * sg.ypitch + col);
                for (int ya = a_row0; ya < sg.yrows; ya += 4 * a_rstep) {
                    f2_t t0[4], t1[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const bool in = ya + q * a_rstep < sg.yrows;
                        const float *xq = xs + (in ? 2 * q * a_rstep * sg.xw : 0);
                        t0[q] = *reinterpret_cast<const f2_t *>(xq);
                        t1[q] = *reinterpret_cast<const f2_t *>(xq + sg.xw);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (ya + q * a_rstep < sg.yrows) {
                            const f2_t sv = fadd2(t0[q], t1[q]), dv = fsub2(t0[q], t1[q]);
                            const float a0 = lo2(sv), a1 = hi2(sv), d0 = lo2(dv), d1 = hi2(dv);
                            float *yq = y0 + 2 * q * a_rstep * sg.ypitch;
                            *reinterpret_cast<float2 *>(yq) = make_float2(a0 + a1, a0 - a1);
                            *reinterpret_cast<float2 *>(yq + sg.yimg) = make_float2(d0 + d1, d0 - d1);
                        }
                    }
                    xs += 8 * a_rstep * sg.xw;
                    y0 += 8 * a_rstep * sg.ypitch;
                }
            }
        }
        __syncthreads();
        if (L >= 2) {
            // levels >= 2 from the level-1 low band (pair image 0, even floats; interior position
            // (i, j) of level 1 sits at (i + P, j + P)).  L = 2: one pass over the level-2
            // positions; L >= 3: two levels per pass, a thread reading a 4 x 4 block of the finer
            // low band and writing four quads of level l and one of level l + 1
            if (L == 2) {
                const int h2 = dg.h[2], w2 = dg.w[2];
                for (int bi = l2_row0, bj = l2_col0; bi < h2; ) {
                    const float *l1 = pairs + 2 * ((2 * bi + P) * sg.ypitch + 2 * bj + P);
                    const Quad q = butterfly(l1[0], l1[2], l1[2 * sg.ypitch], l1[2 * sg.ypitch + 2]);
                    put_quad_pairs(dslot, dg, dg.off_y, 2, bi, bj, q);
                    bj += l2_dcol;
                    bi += l2_drow;
                    if (bj >= w2) { bj -= w2; ++bi; }
                }
                __syncthreads();
            }
            for (int l = 2; L >= 3 && l <= L; l += 2) {
                const bool two = l + 1 <= L;
                const int ho = two ? dg.h[l + 1] : dg.h[l], wo = two ? dg.w[l + 1] : dg.w[l];
                for (int i = tid; i < ho * wo; i += nt) {
                    const int bi = i / wo, bj = i - bi * wo;
                    auto ll = [&](int r, int cc) {  // level l-1 low band at interior (r, cc)
                        return l == 2 ? pairs[2 * ((r + P) * sg.ypitch + cc + P)]
                                      : get_ll(dslot, dg, dg.off_y, l - 1, r, cc);
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
                                put_quad_pairs(dslot, dg, dg.off_y, l, 2 * bi + a2, 2 * bj + b2, q[a2][b2]);
                            }
                        put_quad_pairs(dslot, dg, dg.off_y, l + 1, bi, bj,
                                       butterfly(q[0][0].ll, q[0][1].ll, q[1][0].ll, q[1][1].ll));
                    } else {
                        put_quad_pairs(dslot, dg, dg.off_y, l, bi, bj,
                                       butterfly(ll(2 * bi, 2 * bj), ll(2 * bi, 2 * bj + 1), ll(2 * bi + 1, 2 * bj),
                                                 ll(2 * bi + 1, 2 * bj + 1)));
                    }
                }
                __syncthreads();
            }
            // conv items of every level >= 2 subband-pair image
            for (int it = tid; it < a.n_deep_items; it += nt) {
                int ci = 3;
                while (it >= a.deep_item_start[ci + 1]) ++ci;
                const int l = (ci - 1) / 2 + 1, pp = (ci - 1) & 1;
                const int e = it - a.deep_item_start[ci];
                const int cpad = (dg.cstr[l] + 7) & ~7;  // slots per item row, as for the output items
                const int rs = e / cpad, cs = e - rs * cpad;
                if (cs >= dg.cstr[l]) continue;
                f2_t w[KK];
                load_weights<K>(wts + ci * WP, w);
                const int r0 = rs * kPlaneDeepRows;
                deep_item<K>(dslot + dg.off_y[l] + pp * dg.pimg[l] + 2 * (r0 * dg.pitch[l] + cs * kColsL), dg.pitch[l], w,
                             dslot + dg.off_z[l] + pp * dg.zimg[l] + 2 * (r0 * dg.zpitch[l] + cs * kColsL),
                             dg.zpitch[l]);
            }
            __syncthreads();
            // their synthesis at level-1 resolution -> D
            const int nws = (W1 + 7) / 8;
            for (int it = tid; it < H1 * nws; it += nt) {
                const int i = it / nws, ws = it - i * nws;
                const int j0 = ws * 8;
                float dv[8];
                deep_gather8(dg, dslot, i, j0, dv);
                float *drow = D + i * a.dpitch + j0;
                const int nv = min(8, W1 - j0);
                for (int q = 0; q < nv; ++q) drow[q] = dv[q];
            }
        }
        __syncthreads();
        // fused output items
        for (int it = tid; it < n_fused; it += nt) {
            const int irs = it / fused_cpad, ics = it - irs * fused_cpad;
            if (ics >= sg.items_c) continue;
            const int pr = kRows * irs, pc = kCols * ics;
            f2_t init[kRows][2];
            const float *dt = D + (4 * irs) * a.dpitch + 2 * ics;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 t2 = *reinterpret_cast<const float2 *>(dt + i * a.dpitch);
                init[2 * i][0] = init[2 * i + 1][0] = pk2(t2.x + bias, t2.x + bias);
                init[2 * i][1] = init[2 * i + 1][1] = pk2(t2.y + bias, t2.y + bias);
            }
            const int y_item = 2 * ((4 * irs) * sg.ypitch + 2 * ics);
#pragma unroll 1
            for (int pp = 0; pp < 2; ++pp) {
                f2_t z[4][kColsL];
                level1_item<K>(pairs + y_item + pp * sg.yimg, sg.ypitch, wts + (1 + pp) * WP, z);
                const float sg1 = pp == 0 ? 1.f : -1.f;
                const f2_t sgn = pk2(sg1, sg1);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int q = 0; q < kColsL; ++q) {
                        const float z0 = lo2(z[i][q]), z1 = hi2(z[i][q]);
                        const f2_t sv = pk2(z0 + z1, z0 - z1);
                        init[2 * i][q] = fadd2(init[2 * i][q], sv);
                        init[2 * i + 1][q] = ffma2(sgn, sv, init[2 * i + 1][q]);
                    }
            }
            const int nrows = max(0, min(kRows, H - pr));
            const int ncols = max(0, min(kCols, W - pc));
            T *dst = out + ((size_t)b * a.C + c) * HW + (size_t)pr * W + pc;
            const int x_item = (kRows * irs + P) * sg.xw + kCols * ics + sg.padx - 4;
            base_item_store<K, T>(X + x_item, sg.xw, wts, init, dst, W, nrows, ncols, vec_st);
        }
        __syncthreads();
        if (tid == 0 && b + 1 < b_end) {  // X is free: the next plane's copy
            mbar_arrive_expect_tx(&bar, bytes);
            tma_load_4d(raw, &a.tmap_x, -sg.padx, -2 * P, c, b + 1, &bar);
        }
    }
}

template <int K, typename T>
static cudaError_t launch_plane_t(const PlaneArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_plane_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), kPlaneThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_plane_t(size_t smem) {
    auto kern = wtconv_plane_kernel<K, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kPlaneThreads, smem) != cudaSuccess) return 0;
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

cudaError_t launch_plane(const PlaneArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_plane_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_plane(int dtype, int K, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_plane_t, smem);
    return 0;
}

}  // namespace wtconv
