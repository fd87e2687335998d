// Shallow kernel of the WTConv layer: the base conv and Haar level 1, tile by tile, writing the
// final outputs (forward y, or the input gradient dx with rotated kernels and no bias).
//
// Each CTA is one warp that owns channel c and walks a run of tiles (or, for small planes, of
// groups of whole planes).  Per tile:
//   1. the zero-padded input tile X (output tile + 2P halo) is read once and converted to fp32;
//   2. Haar level 1 of the tile (+ P coefficients of halo) is computed on chip with butterflies
//      and stored as two subband-pair images (LL|LH, HL|HH);
//   3. every lane owns an 8 x 4 pixel output block and computes, in registers:
//        - the level-1 convs of its 4 x 2 coefficients for all four subbands (folded kernels,
//          packed f32x2 FMAs on subband pairs),
//        - their closed-form synthesis onto its 8 x 4 pixels, plus the contribution of the
//          deeper levels (precomputed at level-1 resolution by the deep kernel) and the bias,
//        - the base conv of its block (sliding window, packed f32x2 FMAs on column pairs)
//          accumulated on top of that,
//      and stores each output pixel once.
// No intermediate tensor reaches global memory except the deep contribution (N/4 floats).
#include "wtconv_device.cuh"

namespace wtconv {

// Shared memory: G plane slots ([X tile] + level-1 pair images; X lives in the raw buffer when a
// staged fp32 tile can be used as is), then two raw tile buffers and two deep tiles (staged
// path), then the kernels.
size_t shallow_smem_bytes(const ShallowGeo &sg, int K, bool stage, bool convert) {
    const size_t xfl = (size_t)round_up(sg.xrows * sg.xpitch, 4);
    const size_t pslot = (stage && !convert ? 0 : xfl) + 2 * (size_t)sg.yimg;
    size_t bytes = (size_t)sg.G * pslot * sizeof(float);
    if (stage) bytes += 2 * (size_t)sg.raw_bytes + 2 * (size_t)sg.G * sg.dtile * sizeof(float);
    return bytes + (size_t)3 * wpairs(K) * sizeof(f2_t);
}

// Level-1 pair images start after the X tile in a plane slot, unless X lives in the raw buffer.
__device__ __forceinline__ int yoff_fixed(bool x_in_raw, int xfl) { return x_in_raw ? 0 : xfl; }

__device__ __forceinline__ void cp_async8(void *smem_dst, const void *gmem_src, int src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(d), "l"(gmem_src), "r"(src_bytes) : "memory");
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
// out[r][c] = init[r][c] + sum_{u,v} w[u][v] * X[r + u][c + v] (X window origin at `in`).
template <int K, typename T>
__device__ __forceinline__ void base_item_store(const float *__restrict__ in, int pitch, const f2_t *wsm,
                                                const f2_t (&init)[kRows][2], T *dst, int ld, int nrows,
                                                int ncols, bool vec) {
    constexpr int NV = (kCols + K - 1 + 3) / 4;
    f2_t w[K * K];
    load_weights<K>(wsm, w);
    f2_t acc[kRows][2];
#pragma unroll
    for (int i = 0; i < kRows + K - 1; ++i) {
        f2_t e[2 * NV], o[2 * NV - 1];
        load_row<NV>(in + i * pitch, e, o);
#pragma unroll
        for (int v = 0; v < K; ++v) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < kRows) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const f2_t xv = (v & 1) ? o[q + v / 2] : e[q + v / 2];
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

template <int K, typename T>
__global__ void __launch_bounds__(32) wtconv_shallow_kernel(const ShallowArgs a) {
    constexpr int P = K / 2, WP = wpairs(K);
    constexpr bool kConvert = sizeof(T) != 4;  // narrow inputs are converted into an fp32 X tile
    constexpr int E = 8 / (int)sizeof(T);       // elements per 8-byte staged chunk
    extern __shared__ __align__(16) float smem[];
    const ShallowGeo &sg = a.sg;
    const int lane = threadIdx.x;
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = sg.G;
    const bool stage = a.stage != 0;
    const bool x_in_raw = stage && !kConvert;
    const int xfl = round_up(sg.xrows * sg.xpitch, 4);
    const int pslot = (x_in_raw ? 0 : xfl) + 2 * sg.yimg;  // floats per plane slot
    float *slots = smem;
    char *raw_base = reinterpret_cast<char *>(smem + (size_t)G * pslot);
    float *dtile_base = reinterpret_cast<float *>(raw_base + (stage ? 2 * sg.raw_bytes : 0));
    f2_t *wts = reinterpret_cast<f2_t *>(dtile_base + (stage ? 2 * G * sg.dtile : 0));

    // kernels, scales folded in: 0 base {w, w}; 1, 2 level-1 subband pairs {w_LL, w_LH}, {w_HL, w_HH}
    {
        constexpr int KK = K * K;
        for (int it = lane; it < 3 * KK; it += 32) {
            const int ci = it / KK, t = it - ci * KK;
            const int tu = t / K, tv = t - tu * K;
            const int src_t = a.flip ? (K - 1 - tu) * K + (K - 1 - tv) : t;
            float v0, v1;
            if (ci == 0) {
                v0 = v1 = a.base_scale[c] * a.base_w[(size_t)c * KK + src_t];
            } else {
                const size_t ch = (size_t)4 * c + 2 * (ci - 1);
                v0 = ldexpf(a.wavelet_scale[ch] * a.wavelet_w[ch * KK + src_t], -2);
                v1 = ldexpf(a.wavelet_scale[ch + 1] * a.wavelet_w[(ch + 1) * KK + src_t], -2);
            }
            wts[ci * WP + t] = pk2(v0, v1);
        }
        // zero the slots and the staging buffers once: padding columns that no copy writes stay zero
        float4 *s4 = reinterpret_cast<float4 *>(slots);
        const int nz = (int)((reinterpret_cast<char *>(wts) - reinterpret_cast<char *>(slots)) / 16);
        for (int i = lane; i < nz; i += 32) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float bias = a.with_bias ? a.base_scale[c] * a.base_bias[c] : 0.f;
    __syncthreads();

    const T *x = static_cast<const T *>(a.x);
    T *out = static_cast<T *>(a.out);
    const int H = a.H, W = a.W, H1 = H >> 1, W1 = W >> 1;
    const size_t HW = (size_t)H * W;
    const int nchunk = (sg.TW + 4 * P) / 4;  // 4-pixel chunks per X tile row (unstaged loads)
    const int per_tile_items = sg.items_r * sg.items_c;
    const bool vec_st = a.st_mode >= 1;
    const int dtw = sg.TW / 2;                 // deep tile row length

    const int u_begin = nbi * a.units_per_cta;
    const int u_end = min(a.units, u_begin + a.units_per_cta);

    // this lane's output item (at most one per tile by construction): fixed for the whole CTA
    const bool has_item = lane < G * per_tile_items;
    const int ig = has_item ? lane / per_tile_items : 0;
    const int ie = lane - ig * per_tile_items;
    const int irs = has_item ? ie / sg.items_c : 0, ics = has_item ? ie - irs * sg.items_c : 0;
    const int y_item = ig * pslot + yoff_fixed(x_in_raw, xfl) + 2 * ((4 * irs) * sg.ypitch + 2 * ics);
    const int x_item = (kRows * irs + P) * sg.xpitch + sg.pad_l + kCols * ics + P;
    const int d_item = ig * sg.dtile + (4 * irs) * dtw + 2 * ics;
    const int nrow = (int)a.rchunk_row.d;     // staged 8-byte chunks per raw tile row
    const int ndrow = (int)a.dchunk_row.d;    // staged 8-byte chunks per deep tile row

    // cp.async of unit u's raw input tiles and deep tiles into buffer `buf`; chunks outside the
    // plane are zero-filled (source size 0).  Lanes walk (row, chunk) with incremental indices.
    auto issue_stage = [&](int u, int buf) {
        const int bg = fdiv(a.tiles, u), t = u - bg * (int)a.tiles.d;
        const int tr = fdiv(a.tiles_c, t), tc = t - tr * sg.tiles_c;
        const int rb = tr * sg.TH - 2 * P, cb = tc * sg.TW - 2 * P;
        T *raw = reinterpret_cast<T *>(raw_base + buf * sg.raw_bytes) + sg.roff;
        for (int g = 0; g < G; ++g) {
            const int b = bg * G + g;
            const bool plane_ok = b < a.B;
            const T *src_plane = x + ((size_t)(plane_ok ? b : 0) * a.C + c) * HW;
            T *dst_plane = raw + (size_t)g * sg.xrows * sg.rpitch;
            int row = 0, m = lane;
            while (m >= nrow) { m -= nrow; ++row; }
            for (; row < sg.xrows;) {
                const int pr = rb + row, pc = cb + E * m;
                const bool in = plane_ok && (unsigned)pr < (unsigned)H && (unsigned)pc < (unsigned)W;
                cp_async8(dst_plane + row * sg.rpitch + E * m, in ? src_plane + (size_t)pr * W + pc : x, in ? 8 : 0);
                m += 32;
                while (m >= nrow) { m -= nrow; ++row; }
            }
        }
        if (a.deep != nullptr) {
            float *dt = dtile_base + buf * G * sg.dtile;
            const int drb = tr * (sg.TH >> 1), dcb = tc * (sg.TW >> 1);
            for (int g = 0; g < G; ++g) {
                const int b = bg * G + g;
                const bool plane_ok = b < a.B;
                const float *src_plane = a.deep + ((size_t)(plane_ok ? b : 0) * a.C + c) * H1 * W1;
                int i = 0, m = lane;
                while (m >= ndrow) { m -= ndrow; ++i; }
                for (; i < (sg.TH >> 1);) {
                    const int dr = drb + i, dc = dcb + 2 * m;
                    const bool in = plane_ok && dr < H1 && dc + 1 < W1;
                    cp_async8(dt + g * sg.dtile + i * dtw + 2 * m, in ? src_plane + (size_t)dr * W1 + dc : a.deep,
                              in ? 8 : 0);
                    m += 32;
                    while (m >= ndrow) { m -= ndrow; ++i; }
                }
            }
        }
        cp_async_commit();
    };

    if (stage && u_begin < u_end) issue_stage(u_begin, 0);
    int buf = 0;
    for (int u = u_begin; u < u_end; ++u, buf ^= 1) {
        const int bg = fdiv(a.tiles, u), t = u - bg * (int)a.tiles.d;
        const int tr = fdiv(a.tiles_c, t), tc = t - tr * sg.tiles_c;
        const int r0 = tr * sg.TH, c0 = tc * sg.TW;
        const int b0 = bg * G;

        // 1. input tiles (fp32 X, zero outside the plane)
        if (stage) {
            cp_async_wait_all();
            __syncthreads();
            if (u + 1 < u_end) issue_stage(u + 1, buf ^ 1);
            if constexpr (kConvert) {
                const T *raw = reinterpret_cast<const T *>(raw_base + buf * sg.raw_bytes);
                const int n = sg.TW + 4 * P;
                for (int g = 0; g < G; ++g) {
                    int row = 0, col = lane;
                    while (col >= n) { col -= n; ++row; }
                    for (; row < sg.xrows;) {
                        slots[g * pslot + row * sg.xpitch + sg.pad_l + col] =
                            Act<T>::ld(raw + ((size_t)g * sg.xrows + row) * sg.rpitch + col);
                        col += 32;
                        while (col >= n) { col -= n; ++row; }
                    }
                }
                __syncthreads();
            }
        } else {
            for (int it = lane; it < G * sg.xrows * nchunk; it += 32) {
                const int g = fdiv(a.xload, it), e = it - g * (int)a.xload.d;
                const int row = fdiv(a.xchunk, e), k = e - row * nchunk;
                const int b = b0 + g;
                const int pr = r0 - 2 * P + row, pc = c0 - 2 * P + 4 * k;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (b < a.B && pr >= 0 && pr < H) {
                    const T *src = x + ((size_t)b * a.C + c) * HW + (size_t)pr * W;
                    if (a.vec_ld && pc >= 0 && pc + 3 < W && (pc & 3) == 0) {
                        const float4 f = Act<T>::ld4(src + pc);
                        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (pc + q >= 0 && pc + q < W) v[q] = Act<T>::ld(src + pc + q);
                    }
                }
                float *X = slots + g * pslot + row * sg.xpitch + sg.pad_l + 4 * k;
#pragma unroll
                for (int q = 0; q < 4; ++q) X[q] = v[q];
            }
            __syncthreads();
        }
        const float *xtiles = x_in_raw ? reinterpret_cast<const float *>(raw_base + buf * sg.raw_bytes) : slots;
        const int xstride = x_in_raw ? sg.xrows * sg.rpitch : pslot;  // floats between planes' X tiles
        const int yoff = yoff_fixed(x_in_raw, xfl);                    // Y images within a plane slot

        // 2. Haar level 1 of the tile (unnormalised butterflies) -> pair images
        for (int g = 0; g < G; ++g) {
            const float *Xg = xtiles + g * xstride + sg.pad_l;
            float *Yg = slots + g * pslot + yoff;
            int ya = 0, yb = lane;
            while (yb >= sg.ycols) { yb -= sg.ycols; ++ya; }
            for (; ya < sg.yrows;) {
                const float *X = Xg + (2 * ya) * sg.xpitch + 2 * yb;
                float p, q, r, s;
                if constexpr ((P & 1) == 0) {
                    const float2 t0 = *reinterpret_cast<const float2 *>(X);
                    const float2 t1 = *reinterpret_cast<const float2 *>(X + sg.xpitch);
                    p = t0.x; q = t0.y; r = t1.x; s = t1.y;
                } else {
                    p = X[0]; q = X[1]; r = X[sg.xpitch]; s = X[sg.xpitch + 1];
                }
                const Quad qd = butterfly(p, q, r, s);
                float *y0 = Yg + 2 * (ya * sg.ypitch + yb);
                *reinterpret_cast<float2 *>(y0) = make_float2(qd.ll, qd.lh);
                *reinterpret_cast<float2 *>(y0 + sg.yimg) = make_float2(qd.hl, qd.hh);
                yb += 32;
                while (yb >= sg.ycols) { yb -= sg.ycols; ++ya; }
            }
        }
        __syncthreads();

        // 3. this lane's fused output item: level-1 convs + synthesis + deep contribution + base conv
        if (has_item) {
            const int b = b0 + ig;
            const int pr = r0 + kRows * irs, pc = c0 + kCols * ics;  // block origin in the plane
            const float *dtiles = dtile_base + buf * G * sg.dtile;
            // start values of the base accumulators: deep contribution of levels >= 2 (constant over
            // each 2x2 pixel block) + bias, then the closed-form level-1 synthesis, folded in one
            // subband pair at a time: pixel (2i+a, 2q+b) += (LL + (-1)^b LH) + (-1)^a (HL + (-1)^b HH)
            f2_t init[kRows][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float d0 = 0.f, d1 = 0.f;
                if (a.deep != nullptr) {
                    if (stage) {
                        const float2 t2 = *reinterpret_cast<const float2 *>(dtiles + d_item + i * dtw);
                        d0 = t2.x;
                        d1 = t2.y;
                    } else if (b < a.B) {
                        const int dr = (pr >> 1) + i, dc = pc >> 1;
                        const float *dp = a.deep + ((size_t)b * a.C + c) * H1 * W1;
                        if (dr < H1 && dc + 1 < W1) {
                            const float2 t2 = *reinterpret_cast<const float2 *>(dp + (size_t)dr * W1 + dc);
                            d0 = t2.x;
                            d1 = t2.y;
                        } else if (dr < H1 && dc < W1) {
                            d0 = dp[(size_t)dr * W1 + dc];
                        }
                    }
                }
                init[2 * i][0] = init[2 * i + 1][0] = pk2(d0 + bias, d0 + bias);
                init[2 * i][1] = init[2 * i + 1][1] = pk2(d1 + bias, d1 + bias);
            }
#pragma unroll
            for (int pp = 0; pp < 2; ++pp) {
                f2_t z[4][kColsL];
                level1_item<K>(slots + y_item + pp * sg.yimg, sg.ypitch, wts + (1 + pp) * WP, z);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int q = 0; q < kColsL; ++q) {
                        const float s0 = lo2(z[i][q]), s1 = hi2(z[i][q]);
                        const f2_t sv = pk2(s0 + s1, s0 - s1);
                        init[2 * i][q] = fadd2(init[2 * i][q], sv);
                        init[2 * i + 1][q] = pp == 0 ? fadd2(init[2 * i + 1][q], sv) : fsub2(init[2 * i + 1][q], sv);
                    }
            }
            const int nrows = b < a.B ? max(0, min(kRows, H - pr)) : 0;
            const int ncols = max(0, min(kCols, W - pc));
            T *dst = out + ((size_t)(b < a.B ? b : 0) * a.C + c) * HW + (size_t)pr * W + pc;
            base_item_store<K, T>(xtiles + ig * xstride + x_item, sg.xpitch, wts, init, dst, W, nrows, ncols, vec_st);
        }
        __syncthreads();
    }
}

template <int K, typename T>
static cudaError_t launch_shallow_t(const ShallowArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_shallow_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), 32, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_shallow_t(size_t smem) {
    auto kern = wtconv_shallow_kernel<K, T>;
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

cudaError_t launch_shallow(const ShallowArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_shallow_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_shallow(int dtype, int K, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_shallow_t, smem);
    return 0;
}

}  // namespace wtconv
