// Shallow kernel of the WTConv layer: the base conv and Haar level 1, tile by tile, writing the
// final outputs (forward y, or the input gradient dx with rotated kernels and no bias).
//
// Each CTA is one warp that owns channel c and walks a run of units (a unit is one output tile
// of G planes; G > 1 only when a tile covers a whole plane).  Per unit:
//   1. the input tile (output tile + 2P halo, zero outside the plane) arrives by cp.async in
//      chunks that never straddle the plane edge; fp32 tiles land directly in the conv layout X,
//      narrower types are converted into X by one elementwise pass (after which the raw buffer
//      takes the next unit's copy while this unit computes);
//   2. Haar level 1 of the tile (+ P coefficients of halo) is computed with butterflies and
//      stored as two subband-pair images (LL|LH, HL|HH);
//   3. every lane owns an 8 x 4 pixel output block and computes, in registers:
//        - the level-1 convs of its 4 x 2 coefficients for all four subbands (folded kernels,
//          packed f32x2 FMAs on subband pairs),
//        - their closed-form synthesis onto its 8 x 4 pixels, plus the contribution of the
//          deeper levels (precomputed at level-1 resolution by the deep kernel, staged with the
//          tile) and the bias,
//        - the base conv of its block (sliding window, packed f32x2 FMAs on column pairs)
//          accumulated on top of that,
//      and stores each output pixel once.
// The G planes of a unit are stacked vertically in X and in the pair images, so the per-unit
// loops index rows of one tall image.
#include "wtconv_items.cuh"

namespace wtconv {

// Shared memory: the raw tile buffer (type T; for fp32 it is X itself) and the deep tile (L >= 2),
// each starting 128-byte aligned (bulk tensor copies land there), then the X buffer (narrow types
// only), the pair images and the kernels.
size_t shallow_smem_bytes(const ShallowGeo &sg, int K, bool convert, bool deep) {
    size_t bytes = ((size_t)sg.raw_bytes + 127) / 128 * 128;
    if (deep) bytes += ((size_t)sg.G * sg.dtile * sizeof(float) + 127) / 128 * 128;
    if (convert) bytes += (size_t)sg.xbuf * sizeof(float);
    bytes += (size_t)sg.G * sg.pslot * sizeof(float);
    return bytes + (size_t)3 * wpairs(K) * sizeof(f2_t);
}

template <int K, typename T>
__global__ void __launch_bounds__(32, (K <= 5 ? 16 : 8)) wtconv_shallow_kernel(const __grid_constant__ ShallowArgs a) {
    constexpr int P = K / 2, WP = wpairs(K);
    constexpr bool kConvert = sizeof(T) != 4;  // narrow inputs are converted into an fp32 X tile
    extern __shared__ __align__(128) float smem[];
    __shared__ __align__(8) uint64_t bar_x, bar_d;  // bulk tensor copies of the input / deep tiles
    const ShallowGeo sg = a.sg;
    const int lane = threadIdx.x;
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = sg.G;
    const bool has_deep = a.deep != nullptr;
    // bulk tensor copies land at 128-byte aligned shared addresses (else the cp.async path runs)
    const bool smem128 = ((uint32_t)__cvta_generic_to_shared(smem) & 127u) == 0;
    const bool tma_x = a.tma_x != 0 && smem128, tma_d = has_deep && a.tma_d != 0 && smem128;
    char *raw_base = reinterpret_cast<char *>(smem);
    float *dtile = reinterpret_cast<float *>(raw_base + ((size_t)sg.raw_bytes + 127) / 128 * 128);
    float *xconv = dtile + (has_deep ? (G * sg.dtile + 31) / 32 * 32 : 0);  // narrow types only
    float *pairs = xconv + (kConvert ? sg.xbuf : 0);
    f2_t *wts = reinterpret_cast<f2_t *>(pairs + G * sg.pslot);
    if (lane == 0) {
        mbar_init(&bar_x, 1);
        mbar_init(&bar_d, 1);
        mbar_fence_init();
    }

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
    }
    const float bias = a.with_bias ? a.base_scale[c] * a.base_bias[c] : 0.f;
    __syncthreads();

    const T *x = static_cast<const T *>(a.x);
    T *out = static_cast<T *>(a.out);
    const int B = a.B, H = a.H, W = a.W, H1 = H >> 1, W1 = W >> 1;
    const size_t HW = (size_t)H * W, HW1 = (size_t)H1 * W1;
    const size_t cstride = (size_t)a.C * HW, cstride1 = (size_t)a.C * HW1;  // between batch entries
    const T *xc = x + (size_t)c * HW;
    const float *deepc = has_deep ? a.deep + (size_t)c * HW1 : nullptr;
    const int dtw = sg.TW / 2, dth = sg.TH / 2;
    const FastDiv fd_tiles = a.tiles, fd_tiles_c = a.tiles_c, fd_rrow = a.rchunks_row, fd_drow = a.dchunks_row;
    const int u_begin = nbi * a.units_per_cta;
    const int u_end = min(a.units, u_begin + a.units_per_cta);
    const bool vec_st = a.st_mode >= 1;

    // this lane's output item (at most one per unit by construction): fixed for the whole CTA
    const int per_tile_items = sg.items_r * sg.items_c;
    const bool has_item = lane < G * per_tile_items;
    const int ig = has_item ? lane / per_tile_items : 0;
    const int ie = lane - ig * per_tile_items;
    const int irs = has_item ? ie / sg.items_c : 0, ics = has_item ? ie - irs * sg.items_c : 0;
    const int x_item = (ig * sg.xrows + kRows * irs + P) * sg.xw + kCols * ics + sg.padx - 4;
    const int y_item = 2 * ((ig * sg.yrows + 4 * irs) * sg.ypitch + 2 * ics);
    const int d_item = ig * sg.dtile + (4 * irs) * dtw + 2 * ics;

    // lane layout of the copy and analysis loops: a lane keeps one column (chunk or position) and
    // walks rows with a fixed stride, so no index is divided per element
    const int nrow = (int)fd_rrow.d, ndrow = (int)fd_drow.d;
    const int r_rstep = nrow >= 32 ? 1 : 32 / nrow, r_lanes = nrow >= 32 ? 32 : r_rstep * nrow;
    const int r_row0 = nrow >= 32 ? 0 : lane / nrow, r_col = (nrow >= 32 ? lane : lane - r_row0 * nrow) * sg.chunk_e;
    const int n_rrows = G * sg.xrows;
    const int d_rstep = ndrow >= 32 ? 1 : 32 / ndrow, d_lanes = ndrow >= 32 ? 32 : d_rstep * ndrow;
    const int d_row0 = ndrow >= 32 ? 0 : lane / ndrow, d_col = (ndrow >= 32 ? lane : lane - d_row0 * ndrow) * sg.dchunk_e;
    const int n_drows = G * dth;
    const int ycols = sg.ycols;
    const int a_rstep = ycols >= 32 ? 1 : 32 / ycols, a_lanes = ycols >= 32 ? 32 : a_rstep * ycols;
    const int a_row0 = ycols >= 32 ? 0 : lane / ycols, a_col0 = ycols >= 32 ? lane : lane - a_row0 * ycols;
    const int n_arows = G * sg.yrows;

    // cp.async of unit u's raw input tiles; chunks outside the plane (or past the last batch
    // entry) are zero-filled without a read.  One commit group.
    auto issue_raw = [&](int u) {
        const int bg = (int)fdiv(fd_tiles, (uint32_t)u), t = u - bg * (int)fd_tiles.d;
        const int tr = (int)fdiv(fd_tiles_c, (uint32_t)t), tc = t - tr * sg.tiles_c;
        const int b0 = bg * G;
        const int rb = tr * sg.TH - 2 * P, cb = tc * sg.TW - sg.padx;
        if (tma_x) {  // one bulk tensor copy of the whole box; zero fill outside the tensor
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar_x, (uint32_t)(G * sg.xrows * sg.xw * (int)sizeof(T)));
                tma_load_4d(raw_base, &a.tmap_x, cb, rb, c, b0, &bar_x);
            }
            return;
        }
        T *raw = reinterpret_cast<T *>(raw_base);
        // lane -> fixed chunk column (several columns only for rows of more than 32 chunks); rows
        // advance by r_rstep (lanes past r_rstep * nrow idle)
        if (lane < r_lanes) {
            for (int cc = r_col; cc < sg.xw; cc += 32 * sg.chunk_e) {
                const int pc = cb + cc;
                const long long col_off = (long long)b0 * (long long)cstride + pc;  // + g planes + pr rows
                const bool col_ok = (unsigned)pc < (unsigned)W;
                T *dst = raw + r_row0 * sg.xw + cc;
                int g = 0, row = r_row0;  // row within plane g
#pragma unroll 4
                for (int rowg = r_row0; rowg < n_rrows; rowg += r_rstep) {
                    while (row >= sg.xrows) { row -= sg.xrows; ++g; }
                    const int pr = rb + row;
                    const bool ok = col_ok && (b0 + g) < B && (unsigned)pr < (unsigned)H;
                    const T *src = ok ? xc + (col_off + (long long)g * (long long)cstride + (long long)pr * W) : x;
                    if constexpr (sizeof(T) == 4) {
                        if (sg.chunk_e == 4) cp_async_n<16>(dst, src, ok ? 16 : 0);
                        else cp_async_n<8>(dst, src, ok ? 8 : 0);
                    } else {
                        if (sg.chunk_e == 8) cp_async_n<16>(dst, src, ok ? 16 : 0);
                        else if (sg.chunk_e == 4) cp_async_n<8>(dst, src, ok ? 8 : 0);
                        else cp_async_n<4>(dst, src, ok ? 4 : 0);
                    }
                    dst += r_rstep * sg.xw;
                    row += r_rstep;
                }
            }
        }
        cp_async_commit();
    };
    // cp.async of unit u's deep tiles (L >= 2).  One commit group.
    auto issue_deep = [&](int u) {
        if (!has_deep) return;
        const int bg = (int)fdiv(fd_tiles, (uint32_t)u), t = u - bg * (int)fd_tiles.d;
        const int tr = (int)fdiv(fd_tiles_c, (uint32_t)t), tc = t - tr * sg.tiles_c;
        const int b0 = bg * G;
        if (tma_d) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar_d, (uint32_t)(G * dth * dtw * (int)sizeof(float)));
                tma_load_4d(dtile, &a.tmap_d, tc * dtw, tr * dth, c, b0, &bar_d);
            }
            return;
        }
        if (lane < d_lanes) {
            float *dst = dtile + d_row0 * dtw + d_col;
            const int drb = tr * dth, dc = tc * dtw + d_col;
            const float *src_col = deepc + (size_t)b0 * cstride1 + dc;
            int g = 0, row = d_row0;
            for (int rowg = d_row0; rowg < n_drows; rowg += d_rstep) {
                while (row >= dth) { row -= dth; ++g; }
                const int dr = drb + row;
                const bool ok = (b0 + g) < B && dr < H1 && dc < W1;
                const float *src = ok ? src_col + (size_t)g * cstride1 + (size_t)dr * W1 : a.deep;
                if (sg.dchunk_e == 4) cp_async_n<16>(dst, src, ok ? 16 : 0);
                else cp_async_n<8>(dst, src, ok ? 8 : 0);
                dst += d_rstep * dtw;
                row += d_rstep;
            }
        }
        cp_async_commit();
    };

    // Single-buffered: the next unit's copies start as soon as their buffers are free (raw after
    // the conversion for narrow types, else after the items); the other warps resident on the SM
    // cover the copy latency.
    if (u_begin < u_end) {
        issue_raw(u_begin);
        issue_deep(u_begin);
    }
    for (int u = u_begin; u < u_end; ++u) {
        const int bg = (int)fdiv(fd_tiles, (uint32_t)u), t = u - bg * (int)fd_tiles.d;
        const int tr = (int)fdiv(fd_tiles_c, (uint32_t)t), tc = t - tr * sg.tiles_c;
        const int r0 = tr * sg.TH, c0 = tc * sg.TW;
        const int b0 = bg * G;

        // 1. this unit's tiles have landed
        const uint32_t parity = (uint32_t)(u - u_begin) & 1;
        cp_async_wait_all();
        // a wait that gave up raised the flag: this CTA's remaining outputs stay unwritten
        if (tma_x && !mbar_wait(&bar_x, parity, a.timeout)) return;
        if (tma_d && !mbar_wait(&bar_d, parity, a.timeout)) return;
        __syncthreads();
        const float *X;
        if constexpr (kConvert) {
            // raw -> X in batches of 4 groups per lane: loads first, then the stores (both are
            // shared memory, so an interleaved sequence would serialise on its latency)
            const uint2 *raw = reinterpret_cast<const uint2 *>(raw_base);
            float4 *x4 = reinterpret_cast<float4 *>(xconv);
            const int n4 = sg.xbuf / 4;
            for (int i = lane; i < n4; i += 4 * 32) {
                uint2 v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = raw[i + q * 32 < n4 ? i + q * 32 : i];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (i + q * 32 < n4) x4[i + q * 32] = cvt4<T>(reinterpret_cast<const T *>(&v[q]));
            }
            __syncthreads();
            if (u + 1 < u_end) issue_raw(u + 1);
            X = xconv;
        } else {
            X = reinterpret_cast<const float *>(raw_base);
        }

        // 2. Haar level 1 of the tile (unnormalised butterflies) -> pair images; row ya of the
        //    stacked images comes from X rows 2 ya and 2 ya + 1
        if (lane < a_lanes) {
            for (int col = a_col0; col < ycols; col += 32) {
                const float *xs = X + sg.padx - 2 * P + 2 * col + (2 * a_row0) * sg.xw;
                float *y0 = pairs + 2 * (a_row0 * sg.ypitch + col);
                // batches of kBatch positions: all loads first, then the butterflies and the
                // stores (X and the pair images are both shared memory, so an interleaved
                // load / store sequence would serialise on the shared-memory latency)
                constexpr int kBatch = 4;
                for (int ya = a_row0; ya < n_arows; ya += kBatch * a_rstep) {
                    f2_t t0[kBatch], t1[kBatch];
#pragma unroll
                    for (int q = 0; q < kBatch; ++q) {
                        const bool in = ya + q * a_rstep < n_arows;
                        const float *xq = xs + (in ? 2 * q * a_rstep * sg.xw : 0);
                        t0[q] = *reinterpret_cast<const f2_t *>(xq);
                        t1[q] = *reinterpret_cast<const f2_t *>(xq + sg.xw);
                    }
#pragma unroll
                    for (int q = 0; q < kBatch; ++q) {
                        if (ya + q * a_rstep < n_arows) {
                            // rows (a, b) and (c, d): s = (a+c, b+d), d = (a-c, b-d);
                            // LL = s.x + s.y, LH = s.x - s.y, HL = d.x + d.y, HH = d.x - d.y
                            const f2_t sv = fadd2(t0[q], t1[q]), dv = fsub2(t0[q], t1[q]);
                            const float s0 = lo2(sv), s1 = hi2(sv), d0 = lo2(dv), d1 = hi2(dv);
                            float *yq = y0 + 2 * q * a_rstep * sg.ypitch;
                            *reinterpret_cast<float2 *>(yq) = make_float2(s0 + s1, s0 - s1);
                            *reinterpret_cast<float2 *>(yq + G * sg.yimg) = make_float2(d0 + d1, d0 - d1);
                        }
                    }
                    xs += 2 * kBatch * a_rstep * sg.xw;
                    y0 += 2 * kBatch * a_rstep * sg.ypitch;
                }
            }
        }
        __syncthreads();

        // 3. this lane's fused output item: level-1 convs + synthesis + deep contribution + base conv
        if (has_item) {
            const int b = b0 + ig;
            const int pr = r0 + kRows * irs, pc = c0 + kCols * ics;  // block origin in the plane
            const float *dt = dtile + d_item;
            // start values of the base accumulators: deep contribution of levels >= 2 (constant over
            // each 2x2 pixel block) + bias, then the closed-form level-1 synthesis, folded in one
            // subband pair at a time: pixel (2i+a, 2q+b) += (LL + (-1)^b LH) + (-1)^a (HL + (-1)^b HH)
            f2_t init[kRows][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float d0 = 0.f, d1 = 0.f;
                if (has_deep) {
                    const float2 t2 = *reinterpret_cast<const float2 *>(dt + i * dtw);
                    d0 = t2.x;
                    d1 = t2.y;
                }
                init[2 * i][0] = init[2 * i + 1][0] = pk2(d0 + bias, d0 + bias);
                init[2 * i][1] = init[2 * i + 1][1] = pk2(d1 + bias, d1 + bias);
            }
            // one copy of the level-1 item code for both subband pairs (a smaller instruction
            // footprint); the pair's row sign (+1 for LL|LH, -1 for HL|HH) enters as an FMA factor
#pragma unroll 1
            for (int pp = 0; pp < 2; ++pp) {
                f2_t z[4][kColsL];
                level1_item<K>(pairs + y_item + pp * G * sg.yimg, sg.ypitch, wts + (1 + pp) * WP, z);
                const float sg1 = pp == 0 ? 1.f : -1.f;
                const f2_t sgn = pk2(sg1, sg1);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int q = 0; q < kColsL; ++q) {
                        const float s0 = lo2(z[i][q]), s1 = hi2(z[i][q]);
                        const f2_t sv = pk2(s0 + s1, s0 - s1);
                        init[2 * i][q] = fadd2(init[2 * i][q], sv);
                        init[2 * i + 1][q] = ffma2(sgn, sv, init[2 * i + 1][q]);
                    }
            }
            const int nrows = b < B ? max(0, min(kRows, H - pr)) : 0;
            const int ncols = max(0, min(kCols, W - pc));
            T *dst = out + (size_t)(b < B ? b : 0) * cstride + (size_t)c * HW + (size_t)pr * W + pc;
            base_item_store<K, T>(X + x_item, sg.xw, wts, init, dst, W, nrows, ncols, vec_st);
        }
        __syncthreads();
        if (u + 1 < u_end) {
            if constexpr (!kConvert) issue_raw(u + 1);
            issue_deep(u + 1);
        }
    }
    cp_async_wait_all();
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
