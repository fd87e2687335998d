// Tiled batch-pair shallow kernel of the WTConv forward / input gradient (paper, Resumo Tecnico /
// Metodologia: the Haar butterflies recomputed on chip from one read of the input, the learned
// scales folded into the conv weights, the multi-level synthesis as one closed-form pass):
//     y[h, w] = s_b (conv(x, w_b) + b_b)[h, w]
//             + sum_s sigma_s(h & 1, w & 1) Z^1_s[h >> 1, w >> 1] + D[h >> 1, w >> 1]
// with Z^1_s = conv(Yhat^1_s, 4^-1 s_1 w_1) on the unnormalised level-1 subbands and D the levels
// >= 2 at level-1 resolution, computed before by the deep kernel (constant over each 2 x 2 block,
// so it enters with the low band).  The input gradient is the same operator on dy with every kernel
// rotated by 180 degrees and no bias.
//
// Persistent CTAs walk work items (channel, tile, group of G batch pairs), channel-major.  Per item
// one thread issues two bulk tensor copies: the x tile of 2G planes with a halo of 2P (zero outside
// the plane; P for the base conv, P level-1 positions for the level-1 conv) and the D tile.  Pass 1
// builds, as batch-pair images (two batch entries per packed fp32 pair), the padded x copy X and
// the four level-1 subbands from 2 x 2 blocks, and packs D.  Level-1 conv items write Z^1; output
// items run the base conv, add the synthesis and D, and store each pixel once.  The next item's
// copies run during this item's work.
#pragma once

#include "wtconv_pair_fwd.cuh"
#include "wtconv_pshallow.h"

namespace wtconv {

namespace {

struct PsLayout {
    size_t raw_x, raw_d, slots, wts, total;  // byte offsets from a 128-byte aligned base
};

__host__ __device__ inline size_t ps_round128(size_t b) { return (b + 127) / 128 * 128; }

// Raw x tiles and raw D tiles (bulk copy destinations), the G pair slots, the channel's five
// kernels (base, then level-1 subbands LL, LH, HL, HH) as duplicated pairs.
__host__ __device__ inline PsLayout pshallow_layout(const PsArgs &a) {
    PsLayout p;
    size_t o = 0;
    p.raw_x = o;
    o += (size_t)a.raw_x_bytes;
    p.raw_d = o;
    o += (size_t)a.raw_d_bytes;
    p.slots = o;
    o += ps_round128((size_t)a.G * a.slot * sizeof(f2_t));
    p.wts = o;
    o += (size_t)5 * wpairs(a.K) * sizeof(f2_t);
    p.total = o + 128;
    return p;
}

// Channel c's base kernel s_b w_b and level-1 kernels 4^-1 s_1[4c+s] w_1[4c+s] as {w, w} pairs
// (rotated by 180 degrees for the input gradient).
template <int K>
__device__ __forceinline__ void ps_stage_weights(const PsArgs &a, int c, f2_t *wts) {
    constexpr int KK = K * K, WP = wpairs(K);
    for (int it = threadIdx.x; it < 5 * KK; it += blockDim.x) {
        const int ci = it / KK, t = it - ci * KK;
        const int src_t = a.flip ? KK - 1 - t : t;
        float v;
        if (ci == 0) {
            v = a.base_scale[c] * a.base_w[(size_t)c * KK + src_t];
        } else {
            const size_t ch = (size_t)4 * c + (ci - 1);
            v = 0.25f * a.wavelet_scale[ch] * a.wavelet_w[ch * KK + src_t];
        }
        wts[ci * WP + t] = pk2(v, v);
    }
}

}  // namespace

template <int K, typename T, int NT, int S>
__global__ void __launch_bounds__(NT, (K <= 5 ? 512 : 384) / NT) wtconv_pshallow_kernel(const __grid_constant__ PsArgs a) {
    constexpr int P = K / 2, KK = K * K, WP = wpairs(K);
    extern __shared__ __align__(128) unsigned char ps_smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int copy_ok;
    const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(ps_smem);
    unsigned char *base = ps_smem + (((s0 + 127u) & ~127u) - s0);
    const PsLayout lay = pshallow_layout(a);
    T *raw_x = reinterpret_cast<T *>(base + lay.raw_x);
    float *raw_d = reinterpret_cast<float *>(base + lay.raw_d);
    f2_t *slots = reinterpret_cast<f2_t *>(base + lay.slots);
    f2_t *wts = reinterpret_cast<f2_t *>(base + lay.wts);
    const int tid = threadIdx.x;
    const int B = a.B, C = a.C, H = a.H, W = a.W, G = a.G, TH = a.TH, TW = a.TW, HX = a.HX, HXL = a.HXL;
    const int RXR = a.RXR, RXW = a.RXW, TH1 = TH / 2, TW1 = TW / 2;
    const size_t HW = (size_t)H * W;

    {   // every slot starts at zero: the halos, the rounding rows and columns and (without deeper
        // levels) the D image stay zero
        ulonglong2 *z = reinterpret_cast<ulonglong2 *>(slots);
        const int nz = G * a.slot / 2;
        for (int i = tid; i < nz; i += NT) z[i] = make_ulonglong2(0ull, 0ull);
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();

    const int w0 = (int)((long long)blockIdx.x * a.work / a.grid);
    const int w1 = (int)((long long)(blockIdx.x + 1) * a.work / a.grid);
    const int per_c = (int)a.dv_work_c.d;  // work items per channel: ngroups * tiles
    const uint32_t box_x = (uint32_t)(2 * G * RXR * RXW * (int)sizeof(T));
    const uint32_t box_d = a.has_deep ? (uint32_t)(2 * G * TH1 * TW1 * (int)sizeof(float)) : 0u;
    // work item w -> channel, tile row / column, first pair
    auto decode = [&](int w, int &c, int &tr, int &tc, int &p0) {
        c = (int)fdiv(a.dv_work_c, (uint32_t)w);
        const int rem = w - c * per_c;
        const int grp = (int)fdiv(a.dv_tiles, (uint32_t)rem), t = rem - grp * a.tiles;
        tr = (int)fdiv(a.dv_tiles_c, (uint32_t)t);
        tc = t - tr * a.tiles_c;
        p0 = grp * G;
    };
    auto issue = [&](int w) {  // thread 0: the tiles of work item w
        int c, tr, tc, p0;
        decode(w, c, tr, tc, p0);
        const int r0 = tr * TH, c0 = tc * TW;
        mbar_arrive_expect_tx(&bar, box_x + box_d);
        tma_load_4d(raw_x, &a.tmap_x, c0 - HXL, r0 - HX, c, 2 * p0, &bar);
        if (a.has_deep) tma_load_4d(raw_d, &a.tmap_d, c0 / 2, r0 / 2, c, 2 * p0, &bar);
    };
    if (tid == 0 && w0 < w1) issue(w0);
    int cur_c = -1;
    f2_t bias2 = 0ull;
    const int nxb = (int)a.dv_xb.d, ndb = a.has_deep ? (int)a.dv_db.d : 0;  // pass-1 x blocks, D positions per pair

    for (int w = w0; w < w1; ++w) {
        int c, tr, tc, p0;
        decode(w, c, tr, tc, p0);
        const int np = min(G, a.npairs - p0);
        const int r0 = tr * TH, c0 = tc * TW;
        if (c != cur_c) {  // a new channel: its kernels (nobody reads the old ones any more)
            ps_stage_weights<K>(a, c, wts);
            const float bv = a.with_bias ? a.base_scale[c] * a.base_bias[c] : 0.f;
            bias2 = pk2(bv, bv);
            cur_c = c;
        }
        if (tid == 0) copy_ok = mbar_wait(&bar, (uint32_t)(w - w0) & 1, a.timeout) ? 1 : 0;
        __syncthreads();
        if (!copy_ok) return;  // the flag is raised; this CTA's remaining outputs stay unwritten
        // ---- pass 1: 2 x 2 blocks of the x region (the tile and its halo of 2P) -> X where the
        // base windows read it, the four level-1 subbands where the level-1 windows read them;
        // D -> the fifth image after Z^1
        for (int e = tid; e < np * (nxb + ndb); e += NT) {
            if (e < np * nxb) {
                const int gs = (int)fdiv(a.dv_xb, (uint32_t)e), blk = e - gs * nxb;
                const int bi = (int)fdiv(a.dv_xbw, (uint32_t)blk), bj = blk - bi * (int)a.dv_xbw.d;
                const int r = 2 * bi - HX, cl = 2 * bj - HX;  // block origin, tile-relative
                f2_t X[2][2];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    float v[2][2];
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        ld2f<T>(raw_x + ((size_t)(2 * gs + q) * RXR + r + HX + rr) * RXW + cl + HXL, v[q][0], v[q][1]);
                    X[rr][0] = pk2(v[0][0], v[1][0]);
                    X[rr][1] = pk2(v[0][1], v[1][1]);
                }
                f2_t *slot = slots + (size_t)gs * a.slot;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int y = r + rr, x = cl + cc;
                        if (y >= -P && y < TH + P && x >= -P && x < TW + P)
                            slot[a.off_x + (y + P) * a.ipitch0 + x + P] = X[rr][cc];
                    }
                const QuadP q1 = butterfly2(X[0][0], X[0][1], X[1][0], X[1][1]);
                const int o = (r / 2 + P) * a.ipitch1 + cl / 2 + P;  // level-1 position, always in the halo range
                f2_t *y1 = slot + a.off_y1;
                y1[o] = q1.ll;
                y1[o + a.iimg1] = q1.lh;
                y1[o + 2 * a.iimg1] = q1.hl;
                y1[o + 3 * a.iimg1] = q1.hh;
            } else {
                const int ee = e - np * nxb;
                const int gs = (int)fdiv(a.dv_db, (uint32_t)ee), pos = ee - gs * ndb;
                const int i = (int)fdiv(a.dv_dbw, (uint32_t)pos), j = pos - i * TW1;
                const float *d = raw_d + (size_t)(2 * gs) * TH1 * TW1 + pos;
                slots[(size_t)gs * a.slot + a.off_z1 + 4 * a.zimg1 + i * a.zpitch1 + j] = pk2(d[0], d[TH1 * TW1]);
            }
        }
        __syncthreads();
        if (tid == 0 && w + 1 < w1) issue(w + 1);  // the raw tiles are free
        // ---- level-1 conv items (2 columns x S rows) of the four subband images -> Z^1
        const int nconv = (int)a.dv_conv.d;  // per pair
        for (int e = tid; e < np * nconv; e += NT) {
            const int gs = (int)fdiv(a.dv_conv, (uint32_t)e), rem = e - gs * nconv;
            const int per_img = a.ns1 * a.ng1;
            const int s = rem / per_img, r2 = rem - s * per_img;
            const int seg = (int)fdiv(a.dv_ns1, (uint32_t)r2), strip = r2 - seg * a.ns1;
            f2_t wk[KK];
            load_weights<K>(wts + (1 + s) * WP, wk);
            f2_t *slot = slots + (size_t)gs * a.slot;
            pair_conv_strip<K, 2, S>(slot + a.off_y1 + s * a.iimg1 + seg * S * a.ipitch1 + strip * 2, a.ipitch1, wk,
                                     slot + a.off_z1 + s * a.zimg1 + seg * S * a.zpitch1 + strip * 2, a.zpitch1);
        }
        __syncthreads();
        // ---- output items (2 columns x S rows): base conv + bias + level-1 synthesis + D, one
        // store per pixel
        {
            f2_t wb[KK];
            load_weights<K>(wts, wb);
            const int nout = (int)a.dv_out.d;
            T *out = static_cast<T *>(a.out);
            for (int e = tid; e < np * nout; e += NT) {
                const int gs = (int)fdiv(a.dv_out, (uint32_t)e), rem = e - gs * nout;
                const int seg = (int)fdiv(a.dv_ns0, (uint32_t)rem), strip = rem - seg * a.ns0;
                const int r = seg * S, cc = strip * 2;  // tile-relative
                const int gr = r0 + r, gc = c0 + cc;
                const int nrows = min(S, H - gr), ncols = min(2, W - gc);
                if (nrows <= 0 || ncols <= 0) continue;  // past the plane's last row / column
                const int b0 = 2 * (p0 + gs);
                T *d0 = out + ((size_t)b0 * C + c) * HW + (size_t)gr * W + gc;
                T *d1 = b0 + 1 < B ? d0 + (size_t)C * HW : nullptr;
                const f2_t *slot = slots + (size_t)gs * a.slot;
                pair_out_item<K, 2, S, T, false, true>(slot + a.off_x + r * a.ipitch0 + cc, a.ipitch0, wb, bias2,
                                                       slot + a.off_z1 + (r >> 1) * a.zpitch1 + (cc >> 1), a.zpitch1,
                                                       a.zimg1, d0, d1, W, nrows, ncols, a.vec_st != 0);
            }
        }
        __syncthreads();
    }
}

template <int K, typename T, int NT, int S>
cudaError_t launch_pshallow_one(const PsArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_pshallow_kernel<K, T, NT, S>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)a.grid), (unsigned)NT, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T, int NT, int S>
int occ_pshallow_one(size_t smem) {
    auto kern = wtconv_pshallow_kernel<K, T, NT, S>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NT, smem) != cudaSuccess) return 0;
    return n;
}

// CTA size 64 or 128, item rows 4 or 8
template <int K, typename T>
cudaError_t launch_pshallow_t(const PsArgs &a, size_t smem, cudaStream_t st) {
    if (a.nthreads == 64) return a.s0 == 4 ? launch_pshallow_one<K, T, 64, 4>(a, smem, st) : launch_pshallow_one<K, T, 64, 8>(a, smem, st);
    if (a.nthreads == 128) return a.s0 == 4 ? launch_pshallow_one<K, T, 128, 4>(a, smem, st) : launch_pshallow_one<K, T, 128, 8>(a, smem, st);
    return cudaErrorInvalidValue;
}

template <int K, typename T>
int occ_pshallow_t(size_t smem, int nthreads, int s) {
    if (nthreads == 64) return s == 4 ? occ_pshallow_one<K, T, 64, 4>(smem) : occ_pshallow_one<K, T, 64, 8>(smem);
    if (nthreads == 128) return s == 4 ? occ_pshallow_one<K, T, 128, 4>(smem) : occ_pshallow_one<K, T, 128, 8>(smem);
    return 0;
}

template <typename T>
cudaError_t launch_pshallow_typed(const PsArgs &a, size_t smem, cudaStream_t st) {
    switch (a.K) {
    case 3: return launch_pshallow_t<3, T>(a, smem, st);
    case 5: return launch_pshallow_t<5, T>(a, smem, st);
    case 7: return launch_pshallow_t<7, T>(a, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
int occupancy_pshallow_typed(int K, size_t smem, int nthreads, int s) {
    switch (K) {
    case 3: return occ_pshallow_t<3, T>(smem, nthreads, s);
    case 5: return occ_pshallow_t<5, T>(smem, nthreads, s);
    case 7: return occ_pshallow_t<7, T>(smem, nthreads, s);
    default: return 0;
    }
}

}  // namespace wtconv
