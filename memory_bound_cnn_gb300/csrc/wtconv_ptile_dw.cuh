// Tiled batch-pair weight-gradient kernel of the WTConv layer:
//     dw'_b[u, v]   = sum_{b,h,w} dy[b, h, w] x[b, h+u-P, w+v-P],   db' = sum dy      (base path)
//     dW'^l_s[u, v] = sum_{b,i,j} Ghat^l_s[b, i, j] Yhat^l_s[b, i+u-P, j+v-P]        (level l, subband s)
// with Yhat / Ghat the unnormalised Haar pyramids of x / dy and zero padding outside each level's
// plane (paper, Principais Contribuicoes: all parameter gradients from the same on-chip pyramids;
// Metodologia: the butterflies are recomputed on chip, no intermediate tensor in HBM).
//
// A CTA walks through work units (channel, run of pair groups x tiles).  Per work item one thread
// issues two bulk tensor copies: the x tile of G batch pairs with a halo of 2^LT * P positions
// (zero outside the plane), and the dy tile.  One pass over 2^LT x 2^LT blocks builds, as
// batch-pair images, the padded x copy and its level 1 (and 2) subbands where the correlations
// read them, and the compact dy copy and its subbands.  Every correlation item (Q x S positions
// of one image, all k*k taps) may run on any thread: its tap sums go to a row of shared memory,
// and a fixed-order reduction adds the rows of each (signal, tap) into a sum that one thread keeps
// for the whole work unit, so the result does not depend on scheduling.  At the end of a unit the
// sums are written as that unit's partial; deeper levels come from a further launch on the LL
// planes this one writes.
#pragma once

#include "wtconv_pair.cuh"
#include "wtconv_ptile.h"

#include <type_traits>

namespace wtconv {

namespace {

struct PtLayout {
    size_t raw_x, raw_dy, slots, ip, red, total;  // byte offsets from a 128-byte aligned base
};

__host__ __device__ inline size_t pt_round128(size_t b) { return (b + 127) / 128 * 128; }

// Raw x tiles, raw dy tiles (bulk copy destinations), the G pair slots, one row of k*k tap sums
// per correlation item of a group, and one float per thread for the sum of dy.
__host__ __device__ inline PtLayout ptile_layout(const PtileArgs &a) {
    PtLayout p;
    size_t o = 0;
    p.raw_x = o;
    o += (size_t)a.raw_x_bytes;
    p.raw_dy = o;
    o += (size_t)a.raw_dy_bytes;
    p.slots = o;
    o += pt_round128((size_t)a.G * a.slot * sizeof(f2_t));
    p.ip = o;
    o += pt_round128((size_t)a.G * a.per_pair * a.K * a.K * sizeof(float));
    p.red = o;
    o += (size_t)a.nthreads * sizeof(float);
    p.total = o + 128;
    return p;
}

// Store the four subbands q of one position into the images of level lv at image offset o.
__device__ __forceinline__ void pt_store_quad(f2_t *img, int stride, int o, const QuadP &q) {
    img[o] = q.ll;
    img[o + stride] = q.lh;
    img[o + 2 * stride] = q.hl;
    img[o + 3 * stride] = q.hh;
}

// One correlation item of shape IQ x S (S in {4, 8}; IQ, the item width, is fixed per kernel so
// that the narrow variant holds fewer registers).
template <int K, int IQ>
__device__ __forceinline__ void pt_corr_item(int s, const f2_t *y, int ypitch, const f2_t *g, int gpitch,
                                             f2_t (&acc)[K * K]) {
    if (s == 8) pair_corr_strip<K, IQ, 8>(y, ypitch, g, gpitch, acc);
    else pair_corr_strip<K, IQ, 4>(y, ypitch, g, gpitch, acc);
}

// First item (within a pair) and item count of local signal sig.
__device__ __forceinline__ void pt_signal_items(const PtileArgs &a, int sig, int &start, int &n) {
    if (a.base && sig == 0) { start = 0; n = a.n0; return; }
    const int ls = a.base ? sig - 1 : sig;  // 4 (l - 1) + s
    const int l = ls / 4 + 1, s = ls & 3;
    if (l == 1) { start = a.n0 + s * a.n1; n = a.n1; }
    else { start = a.n0 + 4 * a.n1 + s * a.n2; n = a.n2; }
}

}  // namespace

template <int K, int IQ, int NT>
constexpr int pt_min_blocks() {
    return NT == 128 ? (IQ == 2 ? (K <= 5 ? 4 : 3) : (K <= 5 ? 3 : 2)) : (IQ == 2 ? 2 : 1);
}

template <int K, typename T, int LT, bool BASE, int NT, int IQ>
__global__ void __launch_bounds__(NT, pt_min_blocks<K, IQ, NT>()) wtconv_ptile_dw_kernel(const __grid_constant__ PtileArgs a) {
    constexpr int P = K / 2, KK = K * K, NA = KK + 1;
    constexpr int BS = 1 << LT;                        // pass-1 block: levels 1 .. LT of one position
    constexpr int NSIG = (BASE ? 1 : 0) + 4 * LT;      // signals of this launch
    extern __shared__ __align__(128) unsigned char pt_smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int copy_ok;
    const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(pt_smem);
    unsigned char *base = pt_smem + (((s0 + 127u) & ~127u) - s0);
    const PtLayout lay = ptile_layout(a);
    T *raw_x = reinterpret_cast<T *>(base + lay.raw_x);
    T *raw_dy = reinterpret_cast<T *>(base + lay.raw_dy);
    f2_t *slots = reinterpret_cast<f2_t *>(base + lay.slots);
    float *ip = reinterpret_cast<float *>(base + lay.ip);
    float *red = reinterpret_cast<float *>(base + lay.red);
    const int tid = threadIdx.x;
    const int C = a.C, G = a.G, TH = a.TH, TW = a.TW, HX = a.HX, HXL = a.HXL;
    const int RXR = a.RXR, RXW = a.RXW;
    const int nsig_total = 1 + 4 * a.L_total;
    const PtLevel &L0 = a.lv[0], &L1 = a.lv[1], &L2 = a.lv[LT >= 2 ? 2 : 1];

    {   // every slot starts at zero: the rows and columns that rounding adds stay zero
        ulonglong2 *z = reinterpret_cast<ulonglong2 *>(slots);
        const int nz = G * a.slot / 2;
        for (int i = tid; i < nz; i += NT) z[i] = make_ulonglong2(0ull, 0ull);
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();

    const int u0 = (int)((long long)blockIdx.x * a.units / a.grid);
    const int u1 = (int)((long long)(blockIdx.x + 1) * a.units / a.grid);
    auto wb = [&](int u) { return (int)((long long)(u % a.nchunks) * a.work / a.nchunks); };
    auto we = [&](int u) { return (int)((long long)(u % a.nchunks + 1) * a.work / a.nchunks); };
    const uint32_t box_x = (uint32_t)(2 * G * RXR * RXW * (int)sizeof(T));
    const uint32_t box_dy = (uint32_t)(2 * G * TH * TW * (int)sizeof(T));
    auto issue = [&](int u, int w) {  // thread 0: the two tiles of work item w of unit u
        const int c = u / a.nchunks;
        const int grp = (int)fdiv(a.dv_tiles, (uint32_t)w), t = w - grp * a.tiles;
        const int tr = (int)fdiv(a.dv_tiles_c, (uint32_t)t), tc = t - tr * a.tiles_c;
        const int r0 = tr * TH, c0 = tc * TW, b0 = 2 * grp * G;
        mbar_arrive_expect_tx(&bar, box_x + box_dy);
        tma_load_4d(raw_x, &a.tmap_x, c0 - HXL, r0 - HX, c, b0, &bar);
        tma_load_4d(raw_dy, &a.tmap_dy, c0, r0, c, b0, &bar);
    };
    // the next work item after (u, w) in this CTA's sequence, skipping empty units
    auto advance = [&](int &u, int &w) {
        ++w;
        while (u < u1 && w >= we(u)) {
            ++u;
            if (u < u1) w = wb(u);
        }
        return u < u1;
    };
    if (tid == 0) {
        int u = u0, w = u0 < u1 ? wb(u0) : 0;
        while (u < u1 && w >= we(u)) {
            ++u;
            if (u < u1) w = wb(u);
        }
        if (u < u1) issue(u, w);
    }
    uint32_t step = 0;  // copies waited for so far (mbarrier phase parity)
    const int nxb = (int)a.dv_xb.d, ndb = (int)a.dv_db.d;  // pass-1 blocks per pair: x region, dy tile

    for (int u = u0; u < u1; ++u) {
        const int c = u / a.nchunks, chunk = u - c * a.nchunks;
        float cacc[kPtMaxEntries];
#pragma unroll
        for (int k = 0; k < kPtMaxEntries; ++k) cacc[k] = 0.f;
        f2_t dysum = 0ull;
        const int w1 = we(u);
        for (int w = wb(u); w < w1; ++w, ++step) {
            const int grp = (int)fdiv(a.dv_tiles, (uint32_t)w), t = w - grp * a.tiles;
            const int tr = (int)fdiv(a.dv_tiles_c, (uint32_t)t), tc = t - tr * a.tiles_c;
            const int p0 = grp * G, np = min(G, a.npairs - p0);
            if (tid == 0) copy_ok = mbar_wait(&bar, step & 1, a.timeout) ? 1 : 0;
            __syncthreads();
            if (!copy_ok) {
                // a copy never arrived (the flag is raised): this CTA's partials become NaN, and
                // it leaves without touching the copy's destination
                for (int uu = u; uu < u1; ++uu) {
                    const int cc = uu / a.nchunks, ch = uu - cc * a.nchunks;
                    float *pp = a.partials + ((size_t)ch * C + cc) * nsig_total * NA;
                    for (int i = tid; i < nsig_total * NA; i += NT) pp[i] = __int_as_float(0x7fc00000);
                }
                return;
            }
            // ---- pass 1: x region blocks, then dy tile blocks, of every pair of the group
            for (int e = tid; e < np * (nxb + ndb); e += NT) {
                const bool isx = e < np * nxb;
                const int ee = isx ? e : e - np * nxb;
                const int gs = (int)fdiv(isx ? a.dv_xb : a.dv_db, (uint32_t)ee);
                const int blk = ee - gs * (isx ? nxb : ndb);
                const int bi = (int)fdiv(isx ? a.dv_xbw : a.dv_dbw, (uint32_t)blk);
                const int bj = blk - bi * (int)(isx ? a.dv_xbw.d : a.dv_dbw.d);
                f2_t *slot = slots + (size_t)gs * a.slot;
                // block origin, tile-relative (x: the region starts HX before the tile)
                const int r = BS * bi - (isx ? HX : 0), cl = BS * bj - (isx ? HX : 0);
                float v[2][BS][BS];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const T *src = isx ? raw_x + ((size_t)(2 * gs + q) * RXR + r + HX) * RXW + cl + HXL
                                       : raw_dy + ((size_t)(2 * gs + q) * TH + r) * TW + cl;
                    const int pitch = isx ? RXW : TW;
#pragma unroll
                    for (int rr = 0; rr < BS; ++rr) {
                        if constexpr (BS == 4) {
                            const float4 f = Act<T>::ld4(src + rr * pitch);
                            v[q][rr][0] = f.x; v[q][rr][1] = f.y; v[q][rr][2] = f.z; v[q][rr][3] = f.w;
                        } else {
                            ld2f<T>(src + rr * pitch, v[q][rr][0], v[q][rr][1]);
                        }
                    }
                }
                f2_t X[BS][BS];
#pragma unroll
                for (int rr = 0; rr < BS; ++rr)
#pragma unroll
                    for (int cc = 0; cc < BS; ++cc) X[rr][cc] = pk2(v[0][rr][cc], v[1][rr][cc]);
                if constexpr (BASE) {  // level-0 copies: padded x where the base window reads it, compact dy
                    if (isx) {
#pragma unroll
                        for (int rr = 0; rr < BS; ++rr)
#pragma unroll
                            for (int cc = 0; cc < BS; ++cc) {
                                const int y = r + rr, x = cl + cc;
                                if (y >= -P && y < TH + P && x >= -P && x < TW + P)
                                    slot[L0.off_y + (y + P) * L0.ipitch + x + P] = X[rr][cc];
                            }
                    } else {
#pragma unroll
                        for (int rr = 0; rr < BS; ++rr)
#pragma unroll
                            for (int cc = 0; cc < BS; ++cc) {
                                slot[L0.off_z + (r + rr) * L0.zpitch + cl + cc] = X[rr][cc];
                                dysum = fadd2(dysum, X[rr][cc]);
                            }
                    }
                }
                // level 1: one position per 2 x 2 sub-block
                QuadP q1[BS / 2][BS / 2];
#pragma unroll
                for (int a2 = 0; a2 < BS / 2; ++a2)
#pragma unroll
                    for (int b2 = 0; b2 < BS / 2; ++b2) {
                        q1[a2][b2] = butterfly2(X[2 * a2][2 * b2], X[2 * a2][2 * b2 + 1], X[2 * a2 + 1][2 * b2],
                                                X[2 * a2 + 1][2 * b2 + 1]);
                        const int i1 = r / 2 + a2, j1 = cl / 2 + b2;
                        if (isx) {
                            if (i1 >= -P && i1 < L1.h + P && j1 >= -P && j1 < L1.w + P)
                                pt_store_quad(slot + L1.off_y, L1.iimg, (i1 + P) * L1.ipitch + j1 + P, q1[a2][b2]);
                        } else {
                            pt_store_quad(slot + L1.off_z, L1.zimg, i1 * L1.zpitch + j1, q1[a2][b2]);
                        }
                    }
                if constexpr (LT >= 2) {  // level 2: one position per block
                    const QuadP q2 = butterfly2(q1[0][0].ll, q1[0][1].ll, q1[1][0].ll, q1[1][1].ll);
                    const int i2 = r / 4, j2 = cl / 4;
                    if (isx) {
                        if (i2 >= -P && i2 < L2.h + P && j2 >= -P && j2 < L2.w + P)
                            pt_store_quad(slot + L2.off_y, L2.iimg, (i2 + P) * L2.ipitch + j2 + P, q2);
                    } else {
                        pt_store_quad(slot + L2.off_z, L2.zimg, i2 * L2.zpitch + j2, q2);
                    }
                    if (a.ll_out && i2 >= 0 && i2 < L2.h && j2 >= 0 && j2 < L2.w) {
                        // the LL band, unnormalised, for the launch that takes the deeper levels
                        const int gi = tr * L2.h + i2, gj = tc * L2.w + j2;
                        if (gi < a.ll_h && gj < a.ll_w) {
                            float *dst = isx ? a.ll_x : a.ll_dy;
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                const int b = 2 * (p0 + gs) + q;
                                if (b < a.B)
                                    dst[(((size_t)b * C + c) * a.ll_h + gi) * a.ll_pitch + gj] =
                                        q ? hi2(q2.ll) : lo2(q2.ll);
                            }
                        }
                    }
                }
            }
            __syncthreads();
            if (tid == 0) {  // the raw tiles are free: the next work item's copies
                int un = u, wn = w;
                if (advance(un, wn)) issue(un, wn);
            }
            // ---- correlation items of the group: tap sums to one row per item
            for (int it = tid; it < np * a.per_pair; it += NT) {
                const int gs = (int)fdiv(a.dv_pp, (uint32_t)it);
                int i = it - gs * a.per_pair;
                int l = 0, s = 0;
                if (!BASE || i >= a.n0) {
                    i -= a.n0;
                    if (i < 4 * a.n1) {
                        l = 1;
                        s = (int)fdiv(a.dv_n1, (uint32_t)i);
                        i -= s * a.n1;
                    } else {
                        i -= 4 * a.n1;
                        l = 2;
                        s = (int)fdiv(a.dv_n2, (uint32_t)i);
                        i -= s * a.n2;
                    }
                }
                const PtLevel &lv = a.lv[l];
                const int seg = (int)fdiv(a.dv_ns[l], (uint32_t)i), strip = i - seg * lv.ns;
                const f2_t *slot = slots + (size_t)gs * a.slot;
                const f2_t *yw = slot + lv.off_y + s * lv.iimg + seg * lv.S * lv.ipitch + strip * lv.Q;
                const f2_t *gw = slot + lv.off_z + s * lv.zimg + seg * lv.S * lv.zpitch + strip * lv.Q;
                f2_t acc[KK];
#pragma unroll
                for (int k = 0; k < KK; ++k) acc[k] = 0ull;
                pt_corr_item<K, IQ>(lv.S, yw, lv.ipitch, gw, lv.zpitch, acc);
                float *row = ip + (size_t)it * KK;
#pragma unroll
                for (int k = 0; k < KK; ++k) row[k] = lo2(acc[k]) + hi2(acc[k]);
            }
            __syncthreads();
            // ---- fixed-order reduction of the rows into this thread's (signal, tap) sums
#pragma unroll
            for (int k = 0; k < kPtMaxEntries; ++k) {
                const int e = tid + k * NT;
                if (e < NSIG * KK) {
                    const int sig = e / KK, tap = e - sig * KK;
                    int start, n;
                    pt_signal_items(a, sig, start, n);
                    // four interleaved partial sums (rows j = 0, 1, 2, 3 mod 4), combined in a
                    // fixed order: the loads overlap, and the result depends only on the geometry
                    float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
                    for (int gs = 0; gs < np; ++gs) {
                        const float *col = ip + ((size_t)gs * a.per_pair + start) * KK + tap;
                        int j = 0;
                        for (; j + 4 <= n; j += 4) {
                            v0 += col[j * KK];
                            v1 += col[(j + 1) * KK];
                            v2 += col[(j + 2) * KK];
                            v3 += col[(j + 3) * KK];
                        }
                        for (; j < n; ++j) v0 += col[j * KK];
                    }
                    cacc[k] += (v0 + v1) + (v2 + v3);
                }
            }
        }

        // ---- this unit's partial: every (signal, tap) of the launch, and the sum of dy
        float *pp = a.partials + ((size_t)chunk * C + c) * nsig_total * NA;
#pragma unroll
        for (int k = 0; k < kPtMaxEntries; ++k) {
            const int e = tid + k * NT;
            if (e < NSIG * KK) {
                const int sig = e / KK, tap = e - sig * KK;
                const int gsig = (BASE && sig == 0) ? 0 : 1 + 4 * a.lvl_off + (BASE ? sig - 1 : sig);
                pp[gsig * NA + tap] = cacc[k];
            }
        }
        if constexpr (BASE) {
            red[tid] = lo2(dysum) + hi2(dysum);
            __syncthreads();
            if (tid == 0) {
                float v = 0.f;
                for (int t = 0; t < NT; ++t) v += red[t];
                pp[KK] = v;
            }
            __syncthreads();
        }
    }
}

template <int K, typename T, int LT, bool BASE>
auto ptile_kernel(int nthreads, int iq) {
    return nthreads == 256 ? (iq == 2 ? wtconv_ptile_dw_kernel<K, T, LT, BASE, 256, 2> : wtconv_ptile_dw_kernel<K, T, LT, BASE, 256, 4>)
                           : (iq == 2 ? wtconv_ptile_dw_kernel<K, T, LT, BASE, 128, 2> : wtconv_ptile_dw_kernel<K, T, LT, BASE, 128, 4>);
}

template <int K, typename T, int LT, bool BASE>
cudaError_t launch_ptile_dw_t(const PtileArgs &a, size_t smem, cudaStream_t st) {
    auto kern = ptile_kernel<K, T, LT, BASE>(a.nthreads, a.lv[0].Q);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)a.grid), (unsigned)a.nthreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T, int LT, bool BASE>
int occ_ptile_dw_t(size_t smem, int nthreads, int iq) {
    auto kern = ptile_kernel<K, T, LT, BASE>(nthreads, iq);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, nthreads, smem) != cudaSuccess) return 0;
    return n;
}

// Dispatch over K, LT and the base flag for one activation type (launches without the base path
// run on the fp32 LL planes only).
template <typename T>
cudaError_t launch_ptile_dw_typed(const PtileArgs &a, size_t smem, cudaStream_t st) {
    constexpr bool kF32 = std::is_same<T, float>::value;
    if (!kF32 && !a.base) return cudaErrorInvalidValue;
#define WTCONV_PT_CASE(KV)                                                                             \
    case KV:                                                                                           \
        if constexpr (kF32) {                                                                          \
            if (!a.base) return a.LT == 2 ? launch_ptile_dw_t<KV, T, 2, false>(a, smem, st)            \
                                          : launch_ptile_dw_t<KV, T, 1, false>(a, smem, st);           \
        }                                                                                              \
        return a.LT == 2 ? launch_ptile_dw_t<KV, T, 2, true>(a, smem, st) : launch_ptile_dw_t<KV, T, 1, true>(a, smem, st);
    switch (a.K) {
        WTCONV_PT_CASE(3)
        WTCONV_PT_CASE(5)
        WTCONV_PT_CASE(7)
    default: return cudaErrorInvalidValue;
    }
#undef WTCONV_PT_CASE
}

template <typename T>
int occupancy_ptile_dw_typed(int K, int LT, int base, size_t smem, int nthreads, int iq) {
    constexpr bool kF32 = std::is_same<T, float>::value;
    if (!kF32 && !base) return 0;
#define WTCONV_PT_CASE(KV)                                                                             \
    case KV:                                                                                           \
        if constexpr (kF32) {                                                                          \
            if (!base) return LT == 2 ? occ_ptile_dw_t<KV, T, 2, false>(smem, nthreads, iq)                \
                                      : occ_ptile_dw_t<KV, T, 1, false>(smem, nthreads, iq);               \
        }                                                                                              \
        return LT == 2 ? occ_ptile_dw_t<KV, T, 2, true>(smem, nthreads, iq) : occ_ptile_dw_t<KV, T, 1, true>(smem, nthreads, iq);
    switch (K) {
        WTCONV_PT_CASE(3)
        WTCONV_PT_CASE(5)
        WTCONV_PT_CASE(7)
    default: return 0;
    }
#undef WTCONV_PT_CASE
}

}  // namespace wtconv
