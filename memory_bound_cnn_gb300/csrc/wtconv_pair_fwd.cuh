// Batch-pair forward kernel of the WTConv layer: y (or the input gradient dx, with rotated
// kernels and no bias) for planes whose whole Haar pyramid fits in shared memory.
//
// A CTA owns channel c and walks through groups of G batch pairs (b, b+1) of that channel.  Per
// group, with every image a packed pair of the two planes:
//   1. bulk copies bring the raw planes into shared memory (the next group's copies start as soon
//      as the current group has read its planes, unless the raw area shares space with the
//      level-1 outputs);
//   2. analysis: 4x4 blocks of the planes give the interleaved padded copy X and the quads of Haar
//      levels 1 and 2; later passes build levels 3 .. L from the low band, two levels per pass;
//   3. conv: every subband image of every level runs strip items (folded kernels, packed f32x2
//      FMAs) into compact outputs Z^l_s;
//   4. deep gather: each level-2 position adds the closed-form synthesis of levels >= 2 (signs
//      from the coordinate bits) into the level-1 LL outputs below it;
//   5. output: strip items run the base conv on X (the bias enters with the first tap) and, as
//      each pair of output rows completes, add the level-1 inverse butterflies of Z^1 and store
//      the two planes' pixels.
// x is read once from HBM and y written once; nothing else leaves the chip.
#pragma once

#include "wtconv_pair.cuh"

namespace wtconv {

namespace {

struct PairFwdLayout {
    size_t slots, raw, wts, total;  // byte offsets from a 128-byte aligned base
};

__host__ __device__ inline PairFwdLayout pair_fwd_layout(const PairArgs &a) {
    PairFwdLayout p;
    size_t o = 0;
    p.slots = o;
    o += (size_t)a.G * a.geo.slot * sizeof(f2_t);
    o = (o + 127) / 128 * 128;
    p.raw = o;  // raw planes of the group (the next group's copies land here once pass 1 is done)
    if (a.tma) o += (size_t)a.G * a.raw_pair_bytes;
    o = (o + 15) / 16 * 16;
    p.wts = o;
    o += (size_t)(1 + 4 * a.L) * wpairs(a.K) * sizeof(f2_t);
    p.total = o + 128;  // room to align the base
    return p;
}

// Two activations to a row: fp32 pair, or one packed 32-bit word of a narrow type.
template <typename T> struct Act2;
template <> struct Act2<float> {
    static __device__ __forceinline__ void st(float *p, float a, float b) {
        *reinterpret_cast<float2 *>(p) = make_float2(a, b);
    }
};
template <> struct Act2<__nv_bfloat16> {
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, float a, float b) {
        *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
    }
};
template <> struct Act2<__half> {
    static __device__ __forceinline__ void st(__half *p, float a, float b) {
        *reinterpret_cast<__half2 *>(p) = __floats2half2_rn(a, b);
    }
};

// Store output row `r` (Q packed pairs) of both planes: low halves to d0, high halves to d1.
template <int Q, typename T>
__device__ __forceinline__ void store_row(const f2_t (&acc)[Q], T *d0, T *d1, int ncols, bool vec) {
    float v0[Q], v1[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        v0[q] = lo2(acc[q]);
        v1[q] = hi2(acc[q]);
    }
    if (vec && ncols == Q) {
        if constexpr (Q == 4) {
            Act<T>::st4(d0, v0);
            if (d1) Act<T>::st4(d1, v1);
        } else {
            Act2<T>::st(d0, v0[0], v0[1]);
            if (d1) Act2<T>::st(d1, v1[0], v1[1]);
        }
    } else {
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            if (q < ncols) {
                Act<T>::st(d0 + q, v0[q]);
                if (d1) Act<T>::st(d1 + q, v1[q]);
            }
        }
    }
}

// Output item: Q columns x S rows of pixels of both planes.  Base conv on the padded X window
// (`in` at its origin) with the bias on the first tap.  Each output row is finished and stored as
// soon as its window is complete: an even row 2m adds the level-1 inverse butterflies of row m of
// Z^1 (LL already holding the deeper levels) for a = 0 and keeps those for a = 1 until row 2m+1:
// pixel (a, b) of position (m, p) gains LL + (-1)^b LH + (-1)^a HL + (-1)^(a+b) HH.
// SKIP: as in pair_conv_strip, the first zt and last zb window rows are zero padding.  DEEP: a
// fifth image after the four subband images of z1 (at z1 + 4 zimg) holds the contribution of the
// deeper levels at level-1 resolution, which enters with the low band (all four pixels).
// DREG (Q = 2 only): dreg[m] holds the deeper levels' contribution for the item's level-1 row m,
// added with the low band in place of a deep image.
template <int K, int Q, int S, typename T, bool SKIP = false, bool DEEP = false, bool DREG = false>
__device__ __forceinline__ void pair_out_item(const f2_t *__restrict__ in, int pitch, const f2_t (&w)[K * K],
                                              f2_t bias2, const f2_t *__restrict__ z1, int zpitch, int zimg, T *d0,
                                              T *d1, int W, int nrows, int ncols, bool vec, int zt = 0, int zb = 0,
                                              const f2_t *dreg = nullptr) {
    constexpr int NW = Q + K - 1, NL = (NW + 1) / 2, QL = Q / 2;
    f2_t acc[S][Q];
    f2_t pend[Q];  // the odd row's synthesis terms
    if constexpr (SKIP) {
#pragma unroll
        for (int j = 0; j < S; ++j)
#pragma unroll
            for (int q = 0; q < Q; ++q) acc[j][q] = bias2;
    }
#pragma unroll
    for (int i = 0; i < S + K - 1; ++i) {
        if (!SKIP || (i >= zt && i < S + K - 1 - zb)) {
        f2_t x[2 * NL];
        const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(in + i * pitch);
#pragma unroll
        for (int t = 0; t < NL; ++t) {
            const ulonglong2 v = p[t];
            x[2 * t] = v.x;
            x[2 * t + 1] = v.y;
        }
#pragma unroll
        for (int v = 0; v < K; ++v)
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < S) {
#pragma unroll
                    for (int q = 0; q < Q; ++q) {
                        if (!SKIP && u == 0 && v == 0) acc[j][q] = ffma2(w[0], x[q], bias2);
                        else ffma2_acc(acc[j][q], w[u * K + v], x[q + v]);
                    }
                }
            }
        }
        const int jd = i - (K - 1);
        if (jd < 0) continue;
        if ((jd & 1) == 0) {
            const f2_t *zr = z1 + (jd >> 1) * zpitch;
            f2_t ll[QL], lh[QL], hl[QL], hh[QL];
            if constexpr (QL == 2) {
                const ulonglong2 a0 = *reinterpret_cast<const ulonglong2 *>(zr);
                const ulonglong2 a1 = *reinterpret_cast<const ulonglong2 *>(zr + zimg);
                const ulonglong2 a2 = *reinterpret_cast<const ulonglong2 *>(zr + 2 * zimg);
                const ulonglong2 a3 = *reinterpret_cast<const ulonglong2 *>(zr + 3 * zimg);
                ll[0] = a0.x; ll[1] = a0.y; lh[0] = a1.x; lh[1] = a1.y;
                hl[0] = a2.x; hl[1] = a2.y; hh[0] = a3.x; hh[1] = a3.y;
                if constexpr (DEEP) {
                    const ulonglong2 a4 = *reinterpret_cast<const ulonglong2 *>(zr + 4 * zimg);
                    ll[0] = fadd2(ll[0], a4.x);
                    ll[1] = fadd2(ll[1], a4.y);
                }
            } else {
                ll[0] = zr[0]; lh[0] = zr[zimg]; hl[0] = zr[2 * zimg]; hh[0] = zr[3 * zimg];
                if constexpr (DEEP) ll[0] = fadd2(ll[0], zr[4 * zimg]);
                if constexpr (DREG) ll[0] = fadd2(ll[0], dreg[jd >> 1]);
            }
#pragma unroll
            for (int m = 0; m < QL; ++m) {
                const f2_t t0 = fadd2(ll[m], hl[m]), t1 = fsub2(ll[m], hl[m]);
                const f2_t u0 = fadd2(lh[m], hh[m]), u1 = fsub2(lh[m], hh[m]);
                acc[jd][2 * m] = fadd2(acc[jd][2 * m], fadd2(t0, u0));
                acc[jd][2 * m + 1] = fadd2(acc[jd][2 * m + 1], fsub2(t0, u0));
                pend[2 * m] = fadd2(t1, u1);
                pend[2 * m + 1] = fsub2(t1, u1);
            }
        } else {
#pragma unroll
            for (int q = 0; q < Q; ++q) acc[jd][q] = fadd2(acc[jd][q], pend[q]);
        }
        if (jd < nrows) store_row<Q, T>(acc[jd], d0 + (size_t)jd * W, d1 ? d1 + (size_t)jd * W : nullptr, ncols, vec);
    }
}

// n / d for an index decode: with a compile-time geometry (FIX) d is a constant after inlining
// and the division becomes a multiply-shift; otherwise the planner's fast divisor of d.
template <bool FIX>
__device__ __forceinline__ int divq(int n, int d, const FastDiv &f) {
    if constexpr (FIX) return n / d;
    else return (int)fdiv(f, (uint32_t)n);
}

// Conv items of level l of every slot (every subband image), in the order of a flat item list
// whose first `base` entries went to the threads before: thread tid takes items e with
// (base + e) % nt == tid.  The level's geometry sits in registers for the whole loop.
template <int K, int Q, int S, bool FIX, bool SKIP = false>
__device__ __forceinline__ void conv_level(const PairArgs &a, const PairGeo &g, f2_t *slots, const f2_t *wts, int np,
                                           int l, int base, int t0 = 0, int nt = 0) {
    constexpr int WP = wpairs(K), KK = K * K;
    if (nt == 0) nt = blockDim.x;
    const int ns = g.ns[l], per_img = ns * g.ng[l];
    const int ip = g.ipitch[l], zp = g.zpitch[l], ii = g.iimg[l], zi = g.zimg[l];
    const int oy = g.off_y[l], oz = g.off_z[l], slot = g.slot;
    const FastDiv dpi = a.dv_lvl[l], dns = a.dv_lvl_ns[l];
    const int n = np * 4 * per_img;
    int e = (int)threadIdx.x - t0 - base % nt;
    if (e < 0) e += nt;
    for (; e < n; e += nt) {
        const int img = divq<FIX>(e, per_img, dpi), rem = e - img * per_img;
        const int seg = divq<FIX>(rem, ns, dns), strip = rem - seg * ns;
        const int gs = img >> 2, s = img & 3;
        f2_t w[KK];
        load_weights<K>(wts + (1 + 4 * (l - 1) + s) * WP, w);
        f2_t *sl = slots + (size_t)gs * slot;
        // window rows above the plane / at or below its last row (SKIP only)
        const int zt = max(0, K / 2 - seg * S), zb = max(0, (seg + 1) * S + K / 2 - g.h[l]);
        pair_conv_strip<K, Q, S, SKIP>(sl + oy + s * ii + seg * S * ip + strip * Q, ip, w,
                                       sl + oz + s * zi + seg * S * zp + strip * Q, zp, zt, zb);
    }
}

// Analysis pass building level l0 (and l0+1 when it exists) of every slot's pyramid from the
// low band of level l0-1 (an interior image of the slot).  Blocks are 4x4 of the finer low band
// when two levels are built, 2x2 otherwise.  Threads t0 .. t0+nt-1 share the blocks.
__device__ __forceinline__ void analysis_deep_pass(const PairGeo &g, f2_t *slots, int np, int l0, int L, int t0,
                                                   int nt) {
    const bool two = l0 + 1 <= L;
    const int hs = g.h[l0 - 1], ws = g.w[l0 - 1];
    const int bsz = two ? 4 : 2;
    const int bw = ws / bsz, n = (hs / bsz) * bw;
    const int P = g.P;
    const int sp = g.ipitch[l0 - 1];
    for (int t = (int)threadIdx.x - t0; t < np * n; t += nt) {
        const int gs = t / n, e = t - gs * n;
        const int bi = e / bw, bj = e - bi * bw;
        f2_t *slot = slots + (size_t)gs * g.slot;
        const f2_t *src = slot + g.off_y[l0 - 1] + (bsz * bi + P) * sp + bsz * bj + P;
        f2_t *y0 = slot + g.off_y[l0];
        const int p0 = g.ipitch[l0], i0 = g.iimg[l0];
        if (two) {
            f2_t v[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) v[r][cc] = src[r * sp + cc];
            QuadP q[2][2];
#pragma unroll
            for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2) {
                    q[a2][b2] = butterfly2(v[2 * a2][2 * b2], v[2 * a2][2 * b2 + 1], v[2 * a2 + 1][2 * b2],
                                           v[2 * a2 + 1][2 * b2 + 1]);
                    f2_t *d = y0 + (2 * bi + a2 + P) * p0 + 2 * bj + b2 + P;
                    d[0] = q[a2][b2].ll;
                    d[i0] = q[a2][b2].lh;
                    d[2 * i0] = q[a2][b2].hl;
                    d[3 * i0] = q[a2][b2].hh;
                }
            const QuadP q2 = butterfly2(q[0][0].ll, q[0][1].ll, q[1][0].ll, q[1][1].ll);
            const int p1 = g.ipitch[l0 + 1], i1 = g.iimg[l0 + 1];
            f2_t *d = slot + g.off_y[l0 + 1] + (bi + P) * p1 + bj + P;
            d[0] = q2.ll;
            d[i1] = q2.lh;
            d[2 * i1] = q2.hl;
            d[3 * i1] = q2.hh;
        } else {
            const QuadP q = butterfly2(src[0], src[1], src[sp], src[sp + 1]);
            f2_t *d = y0 + (bi + P) * p0 + bj + P;
            d[0] = q.ll;
            d[i0] = q.lh;
            d[2 * i0] = q.hl;
            d[3 * i0] = q.hh;
        }
    }
}

// The contribution of levels >= 2 to level-1 positions (i1 + m, j1), m < 4 (i1 a multiple of 4):
// per level-2 position (i2, j2) the closed form adds, at level-1 position (2 i2 + a, 2 j2 + b),
// LL + (-1)^b LH + (-1)^a (HL + (-1)^b HH) of level 2 plus the levels >= 3 term v(i2, j2), whose
// signs come from the bits of (i2, j2) as in the gather phase.
__device__ __forceinline__ void deep_col4(const PairGeo &g, const f2_t *slot, int i1, int j1, f2_t (&d)[4]) {
    const int j2 = j1 >> 1;
    const bool b = j1 & 1;
    const int zi2 = g.zimg[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i2 = (i1 >> 1) + h;
        f2_t v = pk2(0.f, 0.f);
#pragma unroll
        for (int l = 3; l <= kMaxLevels; ++l) {
            if (l > g.L) break;
            const int sh = l - 2;
            const f2_t *zl = slot + g.off_z[l] + (i2 >> sh) * g.zpitch[l] + (j2 >> sh);
            const int zi = g.zimg[l];
            const bool ra = (i2 >> (sh - 1)) & 1, cb = (j2 >> (sh - 1)) & 1;
            const f2_t pp = ra ? fsub2(zl[0], zl[2 * zi]) : fadd2(zl[0], zl[2 * zi]);
            const f2_t rr = ra ? fsub2(zl[zi], zl[3 * zi]) : fadd2(zl[zi], zl[3 * zi]);
            v = fadd2(v, cb ? fsub2(pp, rr) : fadd2(pp, rr));
        }
        const f2_t *z2 = slot + g.off_z[2] + i2 * g.zpitch[2] + j2;
        const f2_t t0 = fadd2(fadd2(z2[0], z2[2 * zi2]), v), t1 = fadd2(fsub2(z2[0], z2[2 * zi2]), v);
        const f2_t u0 = fadd2(z2[zi2], z2[3 * zi2]), u1 = fsub2(z2[zi2], z2[3 * zi2]);
        d[2 * h] = b ? fsub2(t0, u0) : fadd2(t0, u0);
        d[2 * h + 1] = b ? fsub2(t1, u1) : fadd2(t1, u1);
    }
}

// Output items of every slot with item shape Q x S (the base kernel in registers for the loop).
// FOLD (Q = 2, S a multiple of 8, L >= 2): the items add the levels >= 2 themselves (deep_col4)
// instead of reading them from a gather phase.
template <int K, int Q, int S, typename T, bool FIX, bool SKIP = false, bool FOLD = false>
__device__ __forceinline__ void out_phase(const PairArgs &a, const PairGeo &g, const f2_t *slots, const f2_t *wts,
                                          int np, int p0, int c, f2_t bias2, T *out) {
    constexpr int KK = K * K;
    f2_t w[KK];
    load_weights<K>(wts, w);
    const int ns0 = g.ns[0], ip0 = g.ipitch[0], zp1 = g.zpitch[1], zi1 = g.zimg[1];
    const int ox = g.off_x, oz1 = g.off_z[1], slot = g.slot, n_out = g.ns[0] * g.ng[0];
    const int B = a.B, C = a.C, H = g.H, W = g.W;
    const size_t HW = (size_t)H * W;
    const bool vec = a.vec_st != 0;
    for (int t = threadIdx.x; t < np * n_out; t += blockDim.x) {
        const int gs = divq<FIX>(t, n_out, a.dv_nout), e = t - gs * n_out;
        const int seg = divq<FIX>(e, ns0, a.dv_out_ns), strip = e - seg * ns0;
        const int r0 = seg * S, c0 = strip * Q;
        const f2_t *sl = slots + (size_t)gs * slot;
        const int b0 = 2 * (p0 + gs);
        T *d0 = out + ((size_t)b0 * C + c) * HW + (size_t)r0 * W + c0;
        T *d1 = b0 + 1 < B ? d0 + (size_t)C * HW : nullptr;
        const int zt = max(0, K / 2 - r0), zb = max(0, r0 + S + K / 2 - H);
        if constexpr (FOLD) {
            static_assert(Q == 2 && S % 8 == 0, "FOLD: items of 2 columns and a multiple of 8 rows");
            f2_t dr[S / 2];
#pragma unroll
            for (int m = 0; m < S / 2; m += 4) {
                f2_t d4[4];
                deep_col4(g, sl, (r0 >> 1) + m, c0 >> 1, d4);
#pragma unroll
                for (int q = 0; q < 4; ++q) dr[m + q] = d4[q];
            }
            pair_out_item<K, Q, S, T, SKIP, false, true>(sl + ox + r0 * ip0 + c0, ip0, w, bias2,
                                                         sl + oz1 + (r0 >> 1) * zp1 + (c0 >> 1), zp1, zi1, d0, d1, W,
                                                         min(S, H - r0), min(Q, W - c0), vec, zt, zb, dr);
        } else {
            pair_out_item<K, Q, S, T, SKIP>(sl + ox + r0 * ip0 + c0, ip0, w, bias2, sl + oz1 + (r0 >> 1) * zp1 + (c0 >> 1),
                                            zp1, zi1, d0, d1, W, min(S, H - r0), min(Q, W - c0), vec, zt, zb);
        }
    }
}

// First analysis pass: 4x4 (L >= 2) or 2x2 (L == 1) blocks of the raw planes -> the interleaved
// padded copy X and the Haar level 1 (and level 2) quads of every slot.  plane(gs, q) gives the raw
// plane q of slot gs, or null past B.
template <int BS, typename T, bool FIX, typename PlaneFn>
__device__ __forceinline__ void pass1(const PairArgs &a, const PairGeo &g, f2_t *slots, int np, PlaneFn plane) {
    const int P = g.P, W = g.W, bw = W / BS, n_a = (g.H / BS) * bw;
    const int p1 = g.ipitch[1], i1 = g.iimg[1], oy1 = g.off_y[1];
    const int p2 = BS == 4 ? g.ipitch[2] : 0, i2 = BS == 4 ? g.iimg[2] : 0, oy2 = BS == 4 ? g.off_y[2] : 0;
    for (int t = threadIdx.x; t < np * n_a; t += blockDim.x) {
        const int gs = divq<FIX>(t, n_a, a.dv_na), blk = t - gs * n_a;
        const int bi = divq<FIX>(blk, bw, a.dv_naw), bj = blk - bi * bw;
        f2_t *slot = slots + (size_t)gs * g.slot;
        f2_t X[BS][BS];
        {
            float v[2][BS][BS];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const T *pl = plane(gs, q);
                if (pl) {
                    const T *src = pl + (size_t)(BS * bi) * W + BS * bj;
#pragma unroll
                    for (int r = 0; r < BS; ++r) {
                        if constexpr (BS == 4) {
                            const float4 f = Act<T>::ld4(src + r * W);
                            v[q][r][0] = f.x; v[q][r][1] = f.y; v[q][r][2] = f.z; v[q][r][3] = f.w;
                        } else {
                            ld2f<T>(src + r * W, v[q][r][0], v[q][r][1]);
                        }
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < BS; ++r)
#pragma unroll
                        for (int cc = 0; cc < BS; ++cc) v[q][r][cc] = 0.f;
                }
            }
#pragma unroll
            for (int r = 0; r < BS; ++r)
#pragma unroll
                for (int cc = 0; cc < BS; ++cc) X[r][cc] = pk2(v[0][r][cc], v[1][r][cc]);
        }
        {   // the interleaved padded copy X (interior at (P, P))
            f2_t *xd = slot + g.off_x + (BS * bi + P) * g.ipitch[0] + BS * bj + P;
#pragma unroll
            for (int r = 0; r < BS; ++r) {
                if (BS == 4 && (P & 1) == 0) {
                    reinterpret_cast<ulonglong2 *>(xd + r * g.ipitch[0])[0] = make_ulonglong2(X[r][0], X[r][1]);
                    reinterpret_cast<ulonglong2 *>(xd + r * g.ipitch[0])[1] = make_ulonglong2(X[r][BS - 2], X[r][BS - 1]);
                } else {
#pragma unroll
                    for (int cc = 0; cc < BS; ++cc) xd[r * g.ipitch[0] + cc] = X[r][cc];
                }
            }
        }
        if constexpr (BS == 4) {
            QuadP q1[2][2];
#pragma unroll
            for (int a2 = 0; a2 < 2; ++a2) {
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2)
                    q1[a2][b2] = butterfly2(X[2 * a2][2 * b2], X[2 * a2][2 * b2 + 1], X[2 * a2 + 1][2 * b2],
                                            X[2 * a2 + 1][2 * b2 + 1]);
                f2_t *d = slot + oy1 + (2 * bi + a2 + P) * p1 + 2 * bj + P;
                if ((P & 1) == 0) {
                    *reinterpret_cast<ulonglong2 *>(d) = make_ulonglong2(q1[a2][0].ll, q1[a2][1].ll);
                    *reinterpret_cast<ulonglong2 *>(d + i1) = make_ulonglong2(q1[a2][0].lh, q1[a2][1].lh);
                    *reinterpret_cast<ulonglong2 *>(d + 2 * i1) = make_ulonglong2(q1[a2][0].hl, q1[a2][1].hl);
                    *reinterpret_cast<ulonglong2 *>(d + 3 * i1) = make_ulonglong2(q1[a2][0].hh, q1[a2][1].hh);
                } else {
#pragma unroll
                    for (int b2 = 0; b2 < 2; ++b2) {
                        d[b2] = q1[a2][b2].ll;
                        d[i1 + b2] = q1[a2][b2].lh;
                        d[2 * i1 + b2] = q1[a2][b2].hl;
                        d[3 * i1 + b2] = q1[a2][b2].hh;
                    }
                }
            }
            const QuadP q2 = butterfly2(q1[0][0].ll, q1[0][1].ll, q1[1][0].ll, q1[1][1].ll);
            f2_t *d2 = slot + oy2 + (bi + P) * p2 + bj + P;
            d2[0] = q2.ll;
            d2[i2] = q2.lh;
            d2[2 * i2] = q2.hl;
            d2[3 * i2] = q2.hh;
        } else {
            const QuadP q1 = butterfly2(X[0][0], X[0][1], X[1][0], X[1][1]);
            f2_t *d = slot + oy1 + (bi + P) * p1 + bj + P;
            d[0] = q1.ll;
            d[i1] = q1.lh;
            d[2 * i1] = q1.hl;
            d[3 * i1] = q1.hh;
        }
    }
}

}  // namespace

// The forward kernel's body, for a geometry `g` that is either the plan's (runtime values) or,
// with FIX, a compile-time constant of a specialised instantiation: then every pitch and offset is
// an immediate, the level loops unroll and index decodes divide by constants.
// Conv items of levels LV .. L of an instantiation with a compile-time geometry: each level's
// item shape is a constant (rows drop to 4 on images of at most 4 rows), so shapes outside the
// run-time menu (e.g. 7-row items on 28 x 28 planes) work as well.
template <int K, class Spec, int LV, int LAST = Spec::kL>
__device__ __forceinline__ void conv_levels_fixed(const PairArgs &a, const PairGeo &g, f2_t *slots, const f2_t *wts,
                                                  int np, int first, int t0 = 0, int nt = 0) {
    if constexpr (LV <= LAST) {
        constexpr int Q = LV == 1 ? Spec::kQL : Spec::kQD;
        constexpr int S = (Spec::kH >> LV) <= 4 ? 4 : (LV == 1 ? Spec::kSL : Spec::kSD);
        conv_level<K, Q, S, true, Spec::kSkip>(a, g, slots, wts, np, LV, np * first, t0, nt);
        conv_levels_fixed<K, Spec, LV + 1, LAST>(a, g, slots, wts, np, first + 4 * g.ns[LV] * g.ng[LV], t0, nt);
    }
}

// Conv items of levels l_lo .. l_hi of a run-time geometry, on threads t0 .. t0+nt-1.
template <int K>
__device__ __forceinline__ void conv_levels_dyn(const PairArgs &a, const PairGeo &g, f2_t *slots, const f2_t *wts,
                                                int np, int l_lo, int l_hi, int t0, int nt) {
    int first = 0;  // conv items of the levels before l, per slot
    for (int l = l_lo; l <= l_hi; ++l) {
        const int base_l = np * first;
        first += 4 * g.ns[l] * g.ng[l];
        const int Ql = g.Q[l], Sl = g.S[l];
        if (Ql == 4) {
            if (Sl == 8) conv_level<K, 4, 8, false>(a, g, slots, wts, np, l, base_l, t0, nt);
            else conv_level<K, 4, 4, false>(a, g, slots, wts, np, l, base_l, t0, nt);
        } else {
            if (Sl == 8) conv_level<K, 2, 8, false>(a, g, slots, wts, np, l, base_l, t0, nt);
            else conv_level<K, 2, 4, false>(a, g, slots, wts, np, l, base_l, t0, nt);
        }
    }
}

// Whether an instantiation's output items add the levels >= 2 themselves (no gather phase): the
// shape-specialised ones with L >= 3 and 2 x 8k output items.  Measured on GB300: 64 x 64 L4 bf16
// 234 -> 230 us (the phase and its barrier cost more than the items' extra loads); 32 x 32 L3
// bf16 and 56 x 56 L3 fp32 unchanged.
template <class Spec>
__host__ __device__ constexpr bool fold_deep() {
    if constexpr (Spec::fixed)
        return Spec::kL >= 3 && Spec::kQ0 == 2 && Spec::kH > 4 && Spec::kS0 % 8 == 0 && Spec::kH % Spec::kS0 == 0;
    else return false;
}

template <int K, typename T, class Spec>
__device__ __forceinline__ void pair_fwd_body(const PairArgs &a, const PairGeo &g) {
    constexpr bool FIX = Spec::fixed;
    extern __shared__ __align__(128) unsigned char pair_smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int copy_ok;
    const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(pair_smem);
    unsigned char *base = pair_smem + (((s0 + 127u) & ~127u) - s0);
    const PairFwdLayout lay = pair_fwd_layout(a);
    f2_t *slots = reinterpret_cast<f2_t *>(base + lay.slots);
    f2_t *wts = reinterpret_cast<f2_t *>(base + lay.wts);
    const int tid = threadIdx.x, nt = blockDim.x;
    const int B = a.B, C = a.C, H = g.H, W = g.W, L = g.L;
    const size_t HW = (size_t)H * W;
    const T *x = static_cast<const T *>(a.x);
    T *out = static_cast<T *>(a.out);

    {   // every slot starts at zero: halos and the padding past each interior read as zero
        ulonglong2 *z = reinterpret_cast<ulonglong2 *>(slots);
        const int nz = a.G * g.slot / 2;
        for (int i = tid; i < nz; i += nt) z[i] = make_ulonglong2(0ull, 0ull);
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();

    // this CTA's work units: (channel, group) pairs, channel-major
    const int u0 = (int)((long long)blockIdx.x * a.units / a.grid);
    const int u1 = (int)((long long)(blockIdx.x + 1) * a.units / a.grid);
    T *raw = reinterpret_cast<T *>(base + lay.raw);
    const int raw_pair = a.raw_pair_bytes / (int)sizeof(T);
    // thread 0: the bulk copies of unit u's planes (a warp-wide issue measured slower: the extra
    // registers it costs outweigh the shorter issue)
    auto issue = [&](int u) {
        const int cu = u / a.ngroups, p0 = (u - cu * a.ngroups) * a.G, np = min(a.G, a.npairs - p0);
        const uint32_t pb = (uint32_t)(HW * sizeof(T));
        if (a.tma_map) {  // one copy of the 2G planes (zero past B; the byte count is the whole box)
            mbar_arrive_expect_tx(&bar, (uint32_t)(2 * a.G) * pb);
            tma_load_4d(raw, &a.tmap_x, 0, 0, cu, 2 * p0, &bar);
            return;
        }
        uint32_t bytes = 0;
        for (int gs = 0; gs < np; ++gs)
            for (int q = 0; q < 2; ++q)
                if (2 * (p0 + gs) + q < B) bytes += pb;
        mbar_arrive_expect_tx(&bar, bytes);
        for (int gs = 0; gs < np; ++gs)
            for (int q = 0; q < 2; ++q) {
                const int b = 2 * (p0 + gs) + q;
                if (b < B) bulk_load(raw + (size_t)gs * raw_pair + q * HW, x + ((size_t)b * C + cu) * HW, pb, &bar);
            }
    };
    if (a.tma && tid == 0 && u0 < u1) issue(u0);
    int cur_c = -1;
    float bias = 0.f;
    // L >= 3 on CTAs of 128 threads or more: the last warp builds levels >= 3 and runs their conv
    // items while the other warps run the conv items of levels 1 and 2
    const bool split = a.split != 0 && L >= 3 && nt >= 128;
    const int nmain = split ? nt - 32 : nt;

    for (int u = u0; u < u1; ++u) {
        const int c = u / a.ngroups, grp = u - c * a.ngroups;
        const int p0 = grp * a.G, np = min(a.G, a.npairs - p0);
        if (c != cur_c) {  // a new channel: its kernels (nobody reads the old ones any more)
            stage_pair_weights<K>(a, c, wts);
            bias = a.with_bias ? a.base_scale[c] * a.base_bias[c] : 0.f;
            cur_c = c;
            __syncthreads();
        }
        if (a.tma) {
            if (tid == 0) copy_ok = mbar_wait(&bar, (uint32_t)(u - u0) & 1, a.timeout) ? 1 : 0;
            __syncthreads();
            if (!copy_ok) return;  // the flag is raised; this CTA's remaining outputs stay unwritten
        }
        // raw plane q of slot gs (staged copy, or global memory), null past B
        auto plane = [&](int gs, int q) -> const T * {
            const int b = 2 * (p0 + gs) + q;
            if (b >= B) return nullptr;
            return a.tma ? raw + (size_t)gs * raw_pair + q * HW : x + ((size_t)b * C + c) * HW;
        };
        // ---- pass 1: X and Haar levels 1 (and 2)
        if (L >= 2) pass1<4, T, FIX>(a, g, slots, np, plane);
        else pass1<2, T, FIX>(a, g, slots, np, plane);
        __syncthreads();
        if (a.tma && tid == 0 && u + 1 < u1) issue(u + 1);  // the raw planes are free
        // ---- conv items of every subband image of every level; levels 3 (and 4), then 5, are
        // built first, on the last warp when the CTA splits, else by every thread
        if (split) {
            if (tid >= nmain) {
#pragma unroll(FIX ? 2 : 1)
                for (int l0 = 3; l0 <= L; l0 += 2) {
                    analysis_deep_pass(g, slots, np, l0, L, nmain, 32);
                    __syncwarp();
                }
                if constexpr (FIX) {
                    conv_levels_fixed<K, Spec, 3>(a, g, slots, wts, np, 0, nmain, 32);
                } else {
                    conv_levels_dyn<K>(a, g, slots, wts, np, 3, L, nmain, 32);
                }
            } else {
                if constexpr (FIX) {
                    conv_levels_fixed<K, Spec, 1, (Spec::kL < 2 ? Spec::kL : 2)>(a, g, slots, wts, np, 0, 0, nmain);
                } else {
                    conv_levels_dyn<K>(a, g, slots, wts, np, 1, 2, 0, nmain);
                }
            }
        } else {
#pragma unroll(FIX ? 2 : 1)
            for (int l0 = 3; l0 <= L; l0 += 2) {
                analysis_deep_pass(g, slots, np, l0, L, 0, nt);
                __syncthreads();
            }
            if constexpr (FIX) {
                conv_levels_fixed<K, Spec, 1>(a, g, slots, wts, np, 0);
            } else {
                conv_levels_dyn<K>(a, g, slots, wts, np, 1, L, 0, nt);
            }
        }
        __syncthreads();
        // ---- levels >= 2 synthesised into the level-1 LL outputs (unless the output items add
        // them themselves: the shape-specialised instantiations with L >= 3 and 2-column items)
        constexpr bool kFold = fold_deep<Spec>();
        if (L >= 2 && !kFold) {
            const int w2 = g.w[2];
            const int zp1 = g.zpitch[1];
            const int n_gather = g.h[2] * w2;
            for (int t = tid; t < np * n_gather; t += nt) {
                const int gs = divq<FIX>(t, n_gather, a.dv_ngather), e = t - gs * n_gather;
                const int i2 = divq<FIX>(e, w2, a.dv_gw), j2 = e - i2 * w2;
                f2_t *slot = slots + (size_t)gs * g.slot;
                const f2_t *z2 = slot + g.off_z[2] + i2 * g.zpitch[2] + j2;
                const int zi2 = g.zimg[2];
                f2_t v = pk2(0.f, 0.f);
#pragma unroll(FIX ? kMaxLevels : 1)
                for (int l = 3; l <= L; ++l) {
                    const int sh = l - 2;
                    const f2_t *zl = slot + g.off_z[l] + (i2 >> sh) * g.zpitch[l] + (j2 >> sh);
                    const int zi = g.zimg[l];
                    const bool ra = (i2 >> (sh - 1)) & 1, cb = (j2 >> (sh - 1)) & 1;
                    const f2_t pp = ra ? fsub2(zl[0], zl[2 * zi]) : fadd2(zl[0], zl[2 * zi]);
                    const f2_t rr = ra ? fsub2(zl[zi], zl[3 * zi]) : fadd2(zl[zi], zl[3 * zi]);
                    v = fadd2(v, cb ? fsub2(pp, rr) : fadd2(pp, rr));
                }
                const f2_t t0 = fadd2(fadd2(z2[0], z2[2 * zi2]), v), t1 = fadd2(fsub2(z2[0], z2[2 * zi2]), v);
                const f2_t u0 = fadd2(z2[zi2], z2[3 * zi2]), u1 = fsub2(z2[zi2], z2[3 * zi2]);
                ulonglong2 *d = reinterpret_cast<ulonglong2 *>(slot + g.off_z[1] + (2 * i2) * zp1 + 2 * j2);
                ulonglong2 r0 = d[0];
                r0.x = fadd2(r0.x, fadd2(t0, u0));
                r0.y = fadd2(r0.y, fsub2(t0, u0));
                d[0] = r0;
                ulonglong2 *d1 = reinterpret_cast<ulonglong2 *>(slot + g.off_z[1] + (2 * i2 + 1) * zp1 + 2 * j2);
                ulonglong2 r1 = d1[0];
                r1.x = fadd2(r1.x, fadd2(t1, u1));
                r1.y = fadd2(r1.y, fsub2(t1, u1));
                d1[0] = r1;
            }
            __syncthreads();
        }
        // ---- output items: base conv + level-1 synthesis, one store per pixel
        const f2_t bias2 = pk2(bias, bias);
        const int Q0 = g.Q[0], S0 = g.S[0];
        if constexpr (FIX) {
            constexpr int kS0 = Spec::kH <= 4 ? 4 : Spec::kS0;
            out_phase<K, Spec::kQ0, kS0, T, true, Spec::kSkip, kFold>(a, g, slots, wts, np, p0, c, bias2, out);
        } else if (Q0 == 4) {
            if (S0 == 8) out_phase<K, 4, 8, T, FIX>(a, g, slots, wts, np, p0, c, bias2, out);
            else out_phase<K, 4, 4, T, FIX>(a, g, slots, wts, np, p0, c, bias2, out);
        } else {
            if (S0 == 8) out_phase<K, 2, 8, T, FIX>(a, g, slots, wts, np, p0, c, bias2, out);
            else out_phase<K, 2, 4, T, FIX>(a, g, slots, wts, np, p0, c, bias2, out);
        }
        __syncthreads();
    }
}

// Geometry of a kernel instantiation: the plan's at run time, or a shape fixed at compile time.
// A fixed geometry lives in a device constant the compiler folds wherever the index is known.
template <int K, int H, int W, int L, int Q0, int S0, int QL, int SL, int QD, int SD, int KIND>
__device__ constexpr PairGeo kPairSpecGeo = make_pair_geo(H, W, L, K, KIND, Q0, S0, QL, SL, QD, SD);

struct PairDynSpec {
    static constexpr bool fixed = false;
};
template <int H_, int W_, int L_, int Q0, int S0, int QL, int SL, int QD, int SD>
struct PairShapeSpec {
    static constexpr bool fixed = true;
    static constexpr int kH = H_, kW = W_, kL = L_;
    static constexpr int kQ0 = Q0, kS0 = S0, kQL = QL, kSL = SL, kQD = QD, kSD = SD;
    // planes of at most 16 x 16: the zero-padding rows of each window are a large share of it
    // (8 x 8, k = 5: 4 of 12 rows), so the items skip them.  On larger planes skipping measured
    // slower (64 x 64: 293 vs 259 us, 28 x 28: 64 vs 60 us): few windows touch the border
    static constexpr bool kSkip = H_ <= 16 && W_ <= 16;
    template <int K, int KIND>
    static __device__ __forceinline__ const PairGeo &geo() {
        return kPairSpecGeo<K, H_, W_, L_, Q0, S0, QL, SL, QD, SD, KIND>;
    }
};

// Resident CTAs the register budget is cut for: a shape-specialised instantiation of 128 threads
// at k = 5 fits four CTAs' shared memory (16 x 16 planes, four pairs), so it is held to 128
// registers (it needs about 122) rather than losing the fourth CTA to a few extra registers.
template <int K, int NT, class Spec>
constexpr int pair_fwd_min_blocks() {
    return NT == 64 ? (K <= 5 ? 6 : 4) : NT == 128 ? (K <= 3 ? 4 : (K == 5 ? (Spec::fixed ? 4 : 3) : 2)) : 1;
}

template <int K, typename T, int NT, class Spec>
__global__ void __launch_bounds__(NT, (pair_fwd_min_blocks<K, NT, Spec>()))
    wtconv_pair_fwd_kernel(const __grid_constant__ PairArgs a) {
    if constexpr (Spec::fixed) {
        pair_fwd_body<K, T, Spec>(a, Spec::template geo<K, 0>());
    } else {
        pair_fwd_body<K, T, Spec>(a, a.geo);
    }
}

template <int K, typename T, class Spec = PairDynSpec>
cudaError_t launch_pair_fwd_t(const PairArgs &a, size_t smem, cudaStream_t st) {
    auto kern = a.nthreads == 256  ? wtconv_pair_fwd_kernel<K, T, 256, Spec>
                : a.nthreads == 64 ? wtconv_pair_fwd_kernel<K, T, 64, Spec>
                                   : wtconv_pair_fwd_kernel<K, T, 128, Spec>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)a.grid), (unsigned)a.nthreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T, class Spec = PairDynSpec>
int occ_pair_fwd_t(size_t smem, int nthreads) {
    auto kern = nthreads == 256  ? wtconv_pair_fwd_kernel<K, T, 256, Spec>
                : nthreads == 64 ? wtconv_pair_fwd_kernel<K, T, 64, Spec>
                                 : wtconv_pair_fwd_kernel<K, T, 128, Spec>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, nthreads, smem) != cudaSuccess) return 0;
    return n;
}

}  // namespace wtconv
