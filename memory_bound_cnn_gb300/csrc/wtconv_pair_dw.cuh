// Batch-pair weight-gradient kernel of the WTConv layer:
//     dw'_b[u, v]   = sum_{b,h,w} dy[b, h, w] x[b, h+u-P, w+v-P],   db' = sum dy      (base path)
//     dW'^l_s[u, v] = sum_{b,i,j} Ghat^l_s[b, i, j] Yhat^l_s[b, i+u-P, j+v-P]        (level l, subband s)
// with Yhat / Ghat the unnormalised Haar pyramids of x / dy and zero padding outside each plane
// (paper, Principais Contribuicoes: all parameter gradients from the same on-chip pyramids).
//
// A CTA owns channel c and walks through groups of G batch pairs of that channel.  Per group the
// raw planes of x and dy arrive by bulk copies; one analysis pass gives the interleaved padded
// copy of x, the compact copy of dy and Haar levels 1 and 2 of both; later passes build the
// deeper levels.  Every thread is pinned, for the whole CTA, to one correlation signal (the base
// path, or one subband of one level) and a fixed share of that signal's strip items, and keeps its
// k*k tap sums (packed pairs: partial sums of the two planes) in registers across all groups.  At
// the end the tap sums are reduced in a fixed thread order into one partial per (channel,
// signal, tap): deterministic, no atomics.
#pragma once

#include "wtconv_pair.cuh"

namespace wtconv {

namespace {

struct PairDwLayout {
    size_t slots, raw, red, total;  // byte offsets from a 128-byte aligned base
};

// Bytes of one activation's raw planes of a group (2G planes, 128-byte rounded).
__host__ __device__ inline size_t pair_dw_raw_half(const PairArgs &a) {
    return ((size_t)a.G * a.raw_pair_bytes / 2 + 127) / 128 * 128;
}

// Slots, then the raw staging area (the next group's copies land there while the current group
// is worked on), then the reduction buffer of the per-unit flush (one row of k*k+1 floats per
// thread).
__host__ __device__ inline PairDwLayout pair_dw_layout(const PairArgs &a) {
    PairDwLayout p;
    size_t o = 0;
    p.slots = o;
    o += (size_t)a.G * a.geo.slot * sizeof(f2_t);
    o = (o + 127) / 128 * 128;
    p.raw = o;  // x planes of the group, then (128-byte aligned) its dy planes
    if (a.tma) o += 2 * pair_dw_raw_half(a);
    p.red = o;
    o += (size_t)a.nthreads * (a.K * a.K + 1) * sizeof(float);
    p.total = o + 128;
    return p;
}

template <int K>
__device__ __forceinline__ void corr_item_dispatch(int q, int s, const f2_t *y, int ypitch, const f2_t *g, int gpitch,
                                                   f2_t (&acc)[K * K], int zt, int zb) {
    if (q == 4) {
        if (s == 8) pair_corr_strip<K, 4, 8>(y, ypitch, g, gpitch, acc, zt, zb);
        else pair_corr_strip<K, 4, 4>(y, ypitch, g, gpitch, acc, zt, zb);
    } else {
        if (s == 8) pair_corr_strip<K, 2, 8>(y, ypitch, g, gpitch, acc, zt, zb);
        else if (s == 7) pair_corr_strip<K, 2, 7>(y, ypitch, g, gpitch, acc, zt, zb);  // planes of 7 * 2^l rows
        else pair_corr_strip<K, 2, 4>(y, ypitch, g, gpitch, acc, zt, zb);
    }
}

// Deeper analysis pass of both pyramids: levels l0 (and l0+1) of x (padded images) and of dy
// (compact images) from the level l0-1 low bands.
__device__ __forceinline__ void dw_deep_pass(const PairGeo &g, f2_t *slots, int np, int l0, int L) {
    const bool two = l0 + 1 <= L;
    const int hs = g.h[l0 - 1], ws = g.w[l0 - 1];
    const int bsz = two ? 4 : 2;
    const int bw = ws / bsz, n = (hs / bsz) * bw;
    const int P = g.P;
    for (int t = threadIdx.x; t < 2 * np * n; t += blockDim.x) {
        const int sgl = t / (np * n), tt = t - sgl * (np * n);  // 0: x pyramid, 1: dy pyramid
        const int gs = tt / n, e = tt - gs * n;
        const int bi = e / bw, bj = e - bi * bw;
        f2_t *slot = slots + (size_t)gs * g.slot;
        // source low band and destination images of this signal
        const int sp = sgl ? g.zpitch[l0 - 1] : g.ipitch[l0 - 1];
        const int so = sgl ? 0 : P;
        const f2_t *src = slot + (sgl ? g.off_z[l0 - 1] : g.off_y[l0 - 1]) + (bsz * bi + so) * sp + bsz * bj + so;
        const int dp0 = sgl ? g.zpitch[l0] : g.ipitch[l0], di0 = sgl ? g.zimg[l0] : g.iimg[l0];
        f2_t *y0 = slot + (sgl ? g.off_z[l0] : g.off_y[l0]);
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
                    f2_t *d = y0 + (2 * bi + a2 + so) * dp0 + 2 * bj + b2 + so;
                    d[0] = q[a2][b2].ll;
                    d[di0] = q[a2][b2].lh;
                    d[2 * di0] = q[a2][b2].hl;
                    d[3 * di0] = q[a2][b2].hh;
                }
            const QuadP q2 = butterfly2(q[0][0].ll, q[0][1].ll, q[1][0].ll, q[1][1].ll);
            const int dp1 = sgl ? g.zpitch[l0 + 1] : g.ipitch[l0 + 1], di1 = sgl ? g.zimg[l0 + 1] : g.iimg[l0 + 1];
            f2_t *d = slot + (sgl ? g.off_z[l0 + 1] : g.off_y[l0 + 1]) + (bi + so) * dp1 + bj + so;
            d[0] = q2.ll;
            d[di1] = q2.lh;
            d[2 * di1] = q2.hl;
            d[3 * di1] = q2.hh;
        } else {
            const QuadP q = butterfly2(src[0], src[1], src[sp], src[sp + 1]);
            f2_t *d = y0 + (bi + so) * dp0 + bj + so;
            d[0] = q.ll;
            d[di0] = q.lh;
            d[2 * di0] = q.hl;
            d[3 * di0] = q.hh;
        }
    }
}

// First analysis pass of one BS x BS block (BS = 4: levels 1 and 2; BS = 2: level 1) of both
// planes of a pair: x goes to the padded copy X (interior at (P, P)) and its padded pyramid, dy to
// the compact copy DY and its compact pyramid (and into the running sum of dy).  plane[q] is null
// for a batch entry past B (zeros).
template <int BS, typename T>
__device__ __forceinline__ void dw_pass1_block(const PairGeo &g, f2_t *slot, const T *const (&plane)[2], int W, int bi,
                                               int bj, int sgl, f2_t &dysum) {
    float v[2][BS][BS];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        if (plane[q]) {
            const T *src = plane[q] + (size_t)(BS * bi) * W + BS * bj;
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
    f2_t X[BS][BS];
#pragma unroll
    for (int r = 0; r < BS; ++r)
#pragma unroll
        for (int cc = 0; cc < BS; ++cc) X[r][cc] = pk2(v[0][r][cc], v[1][r][cc]);
    const int P = g.P;
    const int xp = sgl ? g.zpitch[0] : g.ipitch[0];
    const int so = sgl ? 0 : P;
    f2_t *xd = slot + (sgl ? g.off_dy : g.off_x) + (BS * bi + so) * xp + BS * bj + so;
#pragma unroll
    for (int r = 0; r < BS; ++r)
#pragma unroll
        for (int cc = 0; cc < BS; ++cc) xd[r * xp + cc] = X[r][cc];
    if (sgl) {
#pragma unroll
        for (int r = 0; r < BS; ++r)
#pragma unroll
            for (int cc = 0; cc < BS; ++cc) dysum = fadd2(dysum, X[r][cc]);
    }
    const int p1 = sgl ? g.zpitch[1] : g.ipitch[1], i1 = sgl ? g.zimg[1] : g.iimg[1];
    f2_t *y1 = slot + (sgl ? g.off_z[1] : g.off_y[1]);
    if constexpr (BS == 4) {
        QuadP q1[2][2];
#pragma unroll
        for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
            for (int b2 = 0; b2 < 2; ++b2) {
                q1[a2][b2] = butterfly2(X[2 * a2][2 * b2], X[2 * a2][2 * b2 + 1], X[2 * a2 + 1][2 * b2],
                                        X[2 * a2 + 1][2 * b2 + 1]);
                f2_t *d = y1 + (2 * bi + a2 + so) * p1 + 2 * bj + b2 + so;
                d[0] = q1[a2][b2].ll;
                d[i1] = q1[a2][b2].lh;
                d[2 * i1] = q1[a2][b2].hl;
                d[3 * i1] = q1[a2][b2].hh;
            }
        const QuadP q2 = butterfly2(q1[0][0].ll, q1[0][1].ll, q1[1][0].ll, q1[1][1].ll);
        const int p2 = sgl ? g.zpitch[2] : g.ipitch[2], i2 = sgl ? g.zimg[2] : g.iimg[2];
        f2_t *d = slot + (sgl ? g.off_z[2] : g.off_y[2]) + (bi + so) * p2 + bj + so;
        d[0] = q2.ll;
        d[i2] = q2.lh;
        d[2 * i2] = q2.hl;
        d[3 * i2] = q2.hh;
    } else {
        const QuadP q1 = butterfly2(X[0][0], X[0][1], X[1][0], X[1][1]);
        f2_t *d = y1 + (bi + so) * p1 + bj + so;
        d[0] = q1.ll;
        d[i1] = q1.lh;
        d[2 * i1] = q1.hl;
        d[3 * i1] = q1.hh;
    }
}

}  // namespace

template <int K, typename T, int NT>
__global__ void __launch_bounds__(NT, NT == 64 ? (K <= 5 ? 6 : 4) : NT == 128 ? (K <= 3 ? 4 : (K == 5 ? 3 : 2)) : 1)
    wtconv_pair_dw_kernel(const __grid_constant__ PairArgs a) {
    constexpr int P = K / 2, KK = K * K, NA = KK + 1;
    extern __shared__ __align__(128) unsigned char pair_smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int copy_ok;
    const uint32_t s0 = (uint32_t)__cvta_generic_to_shared(pair_smem);
    unsigned char *base = pair_smem + (((s0 + 127u) & ~127u) - s0);
    const PairDwLayout lay = pair_dw_layout(a);
    const PairGeo &g = a.geo;
    f2_t *slots = reinterpret_cast<f2_t *>(base + lay.slots);
    float *red = reinterpret_cast<float *>(base + lay.red);
    const int tid = threadIdx.x, nt = blockDim.x;
    const int B = a.B, C = a.C, H = a.H, W = a.W, L = a.L;
    const size_t HW = (size_t)H * W;
    const T *xg = static_cast<const T *>(a.x);
    const T *dyg = static_cast<const T *>(a.dy);
    const int nsig = 1 + 4 * L;

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

    // this thread's signal: 0 base, 1 + 4(l-1) + s level l subband s; -1 none
    int sig = -1;
    for (int k = 0; k < nsig; ++k)
        if (tid >= a.sig_start[k] && tid < a.sig_start[k + 1]) sig = k;
    const int lvl = sig <= 0 ? 0 : (sig - 1) / 4 + 1, sub = sig <= 0 ? 0 : (sig - 1) & 3;
    const int t_in = sig < 0 ? 0 : tid - a.sig_start[sig];
    const int nthr = sig < 0 ? 1 : a.sig_start[sig + 1] - a.sig_start[sig];
    const int per_pair = g.ns[lvl] * g.ng[lvl];
    const int ipitch = g.ipitch[lvl], zpitch = g.zpitch[lvl];
    const int Ql = g.Q[lvl], Sl = g.S[lvl], hl = g.h[lvl];
    const int yoff = lvl == 0 ? g.off_x : g.off_y[lvl] + sub * g.iimg[lvl];
    const int goff = lvl == 0 ? g.off_dy : g.off_z[lvl] + sub * g.zimg[lvl];
    const FastDiv dv_pp = a.dv_lvl[lvl], dv_ns = a.dv_lvl_ns[lvl];

    // this CTA's work units: (channel, chunk of groups), channel-major; one partial per unit
    const int u0 = (int)((long long)blockIdx.x * a.units / a.grid);
    const int u1 = (int)((long long)(blockIdx.x + 1) * a.units / a.grid);
    auto first_group = [&](int u) { return (u % a.nchunks) * a.chunk_groups; };
    auto end_group = [&](int u) { return min(a.ngroups, first_group(u) + a.chunk_groups); };
    auto raw_of = [&](int gs, int which) -> T * {  // which: 0 x, 1 dy; two planes each
        return reinterpret_cast<T *>(base + lay.raw + (size_t)which * pair_dw_raw_half(a)) + (size_t)gs * 2 * HW;
    };
    auto issue = [&](int cu, int grp) {  // thread 0: the copies of group grp of channel cu
        const int p0 = grp * a.G, np = min(a.G, a.npairs - p0);
        const uint32_t pb = (uint32_t)(HW * sizeof(T));
        if (a.tma_map) {  // one copy per activation of the 2G planes (zero past B; whole boxes)
            mbar_arrive_expect_tx(&bar, (uint32_t)(4 * a.G) * pb);
            tma_load_4d(raw_of(0, 0), &a.tmap_x, 0, 0, cu, 2 * p0, &bar);
            tma_load_4d(raw_of(0, 1), &a.tmap_dy, 0, 0, cu, 2 * p0, &bar);
            return;
        }
        uint32_t bytes = 0;
        for (int gs = 0; gs < np; ++gs)
            for (int q = 0; q < 2; ++q)
                if (2 * (p0 + gs) + q < B) bytes += 2 * pb;
        mbar_arrive_expect_tx(&bar, bytes);
        for (int gs = 0; gs < np; ++gs)
            for (int q = 0; q < 2; ++q) {
                const int b = 2 * (p0 + gs) + q;
                if (b < B) {
                    bulk_load(raw_of(gs, 0) + q * HW, xg + ((size_t)b * C + cu) * HW, pb, &bar);
                    bulk_load(raw_of(gs, 1) + q * HW, dyg + ((size_t)b * C + cu) * HW, pb, &bar);
                }
            }
    };
    if (a.tma && tid == 0 && u0 < u1) issue(u0 / a.nchunks, first_group(u0));
    uint32_t step = 0;  // copies waited for so far (mbarrier phase parity)

    for (int u = u0; u < u1; ++u) {
        const int c = u / a.nchunks, chunk = u - c * a.nchunks;
        f2_t acc[KK];
#pragma unroll
        for (int i = 0; i < KK; ++i) acc[i] = 0ull;
        f2_t dysum = 0ull;
        const int ge = end_group(u);
        for (int grp = first_group(u); grp < ge; ++grp, ++step) {
            const int p0 = grp * a.G, np = min(a.G, a.npairs - p0);
            if (a.tma) {
                if (tid == 0) copy_ok = mbar_wait(&bar, step & 1, a.timeout) ? 1 : 0;
                __syncthreads();
                if (!copy_ok) {
                    // a copy never arrived (the flag is raised): mark this CTA's partials as
                    // invalid so the gradients come out as NaN, and leave without touching the
                    // copy's destination
                    for (int uu = u; uu < u1; ++uu) {
                        const int cc = uu / a.nchunks, ch = uu - cc * a.nchunks;
                        float *pp = a.partials + ((size_t)ch * C + cc) * nsig * NA;
                        for (int i = tid; i < nsig * NA; i += nt) pp[i] = __int_as_float(0x7fc00000);
                    }
                    return;
                }
            }
            // ---- pass 1: x -> X and levels 1 (and 2) of its pyramid; dy -> DY and levels 1 (and 2)
            for (int t = tid; t < 2 * np * a.n_a; t += nt) {
                const int sgl = t >= np * a.n_a;  // 0: x, 1: dy
                const int tt = t - sgl * np * a.n_a;
                const int gs = (int)fdiv(a.dv_na, (uint32_t)tt), blk = tt - gs * a.n_a;
                const int bi = (int)fdiv(a.dv_naw, (uint32_t)blk);
                f2_t *slot = slots + (size_t)gs * g.slot;
                const T *plane[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int b = 2 * (p0 + gs) + q;
                    plane[q] = b >= B ? nullptr
                               : a.tma ? raw_of(gs, sgl) + q * HW
                                       : (sgl ? dyg : xg) + ((size_t)b * C + c) * HW;
                }
                if (L >= 2) {
                    const int bj = blk - bi * (W >> 2);
                    dw_pass1_block<4, T>(g, slot, plane, W, bi, bj, sgl, dysum);
                } else {
                    const int bj = blk - bi * (W >> 1);
                    dw_pass1_block<2, T>(g, slot, plane, W, bi, bj, sgl, dysum);
                }
            }
            __syncthreads();
            if (a.tma && tid == 0) {  // the raw planes are free: the next group's copies
                if (grp + 1 < ge) issue(c, grp + 1);
                else if (u + 1 < u1) issue((u + 1) / a.nchunks, first_group(u + 1));
            }
            for (int l0 = 3; l0 <= L; l0 += 2) {
                dw_deep_pass(g, slots, np, l0, L);
                __syncthreads();
            }
            // ---- correlation items of this thread's signal
            if (sig >= 0) {
                const int nitems = np * per_pair;
                for (int k = 0; k < a.per_thread; ++k) {
                    const int e = t_in + k * nthr;
                    if (e >= nitems) break;
                    const int gs = (int)fdiv(dv_pp, (uint32_t)e), rem = e - gs * per_pair;
                    const int seg = (int)fdiv(dv_ns, (uint32_t)rem), strip = rem - seg * g.ns[lvl];
                    const f2_t *slot = slots + (size_t)gs * g.slot;
                    const f2_t *yw = slot + yoff + seg * Sl * ipitch + strip * Ql;
                    const f2_t *gw = slot + goff + seg * Sl * zpitch + strip * Ql;
                    // window rows of y outside the plane: zero padding, skipped
                    const int zt = max(0, P - seg * Sl), zb = max(0, (seg + 1) * Sl + P - hl);
                    corr_item_dispatch<K>(Ql, Sl, yw, ipitch, gw, zpitch, acc, zt, zb);
                }
            }
            __syncthreads();
        }

        // ---- flush: per thread the two planes' partial sums of each tap, then per signal the sum
        // over its threads in thread order -> this unit's partial
        if (sig >= 0) {
#pragma unroll
            for (int i = 0; i < KK; ++i) red[tid * NA + i] = lo2(acc[i]) + hi2(acc[i]);
        } else {
#pragma unroll
            for (int i = 0; i < KK; ++i) red[tid * NA + i] = 0.f;
        }
        red[tid * NA + KK] = lo2(dysum) + hi2(dysum);
        __syncthreads();
        float *pp = a.partials + ((size_t)chunk * C + c) * nsig * NA;
        for (int i = tid; i < nsig * NA; i += nt) {
            const int s = i / NA, tap = i - s * NA;
            float v = 0.f;
            if (tap < KK) {
                for (int t = a.sig_start[s]; t < a.sig_start[s + 1]; ++t) v += red[t * NA + tap];
            } else if (s == 0) {
                for (int t = 0; t < nt; ++t) v += red[t * NA + KK];
            }
            pp[i] = v;
        }
        __syncthreads();
    }
}

template <int K, typename T>
cudaError_t launch_pair_dw_t(const PairArgs &a, size_t smem, cudaStream_t st) {
    auto kern = a.nthreads == 256  ? wtconv_pair_dw_kernel<K, T, 256>
                : a.nthreads == 64 ? wtconv_pair_dw_kernel<K, T, 64>
                                   : wtconv_pair_dw_kernel<K, T, 128>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)a.grid), (unsigned)a.nthreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
int occ_pair_dw_t(size_t smem, int nthreads) {
    auto kern = nthreads == 256  ? wtconv_pair_dw_kernel<K, T, 256>
                : nthreads == 64 ? wtconv_pair_dw_kernel<K, T, 64>
                                 : wtconv_pair_dw_kernel<K, T, 128>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, nthreads, smem) != cudaSuccess) return 0;
    return n;
}

}  // namespace wtconv
