// Batch-pair kernels of the WTConv layer: shared geometry and device building blocks.
//
// Every image these kernels keep in shared memory is a batch-pair image: position (i, j) holds
// the packed fp32 pair {v_b[i, j], v_b+1[i, j]} of two batch entries of the same channel.  The
// two planes share every kernel weight, so each k x k conv tap is one fma.rn.f32x2 with the
// duplicated weight {w, w}: no lane shuffles, no shifted copies, and the Haar butterflies and the
// synthesis run as packed adds over both planes at once.
//
// The method (paper "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation", Resumo Tecnico / Metodologia): the Haar pyramid is recomputed on chip from one
// read of the input, the learned scales are folded into the conv weights, and the multi-level
// synthesis is a closed form in which the level-l terms of output pixel (h, w) sit at
// (h >> l, w >> l) with signs set by bit l-1 of h and w.  The pyramid is kept unnormalised
// (Yhat^l = 2^l Y^l, exact), so the level-l kernels carry 4^-l and every synthesis term enters
// with a plain sign.
#pragma once

#include "wtconv_device.cuh"

namespace wtconv {

constexpr int kPairMaxThreads = 256;  // threads per CTA of the batch-pair kernels: 64, 128 or 256
constexpr int kPairMaxSlots = 64;     // pair slots per CTA group

// Shared-memory geometry of one pair slot, in packed pairs (f2, 8 bytes).
//
// Level 0 is the full-resolution plane pair.  Level l >= 1 has four subband images (LL, LH, HL,
// HH).  A conv runs on strip items: Q output columns x S output rows, sliding down the rows of a
// zero-padded input image whose interior starts at (P, P), P = K/2.  Image extents are rounded up
// to whole items (ns strips x ng segments) plus the K-1 halo; row pitches are even, so every
// window row starts 16-byte aligned.  Conv outputs are compact (pitch Q*ns).
struct PairGeo {
    int H, W, L, K, P;
    int kind;                                       // 0: forward slot, 1: weight-gradient slot
    int h[kMaxLevels + 1], w[kMaxLevels + 1];       // interior size per level
    int Q[kMaxLevels + 1], S[kMaxLevels + 1];       // item columns / rows per level (level 0: base)
    int ns[kMaxLevels + 1], ng[kMaxLevels + 1];     // strips per row, segments per image
    int ipitch[kMaxLevels + 1], irows[kMaxLevels + 1], iimg[kMaxLevels + 1];  // padded inputs
    int zpitch[kMaxLevels + 1], zrows[kMaxLevels + 1], zimg[kMaxLevels + 1];  // compact images
    // offsets (pairs) inside a slot: level 0 padded input (x) and compact image (dy, weight
    // gradient only); level l subband s padded input at off_y[l] + s * iimg[l], compact image
    // (forward: conv output Z; weight gradient: the dy pyramid) at off_z[l] + s * zimg[l]
    int off_x, off_dy, off_y[kMaxLevels + 1], off_z[kMaxLevels + 1];
    int slot;                                       // pairs per slot (even)
};

__host__ __device__ constexpr inline int pg_round2(int v) { return (v + 1) & ~1; }

// q0 / s0: item shape of the base path; ql / sl: of level 1; qd / sd: of the levels >= 2 (rows per
// item drop to 4 on images of at most 4 rows).
__host__ __device__ constexpr inline PairGeo make_pair_geo(int H, int W, int L, int K, int kind, int q0, int s0, int ql,
                                                 int sl, int qd, int sd) {
    PairGeo g = {};
    g.H = H; g.W = W; g.L = L; g.K = K; g.P = K / 2; g.kind = kind;
    int off = 0;
    for (int l = 0; l <= L; ++l) {
        g.h[l] = H >> l;
        g.w[l] = W >> l;
        g.Q[l] = l == 0 ? q0 : (l == 1 ? ql : qd);
        const int s = l == 0 ? s0 : (l == 1 ? sl : sd);
        g.S[l] = g.h[l] <= 4 ? 4 : s;
        g.ns[l] = (g.w[l] + g.Q[l] - 1) / g.Q[l];
        g.ng[l] = (g.h[l] + g.S[l] - 1) / g.S[l];
        g.ipitch[l] = pg_round2(g.Q[l] * g.ns[l] + K - 1);
        g.irows[l] = g.ng[l] * g.S[l] + K - 1;
        g.iimg[l] = g.ipitch[l] * g.irows[l];
        g.zpitch[l] = pg_round2(g.Q[l] * g.ns[l]);
        g.zrows[l] = g.ng[l] * g.S[l];
        g.zimg[l] = g.zpitch[l] * g.zrows[l];
    }
    g.off_y[0] = g.off_z[0] = -1;
    g.off_dy = -1;
    g.off_x = off;
    off += g.iimg[0];
    if (kind == 1) { g.off_dy = off; off += g.zimg[0]; }
    for (int l = 1; l <= L; ++l) { g.off_y[l] = off; off += 4 * g.iimg[l]; }
    for (int l = 1; l <= L; ++l) { g.off_z[l] = off; off += 4 * g.zimg[l]; }
    g.slot = pg_round2(off);
    return g;
}

// Per-pair work of the batch-pair kernels and their launch shape (host planner output).
struct PairArgs {
    int B, C, H, W, L, K;
    int npairs;             // ceil(B / 2)
    int G;                  // pair slots per group
    int ngroups;            // groups per channel: ceil(npairs / G)
    int chunk_groups;       // groups per work unit (weight gradient: one partial per unit)
    int nchunks;            // work units per channel: ceil(ngroups / chunk_groups)
    int units;              // C * nchunks; unit u is channel u / nchunks, chunk u % nchunks
    int grid;               // CTAs (persistent): CTA i takes units [i*units/grid, (i+1)*units/grid)
    int nthreads;           // CTA size: 64, 128 or 256
    int nb;                 // partials per (channel, signal, tap) = nchunks
    int tma;                // 1: planes arrive by bulk copies into the raw staging area
    int raw_pair_bytes;     // raw bytes of one pair slot (two planes, or four for the weight gradient)
    int vec_st;             // 1: rows allow 4-element vector stores / loads of activations
    int spec;               // >= 0: the shape-specialised instantiation of this index runs (else -1)
    int split;              // forward, L >= 3, 128 threads or more: the last warp builds and convolves
                            // levels >= 3 while the others convolve levels 1 and 2
    int tma_map;            // 1: a group's planes arrive as one tensor copy per activation (tmap_x,
                            // tmap_dy: each plane viewed as tma_rows rows of tma_rlen elements, box
                            // tma_rlen x tma_rows x 1 x 2G at (0, 0, channel, first batch entry));
                            // 0: one bulk copy per plane
    int tma_rlen, tma_rows;
    const void *x;          // forward: x; input gradient: dy; weight gradient: x
    const void *dy;         // weight gradient: dy
    void *out;              // y or dx
    const float *base_w, *base_bias, *base_scale, *wavelet_w, *wavelet_scale;
    float *partials;        // weight gradient: [nb][C][1+4L][K*K+1]
    int flip, with_bias;
    int *timeout;
    int n_a;                // analysis blocks per pair of the first pass
    int n_conv;             // conv items per pair (levels 1 .. L, four subbands each)
    int conv_start[kMaxLevels + 2];  // first conv item of level l (l = 1 .. L), then n_conv
    int n_gather;           // level-2 positions per pair (L >= 2)
    int n_out;              // output items per pair
    // weight gradient: correlation signal of each thread range and the items each thread takes
    int sig_start[1 + 4 * kMaxLevels + 1];  // first thread of signal sig (0 base, 1 + 4(l-1) + s), then the end
    int per_thread;         // items per thread per group
    FastDiv dv_na, dv_naw, dv_nconv, dv_nout, dv_out_ns, dv_ngather;
    FastDiv dv_lvl[kMaxLevels + 1], dv_lvl_ns[kMaxLevels + 1];  // items per subband image, strips per row
    FastDiv dv_gw;          // level-2 positions per row
    FastDiv dv_xn, dv_xw;   // X build: two-pixel steps per plane, per row
    PairGeo geo;
    CUtensorMap tmap_x, tmap_dy;
};

// Per activation type T (float, __nv_bfloat16, __half), defined in that type's translation unit.
template <typename T> cudaError_t launch_pair_fwd_typed(const PairArgs &a, size_t smem, cudaStream_t st);
template <typename T> int occupancy_pair_fwd_typed(int K, size_t smem, int nthreads);
template <typename T> cudaError_t launch_pair_dw_typed(const PairArgs &a, size_t smem, cudaStream_t st);
template <typename T> int occupancy_pair_dw_typed(int K, size_t smem, int nthreads);

// Index of the shape-specialised instantiation for this layer shape and item shapes (q0, s0, ql,
// sl, qd, sd), or -1; and its occupancy.
int pair_spec_index(int H, int W, int L, int K, int dtype, const int (&shape)[6]);
int occupancy_pair_fwd_spec(int spec, size_t smem, int nthreads);

// What measured fastest on GB300 for a layer shape that has a specialised instantiation: its item
// shapes, the forward's CTA size and pair slots per group (0: the planner's choice), whether
// the batch-pair forward / weight gradient is the default for the shape, and the weight
// gradient's CTA size (0: planner) and item-shape index (-1: planner).
struct PairSpecPref {
    int shape[6];
    int threads, slots, fwd_default, dw_default, dw_threads, dw_shape;
};
bool pair_spec_measured(int H, int W, int L, int K, int dtype, PairSpecPref *pref);

size_t pair_fwd_smem_bytes(const PairArgs &a, int elem_bytes);
cudaError_t launch_pair_fwd(const PairArgs &a, int dtype, size_t smem, cudaStream_t st);
int occupancy_pair_fwd(int dtype, int K, size_t smem, int nthreads);
size_t pair_dw_smem_bytes(const PairArgs &a, int elem_bytes);
cudaError_t launch_pair_dw(const PairArgs &a, int dtype, size_t smem, cudaStream_t st);
int occupancy_pair_dw(int dtype, int K, size_t smem, int nthreads);

#ifdef __CUDACC__

// Bulk copy (no tensor map) of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            (uint32_t)__cvta_generic_to_shared(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"((uint32_t)__cvta_generic_to_shared(bar))
        : "memory");
}

// Stage channel c's kernels as duplicated pairs {w, w}, scales folded in: set 0 is the base
// kernel s_b[c] * w_b[c]; set 1 + 4(l-1) + s is level l subband s, 4^-l * s_l[4c+s] * w_l[4c+s]
// (4^-l: unnormalised pyramid).  `flip` rotates every kernel by 180 degrees (input gradient).
template <int K>
__device__ __forceinline__ void stage_pair_weights(const PairArgs &a, int c, f2_t *wts) {
    constexpr int KK = K * K, WP = wpairs(K);
    const int nset = 1 + 4 * a.L;
    for (int it = threadIdx.x; it < nset * KK; it += blockDim.x) {
        const int ci = it / KK, t = it - ci * KK;
        const int src_t = a.flip ? KK - 1 - t : t;
        float v;
        if (ci == 0) {
            v = a.base_scale[c] * a.base_w[(size_t)c * KK + src_t];
        } else {
            const int l = (ci - 1) / 4 + 1, s = (ci - 1) & 3;
            const size_t ch = (size_t)(l - 1) * 4 * a.C + 4 * c + s;
            v = ldexpf(a.wavelet_scale[ch] * a.wavelet_w[ch * KK + src_t], -2 * l);
        }
        wts[ci * WP + t] = pk2(v, v);
    }
}

// Conv strip: out[j][q] = sum_{u,v} w[u][v] * in[j + u][q + v] (plus `init` on every output when
// kInit), j < S, q < Q.  `in` points at the window origin of the padded image (pitch in pairs, even;
// origin 16-byte aligned), `out` at the compact output (pitch even).  The window slides down one
// input row at a time; each loaded row feeds the (up to K) output rows whose window contains it,
// so only about K x Q accumulators are live at once.
//
// SKIP: the first zt and the last zb window rows are known to be zero padding (small planes,
// where they are a large share of the window): those rows are neither loaded nor multiplied.
template <int K, int Q, int S, bool SKIP = false>
__device__ __forceinline__ void pair_conv_strip(const f2_t *__restrict__ in, int pitch, const f2_t (&w)[K * K],
                                                f2_t *__restrict__ out, int opitch, int zt = 0, int zb = 0) {
    constexpr int NW = Q + K - 1, NL = (NW + 1) / 2;
    f2_t acc[S][Q];
    if constexpr (SKIP) {
#pragma unroll
        for (int j = 0; j < S; ++j)
#pragma unroll
            for (int q = 0; q < Q; ++q) acc[j][q] = 0ull;
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
                        if (!SKIP && u == 0 && v == 0) acc[j][q] = fmul2(w[0], x[q]);
                        else ffma2_acc(acc[j][q], w[u * K + v], x[q + v]);
                    }
                }
            }
        }
        const int jd = i - (K - 1);
        if (jd >= 0) {
            ulonglong2 *o = reinterpret_cast<ulonglong2 *>(out + jd * opitch);
#pragma unroll
            for (int t = 0; t < Q / 2; ++t) {
                ulonglong2 v;
                v.x = acc[jd][2 * t];
                v.y = acc[jd][2 * t + 1];
                o[t] = v;
            }
        }
    }
}

// Correlation strip of the weight gradient: acc[u*K+v] += sum_{j<S, q<Q} g[j][q] * y[j + u][q + v]
// (elementwise on the pair: the two halves are partial sums over the two planes).  `y` points at
// the window origin of the padded image, `g` at the matching interior origin of the compact image.
// The first zt and the last zb window rows of y may be declared zero padding (rows outside the
// plane): they are neither loaded nor multiplied, which leaves the sums exact.
template <int K, int Q, int S>
__device__ __forceinline__ void pair_corr_strip(const f2_t *__restrict__ y, int ypitch, const f2_t *__restrict__ g,
                                                int gpitch, f2_t (&acc)[K * K], int zt = 0, int zb = 0) {
    constexpr int NW = Q + K - 1, NL = (NW + 1) / 2;
    f2_t gr[S][Q];
#pragma unroll
    for (int r = 0; r < S + K - 1; ++r) {
        if (r < S) {
            const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(g + r * gpitch);
#pragma unroll
            for (int t = 0; t < Q / 2; ++t) {
                const ulonglong2 v = p[t];
                gr[r][2 * t] = v.x;
                gr[r][2 * t + 1] = v.y;
            }
        }
        if (r < zt || r >= S + K - 1 - zb) continue;
        f2_t x[2 * NL];
        const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(y + r * ypitch);
#pragma unroll
        for (int t = 0; t < NL; ++t) {
            const ulonglong2 v = p[t];
            x[2 * t] = v.x;
            x[2 * t + 1] = v.y;
        }
#pragma unroll
        for (int q = 0; q < Q; ++q)
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int i = r - u;
                if (i >= 0 && i < S) {
#pragma unroll
                    for (int v = 0; v < K; ++v) ffma2_acc(acc[u * K + v], gr[i][q], x[q + v]);
                }
            }
    }
}

// Unnormalised 2x2 butterfly on pairs: [[a, b], [c, d]] -> LL = a+b+c+d, LH = a-b+c-d,
// HL = a+b-c-d, HH = a-b-c+d (the page-4 filter signs; row bit selects HL, column bit LH).
struct QuadP { f2_t ll, lh, hl, hh; };
__device__ __forceinline__ QuadP butterfly2(f2_t a, f2_t b, f2_t c, f2_t d) {
    const f2_t st = fadd2(a, b), dt = fsub2(a, b), sb = fadd2(c, d), db = fsub2(c, d);
    return {fadd2(st, sb), fadd2(dt, db), fsub2(st, sb), fsub2(dt, db)};
}

// Two activations of type T at p (p[0], p[1]) to fp32.
template <typename T>
__device__ __forceinline__ void ld2f(const T *p, float &v0, float &v1) {
    v0 = Act<T>::ld(p);
    v1 = Act<T>::ld(p + 1);
}

#endif  // __CUDACC__

}  // namespace wtconv
