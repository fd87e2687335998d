// Internal types shared by the host entry points (wtconv_api.cu) and the kernel translation
// units (wtconv_fwd.cu, wtconv_bwd.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace wtconv {

constexpr int kMaxThreads = 256;  // threads per CTA: 128 or 256, chosen per shape
constexpr int kMaxLevels = 5;
constexpr int kMaxSig = 1 + 4 * kMaxLevels;  // base kernel + 4 subbands per level
constexpr int kRows = 8;        // output rows of one sliding-window conv item
constexpr int kCols = 4;        // output columns of one conv item
constexpr int kMaxSmem = 227 * 1024;

__host__ __device__ constexpr int round_up(int a, int m) { return (a + m - 1) / m * m; }
__host__ __device__ constexpr int ceil_div(int a, int m) { return (a + m - 1) / m; }
// packed weight pairs per staged kernel (16-byte aligned)
__host__ __device__ constexpr int wpairs(int K) { return round_up(K * K, 2); }
constexpr int kColsL = 2;       // output positions (subband pairs) of one level conv item

// Shared-memory geometry of one plane slot, in floats.
//
// Level 0 is the full-resolution plane, one fp32 image.  Each Haar level l >= 1 is stored as two
// "pair images": pair 0 interleaves subbands (LL, LH), pair 1 interleaves (HL, HH), so every
// position holds two floats that a packed f32x2 instruction consumes together.
//
// Conv inputs are zero-padded: interior origin (P, P), P = K/2 (in pixels, or in positions for
// pair images), extents rounded up to whole conv items plus the K-1 halo, rows 16-byte aligned.
// Conv outputs (the base buffer, and Z^l as pair images) are compact.
struct Geo {
    int H, W, L, K, P;
    int h[kMaxLevels + 1], w[kMaxLevels + 1];          // interior size per level
    int rseg[kMaxLevels + 1], cstr[kMaxLevels + 1];    // conv items per image: row segments x col strips
    int pitch[kMaxLevels + 1], rows[kMaxLevels + 1];   // padded inputs (level 0: floats, l >= 1: positions)
    int zpitch[kMaxLevels + 1], zrows[kMaxLevels + 1]; // compact outputs (level 0: floats, l >= 1: positions)
    int off_x, off_dy, off_base;
    int off_y[kMaxLevels + 1], off_g[kMaxLevels + 1], off_z[kMaxLevels + 1];  // pair 0 of level l
    int pimg[kMaxLevels + 1], zimg[kMaxLevels + 1];    // floats per padded / compact pair image
    int slot_floats;
};

// kind 0: forward / input-gradient slot (x, pyramid, conv outputs, base buffer)
// kind 1: weight-gradient slot (x, dy and both pyramids)
__host__ __device__ inline Geo make_geo(int H, int W, int L, int K, int kind) {
    Geo g = {};
    g.H = H; g.W = W; g.L = L; g.K = K; g.P = K / 2;
    for (int l = 0; l <= L; ++l) {
        g.h[l] = H >> l;
        g.w[l] = W >> l;
        g.rseg[l] = ceil_div(g.h[l], kRows);
        g.rows[l] = g.rseg[l] * kRows + K - 1;
        g.zrows[l] = g.rseg[l] * kRows;
        if (l == 0) {
            g.cstr[l] = ceil_div(g.w[l], kCols);
            g.pitch[l] = g.cstr[l] * kCols + round_up(K - 1, 4);
            g.zpitch[l] = round_up(W, 8);
        } else {
            g.cstr[l] = ceil_div(g.w[l], kColsL);
            g.pitch[l] = g.cstr[l] * kColsL + round_up(K - 1, 2);
            g.zpitch[l] = round_up(g.w[l], 4);
            g.pimg[l] = 2 * g.rows[l] * g.pitch[l];
            g.zimg[l] = 2 * g.zrows[l] * g.zpitch[l];
        }
    }
    int off = 0;
    g.off_x = off; off += g.rows[0] * g.pitch[0];
    g.off_dy = -1;
    g.off_base = -1;
    if (kind == 1) { g.off_dy = off; off += g.rows[0] * g.pitch[0]; }
    for (int l = 1; l <= L; ++l) { g.off_y[l] = off; off += 2 * g.pimg[l]; }
    for (int l = 1; l <= L; ++l) {
        g.off_g[l] = -1;
        if (kind == 1) { g.off_g[l] = off; off += 2 * g.pimg[l]; }
    }
    for (int l = 1; l <= L; ++l) {
        g.off_z[l] = -1;
        if (kind == 0) { g.off_z[l] = off; off += 2 * g.zimg[l]; }
    }
    if (kind == 0) { g.off_base = off; off += g.zrows[0] * g.zpitch[0]; }
    g.slot_floats = round_up(off, 4);
    return g;
}

// n / d by one multiply-high for n * d < 2^32 (every index range here is far below that).  The
// magic number is computed on the host, once per plan.
struct FastDiv {
    uint32_t d, m;
};
inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.m = d <= 1 ? 0u : (uint32_t)((0x100000000ull + d - 1) / d);
    return f;
}
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fdiv(const FastDiv &f, uint32_t n) { return f.d <= 1 ? n : __umulhi(n, f.m); }
#endif

// Every runtime divisor the kernels use, prepared by the host planner.
struct Divs {
    FastDiv a_n[kMaxLevels + 2], a_w[kMaxLevels + 2];  // analysis pass starting at level l: items per plane, columns
    FastDiv stage_chunks;                              // 16-byte chunks per staged plane
    FastDiv item_plane[kMaxLevels + 1], item_cols[kMaxLevels + 1];  // conv items per image / column strips
    FastDiv out_n, out_w;                              // output segments per plane / per row
};

struct LayerArgs {
    int B, C, H, W, L, K;
    int G;               // planes per slot group (planes of one channel, consecutive b)
    int groups_per_cta;  // slot groups each CTA walks through
    int nb;              // CTAs per channel; grid = nb * C
    int vec_ld;          // 1: rows allow 4-element vector loads of activations
    int st_mode;         // output stores: 2 = 8-element vectors, 1 = 4-element vectors, 0 = scalar
    const void *x;       // forward: x; input gradient: dy; weight gradient: x
    const void *dy;      // weight gradient only
    void *out;           // y or dx
    const float *base_w, *base_bias, *base_scale, *wavelet_w, *wavelet_scale;
    float *partials;     // weight-gradient partials [nb][C][1+4L][K*K+1]
    int threads;         // CTA size (blockDim.x)
    int stage;           // 1: next planes are copied to a shared staging area with cp.async
    int stage_off;       // byte offset of the staging area in dynamic shared memory
    int flip;            // 1: rotate kernels by 180 degrees (input-gradient path)
    Divs dv;
    int with_bias;       // 1: add s_b * b_b (forward only)
    Geo geo;
};

// Dynamic shared memory of the kernels for G planes per slot group; *stage_off receives the
// byte offset of the staging area (staging holds n_in * G raw planes of elem_bytes elements).
size_t fwd_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off);
size_t dw_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off);

// Launchers (host side, in the kernel translation units).  dtype: 0 f32, 1 bf16, 2 f16.
cudaError_t launch_forward(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st);
cudaError_t launch_dw(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st);
cudaError_t launch_dw_finalize(const LayerArgs &a, float *d_base_w, float *d_base_bias,
                               float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale,
                               cudaStream_t st);
int occupancy_forward(int dtype, int K, int threads, size_t smem);
int occupancy_dw(int dtype, int K, int threads, size_t smem);

}  // namespace wtconv
