// Internal types shared by the host entry points (wtconv_api.cu) and the kernel translation
// units (wtconv_fwd.cu, wtconv_bwd.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace wtconv {

constexpr int kThreads = 256;   // threads per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kMaxLevels = 5;
constexpr int kMaxSmem = 227 * 1024;

__host__ __device__ constexpr int round_up(int a, int m) { return (a + m - 1) / m * m; }
// floats per staged kernel slot (16-byte aligned)
__host__ __device__ constexpr int wslot_stride(int K) { return round_up(K * K, 4); }
// accumulators per weight-gradient subband: K*K taps + 1 (sum of the gradient, for the bias)
__host__ __device__ constexpr int dw_na(int K) { return K * K + 1; }
__host__ __device__ constexpr int dw_na32(int K) { return round_up(K * K + 1, 32); }

// Shared-memory geometry of one plane slot, in floats.  Level 0 is full resolution.
// Padded buffers hold a zero border of P = K/2 around the interior (origin (P, P)); their
// extents are rounded so that every 2x4 / 4x4 micro-tile window stays inside the buffer and
// every row starts 16-byte aligned.  Conv outputs Z^l are compact (no border).
struct Geo {
    int H, W, L, K, P;
    int pitch[kMaxLevels + 1], rows[kMaxLevels + 1];
    int zpitch[kMaxLevels + 1], zrows[kMaxLevels + 1];
    int off_x, off_dy;
    int off_y[kMaxLevels + 1], off_g[kMaxLevels + 1], off_z[kMaxLevels + 1];
    int slot_floats;
};

__host__ __device__ inline Geo make_geo(int H, int W, int L, int K, bool with_dy, bool with_z) {
    Geo g = {};
    g.H = H; g.W = W; g.L = L; g.K = K; g.P = K / 2;
    const int padc = round_up(2 * g.P, 4);
    for (int l = 0; l <= L; ++l) {
        const int h = H >> l, w = W >> l;
        g.rows[l] = round_up(h, 4) + 2 * g.P;
        g.pitch[l] = round_up(w, 4) + padc;
        g.zrows[l] = round_up(h, 2);
        g.zpitch[l] = round_up(w, 4);
    }
    int off = 0;
    g.off_x = off; off += round_up(g.rows[0] * g.pitch[0], 4);
    g.off_dy = -1;
    if (with_dy) { g.off_dy = off; off += round_up(g.rows[0] * g.pitch[0], 4); }
    for (int l = 1; l <= L; ++l) { g.off_y[l] = off; off += 4 * g.rows[l] * g.pitch[l]; }
    for (int l = 1; l <= L; ++l) {
        g.off_g[l] = -1;
        if (with_dy) { g.off_g[l] = off; off += 4 * g.rows[l] * g.pitch[l]; }
    }
    for (int l = 1; l <= L; ++l) {
        g.off_z[l] = -1;
        if (with_z) { g.off_z[l] = off; off += 4 * g.zrows[l] * g.zpitch[l]; }
    }
    g.slot_floats = round_up(off, 4);
    return g;
}

struct LayerArgs {
    int B, C, H, W, L, K;
    int G;               // plane slots per CTA (planes of one channel, consecutive b)
    int groups_per_cta;  // plane groups each CTA walks through
    int nb;              // CTAs per channel; grid = nb * C
    const void *x;       // forward: x; input-gradient: dy; backward: x
    const void *dy;      // backward only
    void *out;           // y or dx (may be null in the weights-only backward)
    const float *base_w, *base_bias, *base_scale, *wavelet_w, *wavelet_scale;
    float *partials;     // weight-gradient partials [nb][C][1+4L][K*K+1]
    int flip;            // 1: rotate kernels by 180 degrees (input-gradient path)
    int with_bias;       // 1: add s_b * b_b (forward only)
    int want_dx;         // backward: also produce dx
    Geo geo;
};

// Shared memory of the forward / input-gradient kernel for G slots.
size_t fwd_smem_bytes(const Geo &geo, int G, int L, int K);
// Shared memory of the backward kernel (weights, optionally input gradient) for G slots.
size_t bwd_smem_bytes(const Geo &geo, int G, int L, int K);

// Launchers (host side, in the kernel translation units).  They return cudaSuccess or the
// launch error.  dtype: 0 f32, 1 bf16, 2 f16.  K in {3, 5, 7}.
cudaError_t launch_forward(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st);
cudaError_t launch_backward(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st);
cudaError_t launch_dw_finalize(const LayerArgs &a, float *d_base_w, float *d_base_bias,
                               float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale,
                               cudaStream_t st);
// Occupancy (CTAs per SM) of the forward / backward kernel at this shared-memory size.
int occupancy_forward(int dtype, int K, size_t smem);
int occupancy_backward(int dtype, int K, size_t smem);

}  // namespace wtconv
