// Internal types shared by the host entry points (wtconv_api.cu) and the kernel translation
// units (wtconv_fwd.cu, wtconv_bwd.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>
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
constexpr int kSmemPerSM = 228 * 1024;  // shared memory of one SM (all resident CTAs)

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
// kind 2: deep slot (levels >= 2 only: pyramid and conv outputs; no full-resolution plane)
// kind 3: weight-gradient deep slot (levels >= 2 only: both pyramids)
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
    const int l0 = kind >= 2 ? 2 : 1;  // first stored level
    g.off_x = -1;
    if (kind < 2) { g.off_x = off; off += g.rows[0] * g.pitch[0]; }
    g.off_dy = -1;
    g.off_base = -1;
    if (kind == 1) { g.off_dy = off; off += g.rows[0] * g.pitch[0]; }
    for (int l = 1; l <= L; ++l) {
        g.off_y[l] = -1;
        if (l >= l0) { g.off_y[l] = off; off += 2 * g.pimg[l]; }
    }
    for (int l = 1; l <= L; ++l) {
        g.off_g[l] = -1;
        if (kind == 1 || (kind == 3 && l >= 2)) { g.off_g[l] = off; off += 2 * g.pimg[l]; }
    }
    for (int l = 1; l <= L; ++l) {
        g.off_z[l] = -1;
        if ((kind == 0 && l >= 1) || (kind == 2 && l >= 2)) { g.off_z[l] = off; off += 2 * g.zimg[l]; }
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
// Geometry of the shallow kernel's tiles.  A unit is one output tile of TH x TW pixels of G
// planes (G > 1 only when one tile covers a whole plane).  Its input tile X covers plane rows
// r0 - 2P .. r0 + TH + 2P - 1 and columns c0 - padx .. c0 + TW + padx - 1 (halo 2P: P for the
// base conv, P level-1 coefficients for the level-1 conv; padx = 2P rounded up to a multiple of
// 4 and of the copy chunk, so every chunk lies wholly inside or outside the plane and every base
// window row starts 16-byte aligned).  Level 1 of the tile (+ P coefficients of halo) is kept as
// two subband-pair images (LL|LH, HL|HH).
struct ShallowGeo {
    int TH, TW;            // output tile (TH % 8 == 0, TW % 4 == 0)
    int G;                 // planes per unit
    int tiles_r, tiles_c;  // tiles per plane
    int padx;              // left / right halo columns of X (multiple of 4 and of chunk_e)
    int xrows, xw;         // X tile rows and row length (floats; also the raw tile's row length)
    int yrows, ycols;      // level-1 positions per pair image (TH/2 + 2P) x (TW/2 + 2P)
    int ypitch, yimg;      // pair-image row pitch (positions) and floats per image
    int items_r, items_c;  // fused output items per tile (8 x 4 pixels each)
    int chunk_e;           // elements per cp.async chunk of the raw tile (16, 8 or 4 bytes)
    int dchunk_e;          // floats per cp.async chunk of the deep tile (4 or 2)
    int dtile;             // floats of one deep tile per plane: (TH/2) x (TW/2)
    int raw_bytes;         // one raw tile buffer (G planes), 16-byte rounded
    int xbuf;              // floats of one X buffer (G planes): the raw buffer itself for fp32
    int pslot;             // floats of the pair images of one plane
};

__host__ __device__ inline ShallowGeo make_shallow_geo(int H, int W, int K, int TH, int TW, int G, int elem_bytes,
                                                       int chunk_e, int dchunk_e) {
    ShallowGeo s = {};
    const int P = K / 2;
    s.TH = TH; s.TW = TW; s.G = G;
    s.tiles_r = ceil_div(H, TH);
    s.tiles_c = ceil_div(W, TW);
    const int pq = chunk_e > 4 ? chunk_e : 4;
    s.padx = round_up(2 * P, pq);
    s.xrows = TH + 4 * P;
    s.xw = TW + 2 * s.padx;
    s.yrows = TH / 2 + 2 * P;
    s.ycols = TW / 2 + 2 * P;
    s.ypitch = round_up(s.ycols, 2);
    s.yimg = 2 * s.yrows * s.ypitch;
    s.pslot = 2 * s.yimg;
    s.items_r = TH / kRows;
    s.items_c = TW / kCols;
    s.chunk_e = chunk_e;
    s.dchunk_e = dchunk_e;
    s.dtile = (TH / 2) * (TW / 2);
    s.raw_bytes = round_up(G * s.xrows * s.xw * elem_bytes, 16);
    s.xbuf = G * s.xrows * s.xw;
    return s;
}

struct ShallowArgs {
    int B, C, H, W, L, K;
    int units;            // work units per channel: plane groups x tiles
    int units_per_cta;    // contiguous units each CTA walks through
    int nb;               // CTAs per channel; grid = nb * C
    int st_mode;          // output stores: 1 = 4-element vectors where a row allows, 0 = scalar
    const void *x;        // forward: x; input gradient: dy
    const float *deep;    // deep contribution at level-1 resolution [B][C][H/2][W/2] (L >= 2)
    void *out;            // y or dx
    const float *base_w, *base_bias, *base_scale, *wavelet_w, *wavelet_scale;
    int flip, with_bias;
    ShallowGeo sg;
    // units per plane group (tiles) and tile columns; raw-tile chunks per row and rows per plane;
    // deep-tile chunks per row and rows per plane; level-1 positions per row; X 4-float groups per row
    FastDiv tiles, tiles_c, rchunks_row, xrows, dchunks_row, drows, ycols, xw4;
    // TMA: when set, one lane loads the whole input tile (box xw x xrows x 1 x G of the 4-D
    // tensor W, H, C, B) and / or the deep tile with one bulk tensor copy each; zero fill outside
    int tma_x, tma_d;
    int *timeout;         // sticky device flag raised by a bounded wait that gave up
    CUtensorMap tmap_x, tmap_d;
};

size_t shallow_smem_bytes(const ShallowGeo &sg, int K, bool convert, bool deep);
cudaError_t launch_shallow(const ShallowArgs &a, int dtype, size_t smem, cudaStream_t st);
int occupancy_shallow(int dtype, int K, size_t smem);

// Deep kernel: levels >= 2 of every plane and their closed-form contribution at level-1 resolution.
size_t deep_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off);
cudaError_t launch_deep(const LayerArgs &a, float *deep_out, int dtype, size_t smem, cudaStream_t st);
int occupancy_deep(int dtype, int K, int threads, size_t smem);

// Whole-plane kernel (planes whose pyramid fits in shared memory): forward / input gradient in one pass.
size_t fwd_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off);
cudaError_t launch_forward(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st);
int occupancy_forward(int dtype, int K, int threads, size_t smem);

size_t dw_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off);

// Weight gradient of planes too large for the whole-plane kernel: Haar pyramids of x and dy in
// the workspace (float4 (LL, LH, HL, HH) per position, level l at pyr_*[l]), then tiled
// correlations writing nb partials per (channel, signal, tap) for the finalize kernel.
struct DwPyramidArgs {
    int B, C, H, W, L, K;
    int from_level;            // 1: every correlation; 2: levels >= 2 only (the tiled kernel does the rest)
    int nb;                    // partials per (channel, signal, tap): CTAs per channel of each correlation
    const void *x, *dy;
    float4 *pyr_x[kMaxLevels + 1], *pyr_dy[kMaxLevels + 1];
    float *partials;           // [nb][C][1+4L][K*K+1]
};
size_t dw_pyramid_bytes(int B, int C, int H, int W, int L, int from_level);

// Tiled weight gradient (base path and level 1; levels >= 2 go to the level kernels from level 2):
// one warp per CTA over units of the shallow kernel's tiling, x and dy tiles by bulk tensor copy.
struct DwTileArgs {
    int B, C, H, W, L, K;
    int units, units_per_cta, nb;  // units per channel; grid = nb * C
    float *partials;               // [nb][C][1+4L][K*K+1]; this kernel writes signals 0 .. 4
    ShallowGeo sg;
    FastDiv tiles, tiles_c;
    int *timeout;
    CUtensorMap tmap_x, tmap_dy;   // x: box xw x xrows x 1 x G at (c0 - padx, r0 - 2P); dy: TW x TH x 1 x G
};
// Fused whole-plane forward / input-gradient kernel: one plane per CTA iteration, its whole
// pyramid on chip, the fused output items of the shallow kernel.
constexpr int kPlaneThreads = 128;
constexpr int kPlaneDeepRows = 4;  // rows per conv item of a level >= 2 image in the fused kernel
struct PlaneArgs {
    int B, C, H, W, L, K;
    int nb, planes_per_cta;        // grid = nb * C; CTA n takes batch entries n*ppc .. n*ppc + ppc - 1
    int st_mode;                   // 1: 4-element vector stores where a row allows
    const void *x;                 // forward: x; input gradient: dy
    void *out;                     // y or dx
    const float *base_w, *base_bias, *base_scale, *wavelet_w, *wavelet_scale;
    int flip, with_bias;
    ShallowGeo sg;                 // the whole plane as one tile (TH >= H, TW >= W, G = 1)
    Geo dg;                        // levels >= 2 slot (L >= 2)
    int dpitch;                    // row pitch (floats) of D, the deep contribution at level-1 resolution
    int n_deep_items;              // conv items (kPlaneDeepRows x kColsL) of the levels >= 2 images
    int deep_item_start[1 + 2 * kMaxLevels + 1];  // first item of conv image ci (ci = 3 .. 2L), then the end
    int *timeout;
    CUtensorMap tmap_x;            // box xw x xrows x 1 x 1 at (-padx, -2P, c, b)
};
size_t plane_smem_bytes(const PlaneArgs &a, int elem_bytes);
cudaError_t launch_plane(const PlaneArgs &a, int dtype, size_t smem, cudaStream_t st);
int occupancy_plane(int dtype, int K, size_t smem);

// Fused whole-plane weight gradient: one plane of x and of dy per CTA iteration, both pyramids on
// chip, every thread pinned to a share of one correlation's items for the whole CTA.
constexpr int kDwPlaneMaxThreads = 256;
struct DwPlaneArgs {
    int B, C, H, W, L, K;
    int nthreads;                  // CTA size: a multiple of 32, at most kDwPlaneMaxThreads
    int nb, planes_per_cta;        // grid = nb * C
    int nbuf;                      // copy buffers: 2 = the next plane's copies overlap this plane's work
    float *partials;               // [nb][C][1+4L][K*K+1]
    ShallowGeo sg;                 // x as one tile with a 2P halo (TH >= H, TW >= W, G = 1)
    int th1;                       // level-1 rows padded to the 8-row items: round_up(TH / 2, 8)
    int y1rows;                    // rows of every level-1 pair image (x and dy): th1 + 2P, pitch sg.ypitch
    Geo dg;                        // levels >= 2, both pyramids (kind 3)
    int per_thread_base;           // base-path items each base thread takes per plane
    int per_thread;                // items of its pair image each level thread takes per plane
    int tstart[1 + 2 * kMaxLevels + 1];  // first thread of correlation image ci (base, then level
                                         // l pair p at 1 + 2(l-1) + p), then the end
    int *timeout;
    CUtensorMap tmap_x, tmap_dy;   // x: box xw x xrows x 1 x 1 at (-padx, -2P); dy: TW x TH x 1 x 1 at (0, 0)
};
size_t dw_plane_smem_bytes(const DwPlaneArgs &a, int elem_bytes);
cudaError_t launch_dw_plane(const DwPlaneArgs &a, int dtype, size_t smem, cudaStream_t st);
int occupancy_dw_plane(int dtype, int K, size_t smem, int nthreads);

size_t dw_tile_smem_bytes(const ShallowGeo &sg, int elem_bytes);
cudaError_t launch_dw_tile(const DwTileArgs &a, int dtype, size_t smem, cudaStream_t st);
int occupancy_dw_tile(int dtype, int K, size_t smem);
cudaError_t launch_dw_pyramid(const DwPyramidArgs &a, int dtype, cudaStream_t st);

// Launchers (host side, in the kernel translation units).  dtype: 0 f32, 1 bf16, 2 f16.
cudaError_t launch_dw(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st);
cudaError_t launch_dw_finalize(const LayerArgs &a, float *d_base_w, float *d_base_bias,
                               float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale,
                               cudaStream_t st);
int occupancy_dw(int dtype, int K, int threads, size_t smem);

}  // namespace wtconv
