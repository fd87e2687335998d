// Tiled batch-pair weight-gradient kernel of the WTConv layer: host-visible geometry and launch
// interface.
//
// One launch correlates up to two Haar levels (plus the base path) of planes split into tiles:
// per tile, one bulk tensor copy brings the x tile with the halo the deepest level needs and one
// the dy tile, and the pyramids of both are built on chip.  Planes of more than two levels are
// handled by launching the same kernel again on the level-2 low bands (LL) of x and dy, which the
// previous launch writes as fp32 planes (1/16 of the input): the unnormalised pyramid of the
// unnormalised LL band is the input's own pyramid two levels further down, so each launch only
// shifts the signal index by its level offset.
#pragma once

#include "wtconv_internal.h"

namespace wtconv {

constexpr int kPtMaxLevels = 2;  // levels per launch
constexpr int kPtMaxEntries = 8;  // (signal, tap) sums each thread keeps across a work unit

// One level of a tile (level 0: the base path).  x-side images are zero-padded (interior at
// (P, P)), dy-side images compact; both rounded up to whole Q x S items.
struct PtLevel {
    int h, w;                      // interior of the tile at this level
    int Q, S, ns, ng;              // item columns / rows, strips per row, segments per image
    int ipitch, irows, iimg;       // padded x-side image (pairs)
    int zpitch, zrows, zimg;       // compact dy-side image (pairs)
    int off_y, off_z;              // slot offsets (pairs) of subband 0; subband s at + s * iimg / zimg
    int items;                     // items per subband image: ns * ng
};

struct PtileArgs {
    int B, C, H, W;                // this launch's input planes (x / dy, or the LL planes of a previous launch)
    int K, LT;                     // kernel size; levels correlated here (1 or 2)
    int base;                      // 1: the base path (signal 0, with the sum of dy)
    int lvl_off;                   // global level of this launch's level l is l + lvl_off
    int L_total;                   // levels of the layer: the partials hold 1 + 4 L_total signals
    int TH, TW;                    // tile (positions of this launch's level 0)
    int HX, HXL;                   // halo rows / columns of the raw x tile (HXL: HX rounded to 16 bytes)
    int RXR, RXW;                  // raw x tile rows / row length (elements)
    int tiles_r, tiles_c, tiles;
    int G, npairs, ngroups;        // pair slots per group; ceil(B / 2); groups per tile
    int work;                      // work items per channel: ngroups * tiles (tiles innermost: neighbouring
                                   // tiles of one pair group follow each other, so their halos hit L2)
    int nchunks;                   // partial rows per channel; chunk n covers work [n*work/nchunks, (n+1)*work/nchunks)
    int units, grid, nthreads;     // units = C * nchunks (channel-major); persistent grid
    int per_pair;                  // correlation items per pair
    int n0, n1, n2;                // items per image of level 0 (0 without the base path), 1 and 2
    int slot;                      // pairs per slot
    int raw_x_bytes, raw_dy_bytes; // one group's raw tiles (128-byte rounded)
    int in_pitch;                  // row pitch of the input planes (elements)
    int ll_out;                    // 1: write the level-2 LL bands of x and dy to ll_x / ll_dy
    int ll_h, ll_w, ll_pitch;      // LL planes: ll_h x ll_w positions, row pitch ll_pitch (floats)
    PtLevel lv[kPtMaxLevels + 1];
    FastDiv dv_pp, dv_n1, dv_n2, dv_ns[kPtMaxLevels + 1], dv_tiles, dv_tiles_c;
    FastDiv dv_xb, dv_xbw, dv_db, dv_dbw;  // pass 1: x blocks per pair / per row, dy blocks per pair / per row
    const void *x, *dy;
    float *ll_x, *ll_dy;
    float *partials;               // [nchunks][C][1 + 4 L_total][K*K+1]
    int *timeout;
    CUtensorMap tmap_x, tmap_dy;   // x: box RXW x RXR x 1 x 2G at (c0 - HXL, r0 - HX); dy: TW x TH x 1 x 2G
};

// Dynamic shared memory of one launch (bytes, including 128 bytes of alignment room).
size_t ptile_smem_bytes(const PtileArgs &a, int elem_bytes);
// dtype: 0 fp32, 1 bf16, 2 fp16 (the LL launches are fp32); iq: item width (2 or 4), the same at
// every level of a launch.
cudaError_t launch_ptile_dw(const PtileArgs &a, int dtype, size_t smem, cudaStream_t st);
int occupancy_ptile_dw(int dtype, int K, int LT, int base, size_t smem, int nthreads, int iq);

}  // namespace wtconv
