// Tiled batch-pair shallow kernel of the WTConv forward / input gradient: host-visible geometry and
// launch interface.
//
// For planes too large for the whole-plane kernels the operator runs in two launches: the deep
// kernel computes the contribution of Haar levels >= 2 at level-1 resolution (D, fp32, in the
// workspace), then this kernel computes, per tile of the output, the base conv, the level-1 convs
// and the closed-form synthesis of level 1 with D added to its low band, and stores every pixel
// once.  Two batch entries of one channel share each shared-memory position (packed fp32 pairs),
// as in the whole-plane batch-pair kernels.
#pragma once

#include "wtconv_internal.h"

namespace wtconv {

struct PsArgs {
    int B, C, H, W, K;
    int TH, TW;                    // output tile
    int HX, HXL;                   // halo rows / columns of the raw x tile (2P; HXL rounded to 16 bytes)
    int RXR, RXW;                  // raw x tile rows / row length (elements)
    int tiles_r, tiles_c, tiles;
    int G, npairs, ngroups;        // pair slots per group; ceil(B / 2); groups per tile
    int work;                      // work items (channel, group, tile): channel-major, tiles innermost, so
                                   // that a CTA walks neighbouring tiles of one pair of planes (their
                                   // halos are still in L2)
    int grid, nthreads;            // persistent grid: CTA i takes work [i*work/grid, (i+1)*work/grid)
    // slot geometry (pairs): X padded (interior at (P, P)), level 1 padded (4 images), level-1 conv
    // outputs Z1 (4 compact images) followed by D (one more image of the same shape)
    int q0, s0, ns0, ng0, ipitch0, irows0;  // output items Q0 x S0 over the tile (S0 = S1 = 4 or 8)
    int q1, s1, ns1, ng1, ipitch1, irows1, iimg1, zpitch1, zrows1, zimg1;  // level-1 conv items
    int off_x, off_y1, off_z1;
    int slot;                      // pairs per slot
    int raw_x_bytes, raw_d_bytes;  // one group's raw tiles (128-byte rounded)
    int has_deep;                  // L >= 2: D tiles arrive with the x tiles
    int vec_st;                    // rows allow vector stores
    FastDiv dv_work_c, dv_tiles, dv_tiles_c, dv_xb, dv_xbw, dv_conv, dv_ns1, dv_out, dv_ns0, dv_db, dv_dbw;
    const void *x;                 // forward: x; input gradient: dy
    const float *deep;             // D [B][C][H/2][W/2] fp32, or null
    void *out;
    const float *base_w, *base_bias, *base_scale, *wavelet_w, *wavelet_scale;
    int flip, with_bias;
    int *timeout;
    CUtensorMap tmap_x, tmap_d;    // x: box RXW x RXR x 1 x 2G at (c0 - HXL, r0 - HX); D: TW/2 x TH/2 x 1 x 2G
};

size_t pshallow_smem_bytes(const PsArgs &a);
// dtype: 0 fp32, 1 bf16, 2 fp16
cudaError_t launch_pshallow(const PsArgs &a, int dtype, size_t smem, cudaStream_t st);
// nthreads 64 or 128; s: item rows, 4 or 8
int occupancy_pshallow(int dtype, int K, size_t smem, int nthreads, int s);

}  // namespace wtconv
