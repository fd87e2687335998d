// Zero padding and cropping of whole planes, for layers whose sides are not multiples of 2^L.
//
// The layer on such a plane equals the layer on the plane zero-padded at its end to multiples of
// 2^L, cropped back: padding every odd side of a level by one zero at its end before the Haar
// analysis (the stride-2 'SAME' Haar conv), and cropping that level's reconstruction back to the
// level's input size, never lets a padded row or column reach a pixel inside the plane, since the
// level-l ancestor of row h < H is h >> l < ceil(H / 2^l).  So the library pads the activations
// into the workspace, runs the layer on the padded planes and crops the results.
//
// One warp per destination row, its lanes striding over the columns: one division per row, and
// neighbouring lanes touch neighbouring elements.  Elements are copied as raw bits (2 or 4 bytes);
// the padding is all-zero bits, +0.0 in every supported type.
#include <stdint.h>

#include "wtconv_pad.h"

namespace wtconv {

namespace {

constexpr int kPadThreads = 256;

template <typename E>
__global__ void __launch_bounds__(kPadThreads) wtconv_pad_kernel(const E *__restrict__ src, E *__restrict__ dst,
                                                                 long long planes, int H, int W, int Hp, int Wp) {
    const int lane = threadIdx.x & 31;
    const long long rows = planes * Hp;
    const long long warps = (long long)gridDim.x * (kPadThreads / 32);
    for (long long row = (long long)blockIdx.x * (kPadThreads / 32) + (threadIdx.x >> 5); row < rows; row += warps) {
        const long long p = row / Hp;
        const int r = (int)(row - p * Hp);
        E *d = dst + row * Wp;
        if (r < H) {
            const E *s = src + (p * H + r) * W;
            for (int c = lane; c < Wp; c += 32) d[c] = c < W ? s[c] : E(0);
        } else {
            for (int c = lane; c < Wp; c += 32) d[c] = E(0);
        }
    }
}

template <typename E>
__global__ void __launch_bounds__(kPadThreads) wtconv_crop_kernel(const E *__restrict__ src, E *__restrict__ dst,
                                                                  long long planes, int H, int W, int Hp, int Wp) {
    const int lane = threadIdx.x & 31;
    const long long rows = planes * H;
    const long long warps = (long long)gridDim.x * (kPadThreads / 32);
    for (long long row = (long long)blockIdx.x * (kPadThreads / 32) + (threadIdx.x >> 5); row < rows; row += warps) {
        const long long p = row / H;
        const int r = (int)(row - p * H);
        const E *s = src + (p * Hp + r) * Wp;
        E *d = dst + row * W;
        for (int c = lane; c < W; c += 32) d[c] = s[c];
    }
}

unsigned pad_grid(long long rows) {
    const long long per_block = kPadThreads / 32;
    long long blocks = (rows + per_block - 1) / per_block;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ==
                                                  cudaSuccess && sms > 0)
        blocks = blocks < (long long)sms * 16 ? blocks : (long long)sms * 16;
    return (unsigned)(blocks > 0 ? blocks : 1);
}

}  // namespace

cudaError_t launch_pad_planes(const void *src, void *dst, long long planes, int H, int W, int Hp, int Wp,
                              int elem_bytes, cudaStream_t st) {
    const unsigned grid = pad_grid(planes * Hp);
    if (elem_bytes == 4)
        wtconv_pad_kernel<uint32_t><<<grid, kPadThreads, 0, st>>>(static_cast<const uint32_t *>(src),
                                                                 static_cast<uint32_t *>(dst), planes, H, W, Hp, Wp);
    else if (elem_bytes == 2)
        wtconv_pad_kernel<uint16_t><<<grid, kPadThreads, 0, st>>>(static_cast<const uint16_t *>(src),
                                                                 static_cast<uint16_t *>(dst), planes, H, W, Hp, Wp);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_crop_planes(const void *src, void *dst, long long planes, int H, int W, int Hp, int Wp,
                               int elem_bytes, cudaStream_t st) {
    const unsigned grid = pad_grid(planes * H);
    if (elem_bytes == 4)
        wtconv_crop_kernel<uint32_t><<<grid, kPadThreads, 0, st>>>(static_cast<const uint32_t *>(src),
                                                                  static_cast<uint32_t *>(dst), planes, H, W, Hp, Wp);
    else if (elem_bytes == 2)
        wtconv_crop_kernel<uint16_t><<<grid, kPadThreads, 0, st>>>(static_cast<const uint16_t *>(src),
                                                                  static_cast<uint16_t *>(dst), planes, H, W, Hp, Wp);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace wtconv
