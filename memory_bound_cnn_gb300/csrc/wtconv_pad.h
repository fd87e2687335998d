// Zero padding and cropping of whole planes, for layers whose sides are not multiples of 2^L.
#pragma once

#include <cuda_runtime.h>

namespace wtconv {

// Pad every [H][W] plane of src at the end of each side with zeros into a [planes][Hp][Wp]
// buffer, and the crop back to [planes][H][W]; elements of 2 or 4 bytes, copied as raw bits.
cudaError_t launch_pad_planes(const void *src, void *dst, long long planes, int H, int W, int Hp, int Wp,
                              int elem_bytes, cudaStream_t st);
cudaError_t launch_crop_planes(const void *src, void *dst, long long planes, int H, int W, int Hp, int Wp,
                               int elem_bytes, cudaStream_t st);

}  // namespace wtconv
