// Forward kernel of the WTConv layer (also serves the input gradient: the same operator on dy
// with every kernel rotated by 180 degrees and no bias).
//
// Each CTA owns channel c and a run of batch entries and walks through them in groups of G
// planes.  Per group:
//   A. one read of each plane from HBM builds the padded fp32 plane and the Haar pyramid in
//      shared memory (two levels per pass); the next group is prefetched into L2 meanwhile;
//   C. every k x k conv of the layer -- the base conv of the plane and the conv of every subband
//      of every level, with the folded kernels -- runs as sliding-window items (8 x 4 outputs,
//      packed f32x2 FMAs) spread over all threads; results stay in shared memory;
//   D. each output pixel is written once: base conv + bias + closed-form synthesis gather.
#include "wtconv_analysis.cuh"

namespace wtconv {

size_t fwd_smem_bytes(const Geo &geo, int G, int L, int K, int elem_bytes, bool stage, int *stage_off) {
    size_t bytes = (size_t)G * geo.slot_floats * sizeof(float) + (size_t)(1 + 4 * L) * wpairs(K) * sizeof(f2_t);
    bytes = (bytes + 15) / 16 * 16;
    if (stage_off) *stage_off = (int)bytes;
    if (stage) bytes += (size_t)G * geo.H * geo.W * elem_bytes;
    return (bytes + 15) / 16 * 16;
}

// Closed-form synthesis of the 8 output pixels (h, w0 .. w0+7), w0 % 8 == 0, added to out[]:
//   out[c] += sum_l sum_s sigma_s(bit_{l-1}(h), bit_{l-1}(w0+c)) * Z^l_s[h >> l][(w0+c) >> l]
// (Z carries the 2^-l synthesis factor through the folded kernels).
__device__ __forceinline__ void synth_gather8(const Geo &geo, const float *slot, int h, int w0, float (&out)[8]) {
    {   // level 1: four coefficient columns; row bit a = bit 0 of h, column bit b = c & 1
        const int zp = geo.zpitch[1], zs = geo.zrows[1] * zp;
        const float *z = slot + geo.off_z[1] + (h >> 1) * zp + (w0 >> 1);
        const float4 z0 = *reinterpret_cast<const float4 *>(z);
        const float4 z1 = *reinterpret_cast<const float4 *>(z + zs);
        const float4 z2 = *reinterpret_cast<const float4 *>(z + 2 * zs);
        const float4 z3 = *reinterpret_cast<const float4 *>(z + 3 * zs);
        const float a0[4] = {z0.x, z0.y, z0.z, z0.w}, a1[4] = {z1.x, z1.y, z1.z, z1.w};
        const float a2[4] = {z2.x, z2.y, z2.z, z2.w}, a3[4] = {z3.x, z3.y, z3.z, z3.w};
        const bool ra = h & 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float p = ra ? a0[q] - a2[q] : a0[q] + a2[q];
            const float r = ra ? a1[q] - a3[q] : a1[q] + a3[q];
            out[2 * q] += p + r;
            out[2 * q + 1] += p - r;
        }
    }
    if (geo.L >= 2) {  // level 2: two coefficients, column bit b = bit 1 of c
        const int zp = geo.zpitch[2], zs = geo.zrows[2] * zp;
        const float *z = slot + geo.off_z[2] + (h >> 2) * zp + (w0 >> 2);
        const float2 z0 = *reinterpret_cast<const float2 *>(z);
        const float2 z1 = *reinterpret_cast<const float2 *>(z + zs);
        const float2 z2 = *reinterpret_cast<const float2 *>(z + 2 * zs);
        const float2 z3 = *reinterpret_cast<const float2 *>(z + 3 * zs);
        const float a0[2] = {z0.x, z0.y}, a1[2] = {z1.x, z1.y}, a2[2] = {z2.x, z2.y}, a3[2] = {z3.x, z3.y};
        const bool ra = (h >> 1) & 1;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float p = ra ? a0[q] - a2[q] : a0[q] + a2[q];
            const float r = ra ? a1[q] - a3[q] : a1[q] + a3[q];
            out[4 * q] += p + r;
            out[4 * q + 1] += p + r;
            out[4 * q + 2] += p - r;
            out[4 * q + 3] += p - r;
        }
    }
    if (geo.L >= 3) {  // level 3: one coefficient, column bit b = bit 2 of c
        const int zp = geo.zpitch[3], zs = geo.zrows[3] * zp;
        const float *z = slot + geo.off_z[3] + (h >> 3) * zp + (w0 >> 3);
        const bool ra = (h >> 2) & 1;
        const float p = ra ? z[0] - z[2 * zs] : z[0] + z[2 * zs];
        const float r = ra ? z[zs] - z[3 * zs] : z[zs] + z[3 * zs];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            out[c] += p + r;
            out[c + 4] += p - r;
        }
    }
    float deep = 0.f;  // levels >= 4: one coefficient with tile-uniform signs
    for (int l = 4; l <= geo.L; ++l) {
        const int zp = geo.zpitch[l], zs = geo.zrows[l] * zp;
        const float *z = slot + geo.off_z[l] + (h >> l) * zp + (w0 >> l);
        const bool ra = (h >> (l - 1)) & 1, rb = (w0 >> (l - 1)) & 1;
        const float p = ra ? z[0] - z[2 * zs] : z[0] + z[2 * zs];
        const float r = ra ? z[zs] - z[3 * zs] : z[zs] + z[3 * zs];
        deep += rb ? p - r : p + r;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) out[c] += deep;
}

template <int K, typename T>
__global__ void __launch_bounds__(kMaxThreads, (K <= 5 ? 2 : 1)) wtconv_fwd_kernel(const LayerArgs a) {
    constexpr int P = K / 2, WP = wpairs(K);
    extern __shared__ __align__(16) float smem[];
    __shared__ Geo geo;
    // per conv image (sig 0: base, 1 + 4(l-1) + s: level l subband s): first item, input and
    // output offsets within a slot, pitches
    __shared__ int cstart[kMaxSig + 1], in_off[kMaxSig], out_off[kMaxSig], in_pitch[kMaxSig], out_pitch[kMaxSig],
        sig_lvl[kMaxSig];
    const int c = blockIdx.x % a.C;
    const int nbi = blockIdx.x / a.C;
    const int G = a.G, nsig = 1 + 4 * a.L;
    float *slots = smem;
    f2_t *wts = reinterpret_cast<f2_t *>(smem + (size_t)G * a.geo.slot_floats);

    if (threadIdx.x == 0) {
        geo = a.geo;
        int tot = 0;
        for (int sig = 0; sig < nsig; ++sig) {
            const int l = sig == 0 ? 0 : (sig - 1) / 4 + 1, s = sig == 0 ? 0 : (sig - 1) & 3;
            cstart[sig] = tot;
            sig_lvl[sig] = l;
            in_pitch[sig] = a.geo.pitch[l];
            out_pitch[sig] = a.geo.zpitch[l];
            in_off[sig] = sig == 0 ? a.geo.off_x : a.geo.off_y[l] + s * a.geo.rows[l] * a.geo.pitch[l];
            out_off[sig] = sig == 0 ? a.geo.off_base : a.geo.off_z[l] + s * a.geo.zrows[l] * a.geo.zpitch[l];
            tot += G * a.geo.rseg[l] * a.geo.cstr[l];
        }
        cstart[nsig] = tot;
    }
    {
        float4 *s4 = reinterpret_cast<float4 *>(slots);
        const int n4 = G * a.geo.slot_floats / 4;
        for (int i = threadIdx.x; i < n4; i += blockDim.x) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    stage_weights<K>(a, c, wts);
    const float bias = a.with_bias ? a.base_scale[c] * a.base_bias[c] : 0.f;
    __syncthreads();

    const T *x = static_cast<const T *>(a.x);
    T *y = static_cast<T *>(a.out);
    const size_t HW = (size_t)a.H * a.W;
    T *stg = a.stage ? reinterpret_cast<T *>(reinterpret_cast<char *>(smem) + a.stage_off) : nullptr;
    if (stg) {  // stage the first group
        stage_planes<T>(x, stg, a.B, a.C, c, nbi * a.groups_per_cta * G, G, HW, a.dv.stage_chunks);
        cp_async_commit();
    }
    const int nitems = cstart[nsig];
    const int nws = (int)a.dv.out_w.d, nd = (int)a.dv.out_n.d;
    const int slot_floats = geo.slot_floats;

    for (int grp = 0; grp < a.groups_per_cta; ++grp) {
        const int b0 = (nbi * a.groups_per_cta + grp) * G;
        if (b0 >= a.B) break;
        if (stg) {
            cp_async_wait_all();
            __syncthreads();
        }
        // A. planes -> padded fp32 copy + Haar pyramid; then the next group starts streaming in
        analysis_from_global<T, P>(a, geo, x, stg, c, b0, slots, geo.off_x, geo.off_y);
        __syncthreads();
        if (stg && grp + 1 < a.groups_per_cta && b0 + G < a.B) {
            stage_planes<T>(x, stg, a.B, a.C, c, b0 + G, G, HW, a.dv.stage_chunks);
            cp_async_commit();
        }
        for (int l = 3; l <= geo.L; l += 2) {
            analysis_from_shared<P>(a, geo, slots, G, geo.off_y, l);
            __syncthreads();
        }

        // C. every conv of the layer, as sliding-window items
        for (int it = threadIdx.x; it < nitems; it += blockDim.x) {
            int sig = 0;
            while (it >= cstart[sig + 1]) ++sig;
            const int l = sig_lvl[sig];
            const int local = it - cstart[sig];
            const int g = fdiv(a.dv.item_plane[l], local), e = local - g * (int)a.dv.item_plane[l].d;
            const int rs = fdiv(a.dv.item_cols[l], e), cs = e - rs * (int)a.dv.item_cols[l].d;
            float *slot = slots + g * slot_floats;
            f2_t w[K * K];
            load_weights<K>(wts + sig * WP, w);
            const int pitch = in_pitch[sig], opitch = out_pitch[sig];
            conv_item<K>(slot + in_off[sig] + (rs * kRows) * pitch + cs * kCols, pitch, w,
                         slot + out_off[sig] + (rs * kRows) * opitch + cs * kCols, opitch);
        }
        __syncthreads();

        // D. output pixels: base conv + bias + closed-form synthesis
        for (int it = threadIdx.x; it < G * nd; it += blockDim.x) {
            const int g = fdiv(a.dv.out_n, it), e = it - g * nd;
            const int h = fdiv(a.dv.out_w, e), ws = e - h * nws;
            const int b = b0 + g;
            if (b >= a.B) continue;
            const int w0 = ws * 8;
            const float *slot = slots + g * slot_floats;
            const float *bb = slot + geo.off_base + h * geo.zpitch[0] + w0;
            const float4 b0v = *reinterpret_cast<const float4 *>(bb);
            const float4 b1v = *reinterpret_cast<const float4 *>(bb + 4);
            float out[8] = {b0v.x + bias, b0v.y + bias, b0v.z + bias, b0v.w + bias,
                            b1v.x + bias, b1v.y + bias, b1v.z + bias, b1v.w + bias};
            synth_gather8(geo, slot, h, w0, out);
            T *dst = y + ((size_t)b * a.C + c) * HW + (size_t)h * geo.W + w0;
            const int nv = min(8, geo.W - w0);
            if (a.st_mode == 2 && nv == 8) {
                Act<T>::st8(dst, out);
            } else if (a.st_mode >= 1) {
                Act<T>::st4(dst, out);
                if (nv == 8) Act<T>::st4(dst + 4, out + 4);
            } else {
                for (int i = 0; i < nv; ++i) Act<T>::st(dst + i, out[i]);
            }
        }
        __syncthreads();
    }
}

template <int K, typename T>
static cudaError_t launch_fwd_t(const LayerArgs &a, size_t smem, cudaStream_t st) {
    auto kern = wtconv_fwd_kernel<K, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(a.nb * a.C)), a.threads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int K, typename T>
static int occ_fwd_t(int threads, size_t smem) {
    auto kern = wtconv_fwd_kernel<K, T>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) return 0;
    return n;
}

#define WTCONV_DISPATCH(K_, DT_, FN, ...)                                                 \
    switch ((K_) * 4 + (DT_)) {                                                           \
    case 3 * 4 + 0: return FN<3, float>(__VA_ARGS__);                                     \
    case 3 * 4 + 1: return FN<3, __nv_bfloat16>(__VA_ARGS__);                             \
    case 3 * 4 + 2: return FN<3, __half>(__VA_ARGS__);                                    \
    case 5 * 4 + 0: return FN<5, float>(__VA_ARGS__);                                     \
    case 5 * 4 + 1: return FN<5, __nv_bfloat16>(__VA_ARGS__);                             \
    case 5 * 4 + 2: return FN<5, __half>(__VA_ARGS__);                                    \
    case 7 * 4 + 0: return FN<7, float>(__VA_ARGS__);                                     \
    case 7 * 4 + 1: return FN<7, __nv_bfloat16>(__VA_ARGS__);                             \
    case 7 * 4 + 2: return FN<7, __half>(__VA_ARGS__);                                    \
    default: break;                                                                       \
    }

cudaError_t launch_forward(const LayerArgs &a, int dtype, size_t smem, cudaStream_t st) {
    WTCONV_DISPATCH(a.K, dtype, launch_fwd_t, a, smem, st);
    return cudaErrorInvalidValue;
}

int occupancy_forward(int dtype, int K, int threads, size_t smem) {
    WTCONV_DISPATCH(K, dtype, occ_fwd_t, threads, smem);
    return 0;
}

}  // namespace wtconv
