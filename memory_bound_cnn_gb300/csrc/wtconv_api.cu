// Host side of the C ABI declared in include/wtconv.h: argument validation, launch planning
// (plane slots per CTA, CTAs per channel, workspace) and the launches.  Every check runs before
// anything is launched; on error nothing is written.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "wtconv.h"
#include "wtconv_internal.h"

using namespace wtconv;

namespace {

constexpr int kStaticSmemMargin = 1024;  // static shared memory of the kernels (the Geo copy)
constexpr int kTargetSlotPixels = 1024;  // gather small planes until a CTA holds this many pixels

bool fault_injected() {
    const char *v = getenv("WTCONV_INJECT_FAULT");
    return v && v[0] && strcmp(v, "0") != 0;
}

int validate_shape(int B, int C, int H, int W, int L, int k, int dtype) {
    if (B <= 0 || C <= 0 || H <= 0 || W <= 0) return WTCONV_ERR_INVALID_ARG;
    if (L < 1 || L > WTCONV_MAX_LEVELS) return WTCONV_ERR_INVALID_ARG;
    if (k < 1 || (k % 2) == 0) return WTCONV_ERR_INVALID_ARG;
    if ((H % (1 << L)) != 0 || (W % (1 << L)) != 0) return WTCONV_ERR_INVALID_ARG;
    if ((long long)B * C > (1LL << 31) - 1 || (long long)H * W > (1LL << 30)) return WTCONV_ERR_INVALID_ARG;
    if (dtype != WTCONV_F32 && dtype != WTCONV_BF16 && dtype != WTCONV_F16) return WTCONV_ERR_UNSUPPORTED;
    if (k != 3 && k != 5 && k != 7) return WTCONV_ERR_UNSUPPORTED;
    return WTCONV_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned4(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

struct Plan {
    int status = WTCONV_OK;
    LayerArgs a{};
    size_t smem = 0;
    size_t workspace = 0;
};

int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

// Forward and input-gradient kernels: one plane group per CTA.
Plan plan_forward(int B, int C, int H, int W, int L, int k) {
    Plan p;
    LayerArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    a.geo = make_geo(H, W, L, k, /*with_dy=*/false, /*with_z=*/true);
    int G = kTargetSlotPixels / (H * W);
    if (G < 1) G = 1;
    if (G > B) G = B;
    while (G > 1 && fwd_smem_bytes(a.geo, G, L, k) + kStaticSmemMargin > (size_t)kMaxSmem) --G;
    p.smem = fwd_smem_bytes(a.geo, G, L, k);
    if (p.smem + kStaticSmemMargin > (size_t)kMaxSmem) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    a.G = G;
    a.groups_per_cta = 1;
    a.nb = (B + G - 1) / G;
    return p;
}

// Backward kernel: CTAs walk several plane groups of one channel so that the weight-gradient
// partials stay small; about eight waves of resident CTAs keep the tail short.
Plan plan_backward(int B, int C, int H, int W, int L, int k, int dtype, bool want_dx) {
    Plan p;
    LayerArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    a.want_dx = want_dx ? 1 : 0;
    a.geo = make_geo(H, W, L, k, /*with_dy=*/true, /*with_z=*/want_dx);
    int G = kTargetSlotPixels / (H * W);
    if (G < 1) G = 1;
    if (G > B) G = B;
    while (G > 1 && bwd_smem_bytes(a.geo, G, L, k) + kStaticSmemMargin > (size_t)kMaxSmem) --G;
    p.smem = bwd_smem_bytes(a.geo, G, L, k);
    if (p.smem + kStaticSmemMargin > (size_t)kMaxSmem) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    a.G = G;
    const int sms = device_sms();
    const int occ = occupancy_backward(dtype, k, p.smem);
    if (sms <= 0 || occ <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    const int ngroups = (B + G - 1) / G;
    const long long target = 8LL * sms * occ;
    long long nb = (target + C - 1) / C;
    if (nb < 1) nb = 1;
    if (nb > ngroups) nb = ngroups;
    a.groups_per_cta = (int)((ngroups + nb - 1) / nb);
    a.nb = (ngroups + a.groups_per_cta - 1) / a.groups_per_cta;
    p.workspace = (size_t)a.nb * C * (1 + 4 * L) * dw_na(k) * sizeof(float);
    return p;
}

void set_params(LayerArgs &a, const float *base_w, const float *base_bias, const float *base_scale,
                const float *wavelet_w, const float *wavelet_scale) {
    a.base_w = base_w; a.base_bias = base_bias; a.base_scale = base_scale;
    a.wavelet_w = wavelet_w; a.wavelet_scale = wavelet_scale;
}

bool params_ok(const float *base_w, const float *base_bias, const float *base_scale, const float *wavelet_w,
               const float *wavelet_scale) {
    return aligned4(base_w) && aligned4(base_bias) && aligned4(base_scale) && aligned4(wavelet_w) &&
           aligned4(wavelet_scale);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? WTCONV_OK : WTCONV_ERR_CUDA; }

}  // namespace

extern "C" {

int wtconv_version(void) { return 100; }

const char *wtconv_strerror(int status) {
    switch (status) {
    case WTCONV_OK: return "ok";
    case WTCONV_ERR_INVALID_ARG: return "invalid argument (shape, null or misaligned pointer)";
    case WTCONV_ERR_UNSUPPORTED: return "unsupported configuration (dtype, kernel size or plane size)";
    case WTCONV_ERR_WORKSPACE: return "workspace too small";
    case WTCONV_ERR_CUDA: return "CUDA runtime error";
    case WTCONV_ERR_INJECTED: return "fault injected (WTCONV_INJECT_FAULT)";
    default: return "unknown status";
    }
}

size_t wtconv_workspace_size(int op, int B, int C, int H, int W, int L, int k, int dtype) {
    if (validate_shape(B, C, H, W, L, k, dtype) != WTCONV_OK) return 0;
    if (op == WTCONV_OP_BACKWARD_WEIGHTS || op == WTCONV_OP_BACKWARD) {
        Plan p = plan_backward(B, C, H, W, L, k, dtype, op == WTCONV_OP_BACKWARD);
        return p.status == WTCONV_OK ? p.workspace : 0;
    }
    return 0;
}

int wtconv_forward(int B, int C, int H, int W, int L, int k, int dtype, const void *x, const float *base_w,
                   const float *base_bias, const float *base_scale, const float *wavelet_w,
                   const float *wavelet_scale, void *y, void *workspace, size_t workspace_bytes,
                   wtconv_stream_t stream) {
    (void)workspace; (void)workspace_bytes;
    int st = validate_shape(B, C, H, W, L, k, dtype);
    if (st != WTCONV_OK) return st;
    if (!aligned16(x) || !aligned16(y) || !params_ok(base_w, base_bias, base_scale, wavelet_w, wavelet_scale))
        return WTCONV_ERR_INVALID_ARG;
    if (fault_injected()) return WTCONV_ERR_INJECTED;
    Plan p = plan_forward(B, C, H, W, L, k);
    if (p.status != WTCONV_OK) return p.status;
    p.a.x = x; p.a.out = y;
    set_params(p.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
    p.a.flip = 0; p.a.with_bias = 1;
    return cuda_status(launch_forward(p.a, dtype, p.smem, reinterpret_cast<cudaStream_t>(stream)));
}

int wtconv_backward_input(int B, int C, int H, int W, int L, int k, int dtype, const float *base_w,
                          const float *base_bias, const float *base_scale, const float *wavelet_w,
                          const float *wavelet_scale, const void *dy, void *dx, void *workspace,
                          size_t workspace_bytes, wtconv_stream_t stream) {
    (void)workspace; (void)workspace_bytes;
    int st = validate_shape(B, C, H, W, L, k, dtype);
    if (st != WTCONV_OK) return st;
    if (!aligned16(dy) || !aligned16(dx) || !params_ok(base_w, base_bias, base_scale, wavelet_w, wavelet_scale))
        return WTCONV_ERR_INVALID_ARG;
    if (fault_injected()) return WTCONV_ERR_INJECTED;
    Plan p = plan_forward(B, C, H, W, L, k);
    if (p.status != WTCONV_OK) return p.status;
    p.a.x = dy; p.a.out = dx;
    set_params(p.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
    p.a.flip = 1; p.a.with_bias = 0;
    return cuda_status(launch_forward(p.a, dtype, p.smem, reinterpret_cast<cudaStream_t>(stream)));
}

static int backward_common(bool want_dx, int B, int C, int H, int W, int L, int k, int dtype, const void *x,
                           const void *dy, const float *base_w, const float *base_bias, const float *base_scale,
                           const float *wavelet_w, const float *wavelet_scale, void *dx, float *d_base_w,
                           float *d_base_bias, float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale,
                           void *workspace, size_t workspace_bytes, wtconv_stream_t stream) {
    int st = validate_shape(B, C, H, W, L, k, dtype);
    if (st != WTCONV_OK) return st;
    if (!aligned16(x) || !aligned16(dy) || (want_dx && !aligned16(dx)) ||
        !params_ok(base_w, base_bias, base_scale, wavelet_w, wavelet_scale) ||
        !params_ok(d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale))
        return WTCONV_ERR_INVALID_ARG;
    if (fault_injected()) return WTCONV_ERR_INJECTED;
    Plan p = plan_backward(B, C, H, W, L, k, dtype, want_dx);
    if (p.status != WTCONV_OK) return p.status;
    if (workspace_bytes < p.workspace || (p.workspace > 0 && !aligned16(workspace))) return WTCONV_ERR_WORKSPACE;
    p.a.x = x; p.a.dy = dy; p.a.out = want_dx ? dx : nullptr;
    set_params(p.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
    p.a.flip = 1; p.a.with_bias = 0;
    p.a.partials = static_cast<float *>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_backward(p.a, dtype, p.smem, s);
    if (e != cudaSuccess) return WTCONV_ERR_CUDA;
    return cuda_status(launch_dw_finalize(p.a, d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale, s));
}

int wtconv_backward_weights(int B, int C, int H, int W, int L, int k, int dtype, const void *x, const void *dy,
                            const float *base_w, const float *base_bias, const float *base_scale,
                            const float *wavelet_w, const float *wavelet_scale, float *d_base_w,
                            float *d_base_bias, float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale,
                            void *workspace, size_t workspace_bytes, wtconv_stream_t stream) {
    return backward_common(false, B, C, H, W, L, k, dtype, x, dy, base_w, base_bias, base_scale, wavelet_w,
                           wavelet_scale, nullptr, d_base_w, d_base_bias, d_base_scale, d_wavelet_w,
                           d_wavelet_scale, workspace, workspace_bytes, stream);
}

int wtconv_backward(int B, int C, int H, int W, int L, int k, int dtype, const void *x, const void *dy,
                    const float *base_w, const float *base_bias, const float *base_scale, const float *wavelet_w,
                    const float *wavelet_scale, void *dx, float *d_base_w, float *d_base_bias,
                    float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale, void *workspace,
                    size_t workspace_bytes, wtconv_stream_t stream) {
    return backward_common(true, B, C, H, W, L, k, dtype, x, dy, base_w, base_bias, base_scale, wavelet_w,
                           wavelet_scale, dx, d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale,
                           workspace, workspace_bytes, stream);
}

}  // extern "C"
