// Host side of the C ABI declared in include/wtconv.h: argument validation, launch planning
// (plane slots per CTA, CTAs per channel, workspace) and the launches.  Every check runs before
// anything is launched; on error nothing is written.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>

#include "wtconv.h"
#include "wtconv_internal.h"

using namespace wtconv;

namespace {

constexpr int kStaticSmemMargin = 1024;  // static shared memory of the kernels (the Geo copy)

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

// Conv items of one plane: the base image plus two subband-pair images per level.
int items_per_plane(const Geo &g) {
    int n = 0;
    for (int l = 0; l <= g.L; ++l) n += (l == 0 ? 1 : 2) * g.rseg[l] * g.cstr[l];
    return n;
}

// Item balance of the forward's round-robin conv phase on T threads.
double fwd_balance(const Geo &g, int G, int T) {
    const int items = G * items_per_plane(g);
    const int rounds = (items + T - 1) / T;
    return (double)items / ((double)rounds * T);
}

// Balance of the weight-gradient schedule (mirrors the kernel's: each thread takes d items of a
// single correlation; d is the smallest count for which all correlations fit on T threads).
double dw_balance(const Geo &g, int G, int T) {
    int tot = 0;
    const int nimg = 1 + 2 * g.L;
    for (int s = 0; s < nimg; ++s) {
        const int l = s == 0 ? 0 : (s - 1) / 2 + 1;
        tot += G * g.rseg[l] * g.cstr[l];
    }
    int d = (tot + T - 1) / T;
    if (d < 1) d = 1;
    for (;; ++d) {
        int need = 0;
        for (int s = 0; s < nimg; ++s) {
            const int l = s == 0 ? 0 : (s - 1) / 2 + 1;
            need += (G * g.rseg[l] * g.cstr[l] + d - 1) / d;
        }
        if (need <= T) break;
    }
    return (double)tot / ((double)d * T);
}

int elem_bytes(int dtype) { return dtype == WTCONV_F32 ? 4 : 2; }

void set_io_modes(LayerArgs &a, int dtype) {
    a.vec_ld = (a.W % 4) == 0;
    if (dtype == WTCONV_F32) a.st_mode = (a.W % 4) == 0 ? 2 : 0;
    else a.st_mode = (a.W % 8) == 0 ? 2 : ((a.W % 4) == 0 ? 1 : 0);
    // staged copies move whole planes in 16-byte pieces
    a.stage = ((size_t)a.H * a.W * elem_bytes(dtype)) % 16 == 0;
}

// Fast-division magic numbers of every runtime divisor the kernels use.
void set_divs(LayerArgs &a, int dtype) {
    const Geo &g = a.geo;
    Divs &d = a.dv;
    d = Divs{};
    // analysis pass 1 (levels 1-2 from 4x4 blocks, or level 1 from 2x2 blocks when L == 1)
    if (g.L >= 2) { d.a_w[1] = make_fastdiv(g.W >> 2); d.a_n[1] = make_fastdiv((g.H >> 2) * (g.W >> 2)); }
    else { d.a_w[1] = make_fastdiv(g.W >> 1); d.a_n[1] = make_fastdiv((g.H >> 1) * (g.W >> 1)); }
    for (int l = 3; l <= g.L; l += 2) {  // deeper passes from the level l-1 low band
        const int hs = g.h[l - 1], ws = g.w[l - 1];
        if (l + 1 <= g.L) { d.a_w[l] = make_fastdiv(ws >> 2); d.a_n[l] = make_fastdiv((hs >> 2) * (ws >> 2)); }
        else { d.a_w[l] = make_fastdiv(ws >> 1); d.a_n[l] = make_fastdiv((hs >> 1) * (ws >> 1)); }
    }
    d.stage_chunks = make_fastdiv((uint32_t)((size_t)g.H * g.W * elem_bytes(dtype) / 16));
    for (int l = 0; l <= g.L; ++l) {
        d.item_plane[l] = make_fastdiv(g.rseg[l] * g.cstr[l]);
        d.item_cols[l] = make_fastdiv(g.cstr[l]);
    }
    const int nws = (g.W + 7) / 8;
    d.out_w = make_fastdiv(nws);
    d.out_n = make_fastdiv(g.H * nws);
}

typedef size_t (*SmemFn)(const Geo &, int, int, int, int, bool, int *);
typedef double (*BalFn)(const Geo &, int, int);
typedef int (*OccFn)(int, int, int, size_t);

// Planes per CTA (G), CTA size (T) and staging: score = item balance x resident warps per SM
// (capped at 32), over G whose shared memory fits; ties go to staging, then to the smaller G.
// Staging through shared memory hides the next planes' load latency but costs shared memory;
// without it the next planes are only prefetched into L2.  WTCONV_STAGE=0/1 forces the choice.
bool choose_launch(LayerArgs &a, int dtype, SmemFn smem_fn, BalFn bal_fn, OccFn occ_fn, size_t *smem_out) {
    const int eb = elem_bytes(dtype);
    const bool can_stage = a.stage != 0;
    const char *force = getenv("WTCONV_STAGE");
    double best = -1.0;
    int bestG = 0, bestT = 0, bestS = 0;
    for (int stage : {1, 0}) {
        if (stage && !can_stage) continue;
        if (force && force[0] == '0' && stage) continue;
        if (force && force[0] == '1' && !stage && can_stage) continue;
        for (int T : {256, 128}) {
            for (int G = 1; G <= a.B && G <= 64; ++G) {
                const size_t smem = smem_fn(a.geo, G, a.L, a.K, eb, stage != 0, nullptr);
                if (smem + kStaticSmemMargin > (size_t)kMaxSmem) break;
                const int occ = occ_fn(dtype, a.K, T, smem);
                if (occ <= 0) continue;
                int warps = occ * T / 32;
                if (warps > 32) warps = 32;
                const double score = bal_fn(a.geo, G, T) * warps;
                if (score > best + 1e-9) { best = score; bestG = G; bestT = T; bestS = stage; }
            }
        }
    }
    if (bestG == 0) return false;
    a.G = bestG;
    a.threads = bestT;
    a.stage = bestS;
    int off = 0;
    *smem_out = smem_fn(a.geo, bestG, a.L, a.K, eb, bestS != 0, &off);
    a.stage_off = off;
    return true;
}

// Forward and input-gradient kernel.
Plan plan_forward_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    Plan p;
    LayerArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    a.geo = make_geo(H, W, L, k, 0);
    set_io_modes(a, dtype);
    const int sms = device_sms();
    if (sms <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    if (!choose_launch(a, dtype, fwd_smem_bytes, fwd_balance, occupancy_forward, &p.smem)) {
        p.status = WTCONV_ERR_UNSUPPORTED;
        return p;
    }
    set_divs(a, dtype);
    const int occ = occupancy_forward(dtype, k, a.threads, p.smem);
    const int ngroups = (B + a.G - 1) / a.G;
    const long long target = 4LL * sms * occ;  // about four waves of resident CTAs
    long long nb = (target + C - 1) / C;
    if (nb < 1) nb = 1;
    if (nb > ngroups) nb = ngroups;
    a.groups_per_cta = (int)((ngroups + nb - 1) / nb);
    a.nb = (ngroups + a.groups_per_cta - 1) / a.groups_per_cta;
    return p;
}

// Weight-gradient kernel: fewer, longer-lived CTAs keep the per-CTA partials small.
Plan plan_dw_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    Plan p;
    LayerArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    a.geo = make_geo(H, W, L, k, 1);
    set_io_modes(a, dtype);
    const int sms = device_sms();
    if (sms <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    if (!choose_launch(a, dtype, dw_smem_bytes, dw_balance, occupancy_dw, &p.smem)) {
        p.status = WTCONV_ERR_UNSUPPORTED;
        return p;
    }
    set_divs(a, dtype);
    const int occ = occupancy_dw(dtype, k, a.threads, p.smem);
    const int ngroups = (B + a.G - 1) / a.G;
    const long long target = 4LL * sms * occ;
    long long nb = (target + C - 1) / C;
    if (nb < 1) nb = 1;
    if (nb > ngroups) nb = ngroups;
    a.groups_per_cta = (int)((ngroups + nb - 1) / nb);
    a.nb = (ngroups + a.groups_per_cta - 1) / a.groups_per_cta;
    p.workspace = (size_t)a.nb * C * (1 + 4 * L) * (k * k + 1) * sizeof(float);
    return p;
}

// Plans depend only on the shape, dtype and device; they are computed once and reused (the
// occupancy queries behind them cost far more than a launch).
typedef std::tuple<int, int, int, int, int, int, int, int, int> PlanKey;

Plan cached_plan(int kind, int B, int C, int H, int W, int L, int k, int dtype) {
    static std::mutex mu;
    static std::map<PlanKey, Plan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        Plan p;
        p.status = WTCONV_ERR_CUDA;
        return p;
    }
    const PlanKey key(kind, B, C, H, W, L, k, dtype, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    Plan p = kind == 0 ? plan_forward_uncached(B, C, H, W, L, k, dtype) : plan_dw_uncached(B, C, H, W, L, k, dtype);
    const char *verbose = getenv("WTCONV_VERBOSE");
    if (verbose && verbose[0] == '1')
        fprintf(stderr, "wtconv plan %s B=%d C=%d H=%d W=%d L=%d k=%d dtype=%d: status %d G=%d threads=%d nb=%d "
                        "groups/cta=%d smem=%zu stage=%d workspace=%zu\n",
                kind == 0 ? "fwd" : "dw", B, C, H, W, L, k, dtype, p.status, p.a.G, p.a.threads, p.a.nb,
                p.a.groups_per_cta, p.smem, p.a.stage, p.workspace);
    if (p.status == WTCONV_OK) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, p);
    }
    return p;
}

Plan plan_forward(int B, int C, int H, int W, int L, int k, int dtype) {
    return cached_plan(0, B, C, H, W, L, k, dtype);
}

Plan plan_dw(int B, int C, int H, int W, int L, int k, int dtype) {
    return cached_plan(1, B, C, H, W, L, k, dtype);
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
        Plan p = plan_dw(B, C, H, W, L, k, dtype);
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
    Plan p = plan_forward(B, C, H, W, L, k, dtype);
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
    Plan p = plan_forward(B, C, H, W, L, k, dtype);
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
    Plan pw = plan_dw(B, C, H, W, L, k, dtype);
    if (pw.status != WTCONV_OK) return pw.status;
    Plan pf;
    if (want_dx) {
        pf = plan_forward(B, C, H, W, L, k, dtype);
        if (pf.status != WTCONV_OK) return pf.status;
    }
    if (workspace_bytes < pw.workspace || (pw.workspace > 0 && !aligned16(workspace))) return WTCONV_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (want_dx) {
        pf.a.x = dy; pf.a.out = dx;
        set_params(pf.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
        pf.a.flip = 1; pf.a.with_bias = 0;
        if (launch_forward(pf.a, dtype, pf.smem, s) != cudaSuccess) return WTCONV_ERR_CUDA;
    }
    pw.a.x = x; pw.a.dy = dy;
    set_params(pw.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
    pw.a.partials = static_cast<float *>(workspace);
    if (launch_dw(pw.a, dtype, pw.smem, s) != cudaSuccess) return WTCONV_ERR_CUDA;
    return cuda_status(launch_dw_finalize(pw.a, d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale, s));
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
