// Host side of the C ABI declared in include/wtconv.h: argument validation, launch planning
// (plane slots per CTA, CTAs per channel, workspace) and the launches.  Every check runs before
// anything is launched; on error nothing is written.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "wtconv.h"
#include "wtconv_internal.h"
#include "wtconv_pad.h"
#include "wtconv_pair.cuh"
#include "wtconv_pshallow.h"
#include "wtconv_ptile.h"
#include "wtconv_selftest.h"

using namespace wtconv;

namespace {

constexpr int kStaticSmemMargin = 1024;  // static shared memory of the kernels (the Geo copy)

bool fault_injected() {
    const char *v = getenv("WTCONV_INJECT_FAULT");
    return v && v[0] && strcmp(v, "0") != 0;
}

// Shapes the public entry points accept.  Sides need not be multiples of 2^L: such planes run
// zero-padded to the next multiples (see PadDims); the limits apply to the padded planes.
int validate_shape(int B, int C, int H, int W, int L, int k, int dtype) {
    if (B <= 0 || C <= 0 || H <= 0 || W <= 0) return WTCONV_ERR_INVALID_ARG;
    if (L < 1 || L > WTCONV_MAX_LEVELS) return WTCONV_ERR_INVALID_ARG;
    if (k < 1 || (k % 2) == 0) return WTCONV_ERR_INVALID_ARG;
    if (H > (1 << 30) || W > (1 << 30)) return WTCONV_ERR_INVALID_ARG;
    const long long m = 1LL << L, Hp = (H + m - 1) / m * m, Wp = (W + m - 1) / m * m;
    if ((long long)B * C > (1LL << 31) - 1 || Hp * Wp > (1LL << 30)) return WTCONV_ERR_INVALID_ARG;
    if (dtype != WTCONV_F32 && dtype != WTCONV_BF16 && dtype != WTCONV_F16) return WTCONV_ERR_UNSUPPORTED;
    if (k != 3 && k != 5 && k != 7) return WTCONV_ERR_UNSUPPORTED;
    return WTCONV_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned4(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

// Planes whose sides are not multiples of 2^L run as the plane zero-padded at the end of each
// side to the next multiples, cropped back (equal to padding each level's odd sides with one zero
// at the end before the analysis and cropping each reconstruction: a padded row or column is never
// an ancestor of a pixel inside the plane).  The padded activations live in the workspace.
struct PadDims {
    bool on;
    int Hp, Wp;
    size_t act_bytes;  // one padded activation tensor, 256-byte rounded
};
PadDims pad_dims(int B, int C, int H, int W, int L, int dtype) {
    PadDims p;
    const int m = 1 << L;
    p.Hp = (H + m - 1) / m * m;
    p.Wp = (W + m - 1) / m * m;
    p.on = p.Hp != H || p.Wp != W;
    const size_t eb = dtype == WTCONV_F32 ? 4 : 2;
    p.act_bytes = ((size_t)B * C * p.Hp * p.Wp * eb + 255) / 256 * 256;
    return p;
}

struct Plan {
    int status = WTCONV_OK;
    LayerArgs a{};
    size_t smem = 0;
    size_t workspace = 0;
    int dw_pyramid = 0;  // weight gradient: 1 = pyramids in the workspace + tiled correlations
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
    // tuning restriction: WTCONV_STAGED=G,threads fixes the planes per slot group and CTA size
    int kg = 0, kt = 0;
    const char *kn = getenv("WTCONV_STAGED");
    if (kn && kn[0]) sscanf(kn, "%d,%d", &kg, &kt);
    double best = -1.0;
    int bestG = 0, bestT = 0, bestS = 0;
    for (int stage : {1, 0}) {
        if (stage && !can_stage) continue;
        if (force && force[0] == '0' && stage) continue;
        if (force && force[0] == '1' && !stage && can_stage) continue;
        for (int T : {256, 128}) {
            if (kt && T != kt) continue;
            for (int G = 1; G <= a.B && G <= 64; ++G) {
                if (kg && G != kg) continue;
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

// Whole-plane forward / input-gradient kernel; UNSUPPORTED when a plane's pyramid does not fit.
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
Plan plan_dw_uncached(int B, int C, int H, int W, int L, int k, int dtype, bool force_pyramid) {
    Plan p;
    LayerArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    a.geo = make_geo(H, W, L, k, 1);
    set_io_modes(a, dtype);
    const int sms = device_sms();
    if (sms <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    if (force_pyramid || !choose_launch(a, dtype, dw_smem_bytes, dw_balance, occupancy_dw, &p.smem)) {
        // planes too large for shared memory: pyramids in the workspace, tiled correlations
        p.dw_pyramid = 1;
        const long long units0 = (long long)B * ((H + 15) / 16) * ((W + 63) / 64);
        long long nb = (8LL * sms + C - 1) / C;
        if (nb > units0) nb = units0;
        if (nb < 1) nb = 1;
        a.nb = (int)nb;
        p.workspace = dw_pyramid_bytes(B, C, H, W, L, 1) +
                      ((size_t)a.nb * C * (1 + 4 * L) * (k * k + 1) * sizeof(float) + 255) / 256 * 256;
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

// Deep kernel (levels >= 2; only when L >= 2): like the forward planner, on a levels>=2 slot.
double deep_balance(const Geo &g, int G, int T) {
    int items = 0;
    for (int l = 2; l <= g.L; ++l) items += 2 * g.rseg[l] * g.cstr[l];
    items *= G;
    const int rounds = (items + T - 1) / T;
    return rounds > 0 ? (double)items / ((double)rounds * T) : 0.0;
}

Plan plan_deep_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    Plan p;
    LayerArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    a.geo = make_geo(H, W, L, k, 2);
    set_io_modes(a, dtype);
    const int sms = device_sms();
    if (sms <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    if (!choose_launch(a, dtype, deep_smem_bytes, deep_balance, occupancy_deep, &p.smem)) {
        p.status = WTCONV_ERR_UNSUPPORTED;
        return p;
    }
    set_divs(a, dtype);
    // pass 1 reads 4 x 4 pixel blocks; the output is D at level-1 resolution in segments of 8
    a.dv.a_w[1] = make_fastdiv(W >> 2);
    a.dv.a_n[1] = make_fastdiv((H >> 2) * (W >> 2));
    const int nws = ((W >> 1) + 7) / 8;
    a.dv.out_w = make_fastdiv(nws);
    a.dv.out_n = make_fastdiv((H >> 1) * nws);
    const int occ = occupancy_deep(dtype, k, a.threads, p.smem);
    const int ngroups = (B + a.G - 1) / a.G;
    const long long target = 4LL * sms * occ;
    long long nb = (target + C - 1) / C;
    if (nb < 1) nb = 1;
    if (nb > ngroups) nb = ngroups;
    a.groups_per_cta = (int)((ngroups + nb - 1) / nb);
    a.nb = (ngroups + a.groups_per_cta - 1) / a.groups_per_cta;
    return p;
}

struct SPlan {
    int status = WTCONV_OK;
    ShallowArgs a{};
    size_t smem = 0;
};

// Shallow kernel tiles: full-width tiles up to 64 columns, at most 32 fused 8x4 items per tile
// (one per lane); small planes are packed G to a unit.  Copy chunks are the widest of 16, 8 and
// 4 bytes for which every chunk lies wholly inside or outside the plane.
SPlan plan_shallow_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    SPlan p;
    ShallowArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    a.st_mode = (W % 4) == 0 ? 1 : 0;
    const int W4 = round_up(W, 4);
    const int TW = W4 <= 64 ? W4 : 64;
    const int items_c = TW / kCols;
    int rows_of_items = 32 / items_c;
    if (rows_of_items < 1) rows_of_items = 1;
    int TH = kRows * rows_of_items;
    if (TH > round_up(H, kRows)) TH = round_up(H, kRows);
    int G = 1;
    if (TH >= H && TW >= W) {
        G = 32 / (items_c * (TH / kRows));
        if (G < 1) G = 1;
        if (G > B) G = B;
    }
    const int eb = elem_bytes(dtype);
    int chunk_e = 16 / eb;
    while (chunk_e > 1 && (W % chunk_e != 0 || TW % chunk_e != 0)) chunk_e /= 2;
    if (chunk_e * eb < 4) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    const int W1 = W / 2;
    const int dchunk_e = (W1 % 4 == 0 && (TW / 2) % 4 == 0) ? 4 : 2;
    const bool convert = eb != 4, deep = L >= 2;
    a.sg = make_shallow_geo(H, W, k, TH, TW, G, eb, chunk_e, dchunk_e);
    p.smem = shallow_smem_bytes(a.sg, k, convert, deep);
    // planes per unit: as many as fill the warp's lanes and fit in shared memory
    while (G > 1 && p.smem + kStaticSmemMargin > (size_t)kMaxSmem) {
        --G;
        a.sg = make_shallow_geo(H, W, k, TH, TW, G, eb, chunk_e, dchunk_e);
        p.smem = shallow_smem_bytes(a.sg, k, convert, deep);
    }
    if (p.smem + kStaticSmemMargin > (size_t)kMaxSmem) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    const int sms = device_sms();
    const int occ = occupancy_shallow(dtype, k, p.smem);
    if (sms <= 0 || occ <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    const int tiles = a.sg.tiles_r * a.sg.tiles_c;
    a.units = ((B + G - 1) / G) * tiles;
    // CTAs per channel: minimise (waves of resident CTAs) x (units per CTA)
    const long long slots = (long long)sms * occ;
    long long best_nb = 1, best_cost = -1;
    const long long max_nb = std::max(1, a.units);
    for (long long nb = 1; nb <= max_nb; ++nb) {
        const long long upc = (a.units + nb - 1) / nb;
        const long long waves = (C * nb + slots - 1) / slots;
        const long long cost = waves * upc;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_nb = nb; }
    }
    a.units_per_cta = (int)((a.units + best_nb - 1) / best_nb);
    a.nb = (a.units + a.units_per_cta - 1) / a.units_per_cta;
    a.tiles = make_fastdiv(tiles);
    a.tiles_c = make_fastdiv(a.sg.tiles_c);
    a.rchunks_row = make_fastdiv(a.sg.xw / chunk_e);
    a.xrows = make_fastdiv(a.sg.xrows);
    a.dchunks_row = make_fastdiv((TW / 2) / dchunk_e);
    a.drows = make_fastdiv(TH / 2);
    a.ycols = make_fastdiv(a.sg.ycols);
    a.xw4 = make_fastdiv(a.sg.xw / 4);
    return p;
}

// Bytes of the deep contribution (level-1 resolution, fp32, 16-byte rounded); 0 when L == 1.
size_t deep_bytes(int B, int C, int H, int W, int L) {
    if (L < 2) return 0;
    return ((size_t)B * C * (H >> 1) * (W >> 1) * sizeof(float) + 255) / 256 * 256;
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
    // the tuning restrictions are part of the key
    int kg = 0, kt = 0;
    const char *kn = getenv("WTCONV_STAGED"), *ks = getenv("WTCONV_STAGE");
    if (kn && kn[0]) sscanf(kn, "%d,%d", &kg, &kt);
    const int knobs = (kg * 512 + kt) * 4 + (ks && ks[0] ? (ks[0] == '1' ? 1 : 2) : 0);
    const PlanKey key(kind + 16 * knobs, B, C, H, W, L, k, dtype, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    Plan p = kind == 0   ? plan_forward_uncached(B, C, H, W, L, k, dtype)
             : kind == 1 ? plan_dw_uncached(B, C, H, W, L, k, dtype, false)
             : kind == 5 ? plan_dw_uncached(B, C, H, W, L, k, dtype, true)
                         : plan_deep_uncached(B, C, H, W, L, k, dtype);
    const char *verbose = getenv("WTCONV_VERBOSE");
    if (verbose && verbose[0] == '1')
        fprintf(stderr, "wtconv plan %s B=%d C=%d H=%d W=%d L=%d k=%d dtype=%d: status %d G=%d threads=%d nb=%d "
                        "groups/cta=%d smem=%zu stage=%d workspace=%zu\n",
                kind == 0 ? "fwd" : kind == 1 ? "dw" : "deep", B, C, H, W, L, k, dtype, p.status, p.a.G, p.a.threads, p.a.nb,
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

Plan plan_deep(int B, int C, int H, int W, int L, int k, int dtype) {
    return cached_plan(2, B, C, H, W, L, k, dtype);
}

SPlan plan_shallow(int B, int C, int H, int W, int L, int k, int dtype) {
    static std::mutex mu;
    static std::map<PlanKey, SPlan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        SPlan p;
        p.status = WTCONV_ERR_CUDA;
        return p;
    }
    const PlanKey key(3, B, C, H, W, L, k, dtype, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    SPlan p = plan_shallow_uncached(B, C, H, W, L, k, dtype);
    const char *verbose = getenv("WTCONV_VERBOSE");
    if (verbose && verbose[0] == '1')
        fprintf(stderr, "wtconv plan shallow B=%d C=%d H=%d W=%d L=%d k=%d dtype=%d: status %d TH=%d TW=%d G=%d "
                        "units=%d units/cta=%d nb=%d smem=%zu\n",
                B, C, H, W, L, k, dtype, p.status, p.a.sg.TH, p.a.sg.TW, p.a.sg.G, p.a.units, p.a.units_per_cta,
                p.a.nb, p.smem);
    if (p.status == WTCONV_OK) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, p);
    }
    return p;
}

Plan plan_dw(int B, int C, int H, int W, int L, int k, int dtype) {
    return cached_plan(1, B, C, H, W, L, k, dtype);
}

Plan plan_dw_pyramid_only(int B, int C, int H, int W, int L, int k, int dtype) {
    return cached_plan(5, B, C, H, W, L, k, dtype);
}

// ------------------------------------------------------------------ bulk tensor copies (TMA)

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once (nullptr if unavailable).
EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor map of a contiguous [B][C][H][W] tensor with a box of bw x bh x 1 x bb elements
// (zero fill outside).  False if the driver refuses it.
bool encode_map(CUtensorMap *m, CUtensorMapDataType dt, int eb, const void *base, int W, int H, int C, int B,
                int bw, int bh, int bb) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)C, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)W * eb, (cuuint64_t)H * W * eb, (cuuint64_t)C * H * W * eb};
    const cuuint32_t box[4] = {(cuuint32_t)bw, (cuuint32_t)bh, 1u, (cuuint32_t)bb};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same for planes stored with a row pitch of `pitch` elements (pitch * eb a multiple of 16).
bool encode_map_pitched(CUtensorMap *m, CUtensorMapDataType dt, int eb, const void *base, int W, int H, int C, int B,
                        int pitch, int bw, int bh, int bb) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)C, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)pitch * eb, (cuuint64_t)H * pitch * eb, (cuuint64_t)C * H * pitch * eb};
    const cuuint32_t box[4] = {(cuuint32_t)bw, (cuuint32_t)bh, 1u, (cuuint32_t)bb};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Whether the shallow kernel's tiles can move as bulk tensor copies: every row, box row and box
// origin 16-byte aligned, box extents within the hardware limit of 256.
bool shallow_tma_x_ok(const ShallowArgs &a, int eb) {
    const ShallowGeo &g = a.sg;
    return ((size_t)a.W * eb) % 16 == 0 && ((size_t)g.xw * eb) % 16 == 0 && ((size_t)g.padx * eb) % 16 == 0 &&
           ((size_t)g.TW * eb) % 16 == 0 && g.xw <= 256 && g.xrows <= 256 && g.G <= 256;
}
bool shallow_tma_d_ok(const ShallowArgs &a) {
    const ShallowGeo &g = a.sg;
    return a.L >= 2 && ((a.W / 2) % 4) == 0 && ((g.TW / 2) % 4) == 0 && g.TW / 2 <= 256 && g.TH / 2 <= 256;
}

CUtensorMapDataType tma_dtype(int dtype) {
    return dtype == WTCONV_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                               : dtype == WTCONV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// ------------------------------------------------------------------ tiled batch-pair shallow kernel

struct PsPlan {
    int status = WTCONV_ERR_UNSUPPORTED;
    PsArgs a{};
    size_t smem = 0;
    int occ = 0;
};

// Geometry of one tile shape: false where the bulk tensor copies or the item shapes do not apply
// (tile rows a multiple of 16 so that level 1 holds whole 8-row items; every copy origin, row and
// box row 16-byte aligned; box extents within 256).
bool ps_make(PsArgs &a, int B, int C, int H, int W, int K, int eb, bool deep, int TH, int TW, int G, int nt, int S) {
    a = PsArgs{};
    const int P = K / 2, al = 16 / eb;
    a.B = B; a.C = C; a.H = H; a.W = W; a.K = K;
    a.TH = TH; a.TW = TW; a.G = G; a.nthreads = nt;
    a.HX = 2 * P;
    a.HXL = (a.HX + al - 1) / al * al;
    a.RXR = TH + 2 * a.HX;
    a.RXW = (a.HXL + TW + a.HX + al - 1) / al * al;
    if (TH <= 0 || TW <= 0 || TH % 16 != 0 || TW % 8 != 0 || H % 2 != 0 || W % 8 != 0) return false;
    if (S != 4 && S != 8) return false;
    if (((size_t)W * eb) % 16 != 0 || ((size_t)TW * eb) % 16 != 0) return false;
    if (a.RXW > 256 || a.RXR > 256 || 2 * G > 256 || TW / 2 > 256 || TH / 2 > 256) return false;
    const int TH1 = TH / 2, TW1 = TW / 2;
    a.tiles_r = (H + TH - 1) / TH;
    a.tiles_c = (W + TW - 1) / TW;
    a.tiles = a.tiles_r * a.tiles_c;
    a.npairs = (B + 1) / 2;
    a.ngroups = (a.npairs + G - 1) / G;
    if ((long long)C * a.tiles * a.ngroups > (long long)INT32_MAX / 2) return false;
    a.work = C * a.tiles * a.ngroups;
    a.q0 = 2; a.s0 = S;
    a.ns0 = TW / 2; a.ng0 = TH / S;
    a.ipitch0 = pg_round2(TW + 2 * P);
    a.irows0 = TH + 2 * P;
    a.q1 = 2; a.s1 = S;
    a.ns1 = TW1 / 2; a.ng1 = TH1 / S;
    a.ipitch1 = pg_round2(TW1 + 2 * P);
    a.irows1 = TH1 + 2 * P;
    a.iimg1 = a.ipitch1 * a.irows1;
    a.zpitch1 = pg_round2(TW1);
    a.zrows1 = TH1;
    a.zimg1 = a.zpitch1 * a.zrows1;
    a.off_x = 0;
    a.off_y1 = a.ipitch0 * a.irows0;
    a.off_z1 = a.off_y1 + 4 * a.iimg1;
    a.slot = pg_round2(a.off_z1 + 5 * a.zimg1);
    a.raw_x_bytes = (int)(((size_t)2 * G * a.RXR * a.RXW * eb + 127) / 128 * 128);
    a.has_deep = deep ? 1 : 0;
    a.raw_d_bytes = deep ? (int)(((size_t)2 * G * TH1 * TW1 * sizeof(float) + 127) / 128 * 128) : 0;
    a.vec_st = 1;  // W even, items 2 columns wide at even columns
    const int xbw = (TW + 2 * a.HX) / 2, xbh = (TH + 2 * a.HX) / 2;
    a.dv_work_c = make_fastdiv(a.tiles * a.ngroups);
    a.dv_tiles = make_fastdiv(a.tiles);
    a.dv_tiles_c = make_fastdiv(a.tiles_c);
    a.dv_xb = make_fastdiv(xbw * xbh);
    a.dv_xbw = make_fastdiv(xbw);
    a.dv_conv = make_fastdiv(4 * a.ns1 * a.ng1);
    a.dv_ns1 = make_fastdiv(a.ns1);
    a.dv_out = make_fastdiv(a.ns0 * a.ng0);
    a.dv_ns0 = make_fastdiv(a.ns0);
    a.dv_db = make_fastdiv(TH1 * TW1);
    a.dv_dbw = make_fastdiv(TW1);
    return true;
}

// Tuning restrictions (0: planner's choice): WTCONV_PSHALLOW=TH,TW,G,threads,item rows.
void ps_knobs(int &th, int &tw, int &g, int &nt, int &sr) {
    th = tw = g = nt = sr = 0;
    const char *v = getenv("WTCONV_PSHALLOW");
    if (v && v[0]) sscanf(v, "%d,%d,%d,%d,%d", &th, &tw, &g, &nt, &sr);
}

PsPlan plan_pshallow_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    PsPlan p;
    const int eb = elem_bytes(dtype);
    if (B < 1 || L < 1 || H % (1 << L) != 0 || W % (1 << L) != 0) return p;
    const int sms = device_sms();
    if (sms <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    int kth = 0, ktw = 0, kg = 0, knt = 0, ksr = 0;
    ps_knobs(kth, ktw, kg, knt, ksr);
    const int Hr = (H + 15) / 16 * 16, Wr = (W + 7) / 8 * 8;
    double best_score = -1.0;
    for (int th0 : {16, 32}) {
        const int TH = std::min(th0, Hr);
        if (kth && TH != kth) continue;
        if (th0 > 16 && TH < th0) continue;  // the same tile as th0 = 16
        for (int tw0 : {32, 64}) {
            const int TW = std::min(tw0, Wr);
            if (ktw && TW != ktw) continue;
            if (tw0 > 32 && TW < tw0) continue;
            for (int ns : {0, 1, 2, 3}) {  // (threads, item rows): (64, 8), (64, 4), (128, 8), (128, 4)
                const int nt = ns < 2 ? 64 : 128, S = (ns & 1) ? 4 : 8;
                if (knt && nt != knt) continue;
                if (ksr && S != ksr) continue;
                for (int G = 1; G <= 8; ++G) {
                    if (kg && G != kg) continue;
                    PsArgs a;
                    if (!ps_make(a, B, C, H, W, k, eb, L >= 2, TH, TW, G, nt, S)) break;
                    if (G > a.npairs) break;
                    const size_t smem = pshallow_smem_bytes(a);
                    if (smem + kStaticSmemMargin > (size_t)kMaxSmem) break;
                    const int occ = occupancy_pshallow(dtype, k, smem, nt, S);
                    if (occ <= 0) break;
                    // resident threads first (the FMA chains of one item are long; more warps hide
                    // the shared-memory latency), then how evenly a group's items fill the threads,
                    // then the share of the x tile that is halo (pass-1 work and L2 reads)
                    const long long items = (long long)G * a.ns0 * a.ng0;
                    const double fill = (double)items / ((double)((items + nt - 1) / nt) * nt);
                    const double resident = std::min(768.0, (double)occ * nt) / 768.0;
                    const double halo = (double)(TH * TW) / ((double)a.RXR * (TW + 2 * a.HX));
                    const double tiles_used = (double)H * W / ((double)a.tiles * TH * TW);
                    const double score = resident * std::sqrt(fill) * std::sqrt(halo) * tiles_used;
                    const char *vb = getenv("WTCONV_VERBOSE");
                    if (vb && vb[0] == '2')
                        fprintf(stderr, "  pshallow candidate %dx%d G=%d nt=%d S=%d smem=%zu occ=%d fill=%.3f halo=%.3f score=%.4f\n",
                                TH, TW, G, nt, S, smem, occ, fill, halo, score);
                    if (score > best_score) {
                        best_score = score;
                        p.a = a;
                        p.smem = smem;
                        p.occ = occ;
                    }
                }
            }
        }
    }
    if (best_score <= 0.0) return p;
    p.a.grid = (int)std::min<long long>(p.a.work, (long long)sms * p.occ);
    p.status = WTCONV_OK;
    return p;
}

PsPlan plan_pshallow(int B, int C, int H, int W, int L, int k, int dtype) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, int, int, int, std::string>, PsPlan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        PsPlan p;
        p.status = WTCONV_ERR_CUDA;
        return p;
    }
    const char *kn = getenv("WTCONV_PSHALLOW");
    const auto key = std::make_tuple(B, C, H, W, L, k, dtype, dev, std::string(kn ? kn : ""));
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    PsPlan p = plan_pshallow_uncached(B, C, H, W, L, k, dtype);
    const char *verbose = getenv("WTCONV_VERBOSE");
    if (verbose && verbose[0] == '1')
        fprintf(stderr, "wtconv plan pshallow B=%d C=%d H=%d W=%d L=%d k=%d dtype=%d: status %d tile=%dx%d G=%d "
                        "threads=%d rows=%d work=%d grid=%d smem=%zu occ=%d\n",
                B, C, H, W, L, k, dtype, p.status, p.a.TH, p.a.TW, p.a.G, p.a.nthreads, p.a.s0, p.a.work, p.a.grid,
                p.smem, p.occ);
    if (p.status == WTCONV_OK || p.status == WTCONV_ERR_UNSUPPORTED) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, p);
    }
    return p;
}

// Tiled weight gradient: the shallow kernel's tiles (bulk tensor copies of x and dy, tiles of a
// multiple of 16 rows); UNSUPPORTED where those do not apply.
struct TPlan {
    int status = WTCONV_OK;
    DwTileArgs a{};
    size_t smem = 0;
    size_t workspace = 0;  // partials, then the pyramids of levels >= 2
    size_t partial_bytes = 0;
};

TPlan plan_dw_tile_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    TPlan p;
    const SPlan ps = plan_shallow(B, C, H, W, L, k, dtype);
    if (ps.status != WTCONV_OK) { p.status = ps.status; return p; }
    const ShallowGeo &sg = ps.a.sg;
    const int eb = elem_bytes(dtype);
    if (!shallow_tma_x_ok(ps.a, eb) || sg.TH % 16 != 0 || ((size_t)sg.TW * eb) % 16 != 0 || sg.TH > 256 ||
        sg.TW > 256) {
        p.status = WTCONV_ERR_UNSUPPORTED;
        return p;
    }
    DwTileArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    a.sg = sg;
    p.smem = dw_tile_smem_bytes(sg, eb);
    if (p.smem + kStaticSmemMargin > (size_t)kMaxSmem) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    const int sms = device_sms();
    const int occ = occupancy_dw_tile(dtype, k, p.smem);
    if (sms <= 0 || occ <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    const int tiles = sg.tiles_r * sg.tiles_c;
    a.units = ((B + sg.G - 1) / sg.G) * tiles;
    // CTAs per channel: minimise (waves) x (units per CTA) over at most two waves of resident
    // CTAs -- every CTA per channel adds a row of partials and a CTA to each level correlation
    const long long slots = (long long)sms * occ;
    const long long nb_max = std::max(1LL, std::min((long long)a.units, 2 * slots / C));
    long long best_nb = 1, best_cost = -1;
    for (long long nb = 1; nb <= nb_max; ++nb) {
        const long long cost = ((C * nb + slots - 1) / slots) * ((a.units + nb - 1) / nb);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_nb = nb; }
    }
    a.units_per_cta = (int)((a.units + best_nb - 1) / best_nb);
    a.nb = (a.units + a.units_per_cta - 1) / a.units_per_cta;
    a.tiles = make_fastdiv(tiles);
    a.tiles_c = make_fastdiv(sg.tiles_c);
    p.partial_bytes = ((size_t)a.nb * C * (1 + 4 * L) * (k * k + 1) * sizeof(float) + 255) / 256 * 256;
    p.workspace = p.partial_bytes + (L >= 2 ? dw_pyramid_bytes(B, C, H, W, L, 2) : 0);
    return p;
}

TPlan plan_dw_tile(int B, int C, int H, int W, int L, int k, int dtype) {
    static std::mutex mu;
    static std::map<PlanKey, TPlan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        TPlan p;
        p.status = WTCONV_ERR_CUDA;
        return p;
    }
    const PlanKey key(6, B, C, H, W, L, k, dtype, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    TPlan p = plan_dw_tile_uncached(B, C, H, W, L, k, dtype);
    if (p.status == WTCONV_OK || p.status == WTCONV_ERR_UNSUPPORTED) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, p);
    }
    return p;
}

// Fused whole-plane kernel: the plane (+ halo) must move as one bulk tensor copy and its whole
// pyramid, D and one input tile must fit in shared memory.
struct PPlan {
    int status = WTCONV_OK;
    PlaneArgs a{};
    size_t smem = 0;
    int occ = 0;  // resident CTAs per SM
};

PPlan plan_plane_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    PPlan p;
    PlaneArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    const int eb = elem_bytes(dtype);
    const int e16 = 16 / eb;
    if (((size_t)W * eb) % 16 != 0) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    const int TW = round_up(W, e16 > 4 ? e16 : 4), TH = round_up(H, kRows);
    const int dchunk_e = ((W / 2) % 4 == 0 && (TW / 2) % 4 == 0) ? 4 : 2;
    a.sg = make_shallow_geo(H, W, k, TH, TW, 1, eb, e16, dchunk_e);
    const ShallowGeo &sg = a.sg;
    if (((size_t)sg.xw * eb) % 16 != 0 || ((size_t)sg.padx * eb) % 16 != 0 || sg.xw > 256 || sg.xrows > 256) {
        p.status = WTCONV_ERR_UNSUPPORTED;
        return p;
    }
    a.st_mode = (W % 4) == 0 ? 1 : 0;
    a.dpitch = round_up(TW / 2, 2);
    if (L >= 2) {
        a.dg = make_geo(H, W, L, k, 2);
        int tot = 0;
        for (int ci = 3; ci < 1 + 2 * L; ++ci) {
            const int l = (ci - 1) / 2 + 1;
            a.deep_item_start[ci] = tot;
            tot += ceil_div(a.dg.h[l], kPlaneDeepRows) * round_up(a.dg.cstr[l], 8);  // 8-slot item rows
        }
        a.deep_item_start[1 + 2 * L] = tot;
        a.n_deep_items = tot;
    }
    p.smem = plane_smem_bytes(a, eb);
    if (p.smem + kStaticSmemMargin > (size_t)kMaxSmem) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    const int sms = device_sms();
    const int occ = occupancy_plane(dtype, k, p.smem);
    if (sms <= 0 || occ <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    p.occ = occ;
    const long long slots = (long long)sms * occ;
    long long best_nb = 1, best_cost = -1;
    for (long long nb = 1; nb <= B; ++nb) {
        const long long cost = ((C * nb + slots - 1) / slots) * ((B + nb - 1) / nb);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_nb = nb; }
    }
    a.planes_per_cta = (int)((B + best_nb - 1) / best_nb);
    a.nb = (B + a.planes_per_cta - 1) / a.planes_per_cta;
    return p;
}

PPlan plan_plane(int B, int C, int H, int W, int L, int k, int dtype) {
    static std::mutex mu;
    static std::map<PlanKey, PPlan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        PPlan p;
        p.status = WTCONV_ERR_CUDA;
        return p;
    }
    const PlanKey key(7, B, C, H, W, L, k, dtype, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    PPlan p = plan_plane_uncached(B, C, H, W, L, k, dtype);
    const char *verbose = getenv("WTCONV_VERBOSE");
    if (verbose && verbose[0] == '1')
        fprintf(stderr, "wtconv plan fused B=%d C=%d H=%d W=%d L=%d k=%d dtype=%d: status %d nb=%d planes/cta=%d smem=%zu\n",
                B, C, H, W, L, k, dtype, p.status, p.a.nb, p.a.planes_per_cta, p.smem);
    if (p.status == WTCONV_OK || p.status == WTCONV_ERR_UNSUPPORTED) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, p);
    }
    return p;
}

// Fused whole-plane weight gradient: x (+ halo) and dy each move as one bulk tensor copy, both
// pyramids fit in shared memory.  Threads: whole warps for the base path's items, then one run
// of threads per level pair image; the split minimises the items per thread per plane.
struct FPlan {
    int status = WTCONV_OK;
    DwPlaneArgs a{};
    size_t smem = 0;
    int occ = 0;
    size_t partial_bytes = 0;
};

FPlan plan_dw_fused_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    FPlan p;
    DwPlaneArgs &a = p.a;
    a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
    const int eb = elem_bytes(dtype);
    const int e16 = 16 / eb;
    if (((size_t)W * eb) % 16 != 0) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    const int TW = round_up(W, e16 > 4 ? e16 : 4), TH = round_up(H, kRows);
    a.sg = make_shallow_geo(H, W, k, TH, TW, 1, eb, e16, 4);
    const ShallowGeo &sg = a.sg;
    if (((size_t)sg.xw * eb) % 16 != 0 || ((size_t)sg.padx * eb) % 16 != 0 || ((size_t)TW * eb) % 16 != 0 ||
        sg.xw > 256 || sg.xrows > 256 || TW > 256 || TH > 256) {
        p.status = WTCONV_ERR_UNSUPPORTED;
        return p;
    }
    a.th1 = round_up(TH / 2, kRows);
    a.y1rows = a.th1 + 2 * (k / 2);
    a.dg = make_geo(H, W, L, k, 3);
    // thread split: CTA size, base warps and items per thread minimising the item rounds per plane
    // (ties: fewer threads).  Items are counted by slot, item rows padded to multiples of 8 slots,
    // and every image's threads start at a multiple of 8 (the kernel's quarter-warp layout).
    const int nbase = sg.items_r * round_up(sg.items_c, 8);
    auto level_slots = [&](int l) { return a.dg.rseg[l] * round_up(a.dg.cstr[l], 8); };
    int best_nt = 0, best_wb = -1, best_pb = 0, best_pl = 0, best_span = 0;
    for (int nt = 256; nt <= kDwPlaneMaxThreads; nt += 32) {
        for (int wb = 1; 32 * wb < nt; ++wb) {
            const int pb = ceil_div(nbase, 32 * wb), avail = nt - 32 * wb;
            int max_slots = 1;
            for (int l = 1; l <= L; ++l) max_slots = std::max(max_slots, level_slots(l));
            int pl = 0;  // fewest items per level thread whose threads fit (0: none do)
            for (int t = 1; t <= max_slots && pl == 0; ++t) {
                int need = 0;
                for (int l = 1; l <= L; ++l) need += 2 * round_up(ceil_div(level_slots(l), t), 8);
                if (need <= avail) pl = t;
            }
            if (pl == 0) continue;
            const int span = std::max(pb, pl);
            if (best_wb < 0 || span < best_span) {
                best_nt = nt; best_wb = wb; best_pb = pb; best_pl = pl; best_span = span;
            }
        }
    }
    if (best_wb < 0) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    a.nthreads = best_nt;
    a.per_thread_base = best_pb;
    a.per_thread = best_pl;
    a.tstart[0] = 0;
    a.tstart[1] = 32 * best_wb;
    for (int ci = 1; ci < 1 + 2 * L; ++ci) {
        const int l = (ci - 1) / 2 + 1;
        a.tstart[ci + 1] = a.tstart[ci] + round_up(ceil_div(level_slots(l), best_pl), 8);
    }
    // two copy buffers where that keeps as many CTAs resident per SM as one
    a.nbuf = 1;
    p.smem = dw_plane_smem_bytes(a, eb);
    if (p.smem + kStaticSmemMargin > (size_t)kMaxSmem) { p.status = WTCONV_ERR_UNSUPPORTED; return p; }
    const int sms = device_sms();
    int occ = occupancy_dw_plane(dtype, k, p.smem, a.nthreads);
    if (sms <= 0 || occ <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    {
        DwPlaneArgs a2 = a;
        a2.nbuf = 2;
        const size_t smem2 = dw_plane_smem_bytes(a2, eb);
        if (smem2 + kStaticSmemMargin <= (size_t)kMaxSmem && occupancy_dw_plane(dtype, k, smem2, a.nthreads) >= occ) {
            a.nbuf = 2;
            p.smem = smem2;
        }
    }
    p.occ = occ;
    const long long slots = (long long)sms * occ;
    long long best_nb = 1, best_cost = -1;
    for (long long nb = 1; nb <= B; ++nb) {
        const long long cost = ((C * nb + slots - 1) / slots) * ((B + nb - 1) / nb);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_nb = nb; }
    }
    a.planes_per_cta = (int)((B + best_nb - 1) / best_nb);
    a.nb = (B + a.planes_per_cta - 1) / a.planes_per_cta;
    p.partial_bytes = ((size_t)a.nb * C * (1 + 4 * L) * (k * k + 1) * sizeof(float) + 255) / 256 * 256;
    return p;
}

FPlan plan_dw_fused(int B, int C, int H, int W, int L, int k, int dtype) {
    static std::mutex mu;
    static std::map<PlanKey, FPlan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        FPlan p;
        p.status = WTCONV_ERR_CUDA;
        return p;
    }
    const PlanKey key(8, B, C, H, W, L, k, dtype, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    FPlan p = plan_dw_fused_uncached(B, C, H, W, L, k, dtype);
    const char *verbose = getenv("WTCONV_VERBOSE");
    if (verbose && verbose[0] == '1')
        fprintf(stderr,
                "wtconv plan dw fused B=%d C=%d H=%d W=%d L=%d k=%d dtype=%d: status %d nb=%d planes/cta=%d "
                "smem=%zu occ=%d buffers %d items/thread base %d levels %d, threads %d of %d\n",
                B, C, H, W, L, k, dtype, p.status, p.a.nb, p.a.planes_per_cta, p.smem, p.occ, p.a.nbuf,
                p.a.per_thread_base, p.a.per_thread, p.a.tstart[1 + 2 * L], p.a.nthreads);
    if (p.status == WTCONV_OK || p.status == WTCONV_ERR_UNSUPPORTED) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, p);
    }
    return p;
}

// ------------------------------------------------------------------ batch-pair kernels
// Item shapes the pair kernels can take (base columns x rows, level columns x rows) and their
// relative per-FMA speed measured on GB300 (isolated strip items: two-column strips have no
// shared-memory bank conflicts; four-row strips re-read a larger share of halo rows).
struct PairShape { int q0, s0, ql, sl, qd, sd; double eff; };
const PairShape kPairShapes[] = {
    {4, 8, 4, 8, 4, 8, 1.00}, {4, 8, 2, 8, 2, 8, 1.05}, {2, 8, 2, 8, 2, 8, 1.10}, {2, 8, 2, 8, 2, 4, 1.08},
    {4, 4, 4, 4, 4, 4, 0.76}, {2, 4, 2, 4, 2, 4, 0.70},
};

// Relative speed of a shape-specialised forward instantiation over the generic one (GB300).
constexpr double kSpecGain = 1.4;

struct PairPlan {
    int status = WTCONV_ERR_UNSUPPORTED;
    PairArgs a{};
    size_t smem = 0;
    int occ = 0;
    double score = 0.0;
    size_t workspace = 0;  // weight gradient: partials
};

// Planner restrictions for tuning runs: WTCONV_PAIR_THREADS (64, 128 or 256) keeps one CTA
// size, WTCONV_PAIR_SHAPE (an index into kPairShapes) one item shape.
bool pair_threads_allowed(int T) {
    const char *v = getenv("WTCONV_PAIR_THREADS");
    return !(v && v[0]) || atoi(v) == T;
}
bool pair_shape_allowed(int i) {
    const char *v = getenv("WTCONV_PAIR_SHAPE");
    return !(v && v[0]) || atoi(v) == i;
}

void pair_counts(PairArgs &a) {
    const PairGeo &g = a.geo;
    const int L = a.L;
    a.n_a = L >= 2 ? (a.H / 4) * (a.W / 4) : (a.H / 2) * (a.W / 2);
    a.dv_na = make_fastdiv((uint32_t)a.n_a);
    a.dv_naw = make_fastdiv((uint32_t)(L >= 2 ? a.W / 4 : a.W / 2));
    int tot = 0;
    for (int l = 1; l <= L; ++l) {
        a.conv_start[l] = tot;
        tot += 4 * g.ns[l] * g.ng[l];
    }
    a.conv_start[L + 1] = tot;
    a.n_conv = tot;
    a.dv_nconv = make_fastdiv((uint32_t)tot);
    for (int l = 0; l <= L; ++l) {
        a.dv_lvl[l] = make_fastdiv((uint32_t)(g.ns[l] * g.ng[l]));
        a.dv_lvl_ns[l] = make_fastdiv((uint32_t)g.ns[l]);
    }
    a.n_gather = L >= 2 ? g.h[2] * g.w[2] : 0;
    a.dv_ngather = make_fastdiv((uint32_t)(a.n_gather > 0 ? a.n_gather : 1));
    a.dv_gw = make_fastdiv((uint32_t)(L >= 2 ? g.w[2] : 1));
    a.n_out = g.ns[0] * g.ng[0];
    a.dv_nout = make_fastdiv((uint32_t)a.n_out);
    a.dv_out_ns = make_fastdiv((uint32_t)g.ns[0]);
    a.dv_xn = make_fastdiv((uint32_t)(a.H * (a.W / 2)));
    a.dv_xw = make_fastdiv((uint32_t)(a.W / 2));
}

// Persistent grid: one CTA per resident slot (at most one per unit), contiguous unit ranges.
void pair_grid(PairArgs &a, int sms, int occ, int chunk_groups) {
    a.chunk_groups = chunk_groups;
    a.nchunks = (a.ngroups + chunk_groups - 1) / chunk_groups;
    a.nb = a.nchunks;
    a.units = a.C * a.nchunks;
    a.grid = std::min(a.units, sms * occ);
}

// Thread-slot utilisation of a phase of n items (cost c each, thread-time c / eff) on T threads.
void add_phase(double &work, double &tim, long long n, double c, double eff, int T) {
    if (n <= 0) return;
    work += n * c;
    tim += (double)((n + T - 1) / T) * T * c / eff;
}

// A group's planes as one tensor copy per activation: each H x W plane viewed as R rows of Wr
// elements (Wr dividing H W, rows of a multiple of 16 bytes, Wr and R at most 256, the box limit).
// WTCONV_PAIR_TMAP=0 keeps one bulk copy per plane.
void pair_tma_map_geometry(PairArgs &a, int eb) {
    a.tma_map = 0;
    const char *kn = getenv("WTCONV_PAIR_TMAP");
    if (!a.tma || (kn && kn[0] == '0') || 2 * a.G > 256) return;
    const int HW = a.H * a.W;
    for (int wr = std::min(256, HW); wr >= 1; --wr) {
        if (HW % wr != 0 || ((size_t)wr * eb) % 16 != 0) continue;
        if (HW / wr > 256) break;
        a.tma_map = 1;
        a.tma_rlen = wr;
        a.tma_rows = HW / wr;
        return;
    }
}

// Forward / input gradient on batch pairs: every pair's pyramid and outputs in shared memory.
PairPlan plan_pair_fwd_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    PairPlan best;
    const int eb = elem_bytes(dtype);
    const int sms = device_sms();
    if (sms <= 0) { best.status = WTCONV_ERR_CUDA; return best; }
    const int npairs = (B + 1) / 2;
    const int KK = k * k;
    // a shape with a specialised instantiation takes the CTA size and slots that measured fastest
    PairSpecPref pref{};
    const char *knob_t = getenv("WTCONV_PAIR_THREADS"), *knob_s = getenv("WTCONV_PAIR_SHAPE");
    const char *knob_gs = getenv("WTCONV_PAIR_SLOTS");  // tuning: pair slots per group
    const int knob_g = knob_gs && knob_gs[0] ? atoi(knob_gs) : 0;
    const bool tuned = pair_spec_measured(H, W, L, k, dtype, &pref) && !(knob_t && knob_t[0]) && !(knob_s && knob_s[0]);
    // candidate item shapes: the instantiation's own (which may lie outside the run-time menu)
    // for a tuned shape, else the menu
    std::vector<PairShape> shapes;
    if (tuned) {
        shapes.push_back({pref.shape[0], pref.shape[1], pref.shape[2], pref.shape[3], pref.shape[4], pref.shape[5], 1.0});
    } else {
        for (int si = 0; si < (int)(sizeof(kPairShapes) / sizeof(kPairShapes[0])); ++si)
            if (pair_shape_allowed(si)) shapes.push_back(kPairShapes[si]);
    }
    for (const PairShape &sh : shapes) {
        for (int T : {64, 128, 256}) {
            if (!pair_threads_allowed(T)) continue;
            if (tuned && pref.threads && T != pref.threads) continue;
            for (int G = 1; G <= std::min(npairs, kPairMaxSlots); ++G) {
                if (tuned && pref.slots && G != std::min(pref.slots, npairs)) continue;
                if (knob_g > 0 && G != std::min(knob_g, npairs)) continue;
                PairArgs a{};
                a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
                a.npairs = npairs;
                a.G = G;
                a.ngroups = (npairs + G - 1) / G;
                a.nthreads = T;
                a.geo = make_pair_geo(H, W, L, k, 0, sh.q0, sh.s0, sh.ql, sh.sl, sh.qd, sh.sd);
                a.tma = ((size_t)H * W * eb) % 16 == 0;
                a.raw_pair_bytes = (int)(((size_t)2 * H * W * eb + 15) / 16 * 16);
                a.vec_st = (W % 4) == 0;
                const int shp[6] = {sh.q0, sh.s0, sh.ql, sh.sl, sh.qd, sh.sd};
                a.spec = pair_spec_index(H, W, L, k, dtype, shp);
                if (a.spec < 0 && tuned) break;  // only the instantiation runs its own shapes
                pair_counts(a);
                const size_t smem = pair_fwd_smem_bytes(a, eb);
                if (smem + kStaticSmemMargin > (size_t)kMaxSmem) break;
                const int occ = a.spec >= 0 ? occupancy_pair_fwd_spec(a.spec, smem, T)
                                            : occupancy_pair_fwd(dtype, k, smem, T);
                if (occ <= 0) break;
                const PairGeo &g = a.geo;
                double work = 0.0, tim = 0.0;
                add_phase(work, tim, (long long)G * a.n_out, (double)g.Q[0] * g.S[0] * KK, sh.eff, T);
                double cmax = 0.0;
                for (int l = 1; l <= L; ++l) cmax = std::max(cmax, (double)g.Q[l] * g.S[l] * KK);
                double wconv = 0.0;
                for (int l = 1; l <= L; ++l) wconv += 4.0 * G * g.ns[l] * g.ng[l] * g.Q[l] * g.S[l] * KK;
                const long long nconv = (long long)G * a.n_conv;
                work += wconv;
                tim += (double)((nconv + T - 1) / T) * T * cmax / sh.eff;
                // resident warps (beyond 16 per SM more warps no longer help); a single resident
                // CTA also loses its phases' barrier waits, which other CTAs would fill
                const double warps = std::min((double)occ * T / 32.0, 16.0) * (occ >= 2 ? 1.0 : 0.8);
                // a shape-specialised instantiation issues far fewer index instructions
                const double score = work / tim * warps * (a.spec >= 0 ? kSpecGain : 1.0);
                if (score > best.score * 1.02) {
                    best.status = WTCONV_OK;
                    best.a = a;
                    best.smem = smem;
                    best.occ = occ;
                    best.score = score;
                }
            }
        }
    }
    if (best.status == WTCONV_OK) {
        const char *ks = getenv("WTCONV_PAIR_SPLIT");  // tuning: 0 keeps every warp on every level
        best.a.split = (L >= 3 && best.a.nthreads >= 128 && !(ks && ks[0] == '0')) ? 1 : 0;
        pair_tma_map_geometry(best.a, eb);
        pair_grid(best.a, sms, best.occ, 1);
    }
    return best;
}

// Weight gradient on batch pairs: both pyramids in shared memory; threads pinned to signals.
PairPlan plan_pair_dw_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    PairPlan best;
    const int eb = elem_bytes(dtype);
    const int sms = device_sms();
    if (sms <= 0) { best.status = WTCONV_ERR_CUDA; return best; }
    const int npairs = (B + 1) / 2;
    const int KK = k * k, nsig = 1 + 4 * L;
    const char *knob_gs = getenv("WTCONV_PAIR_SLOTS");  // tuning: pair slots per group
    const int knob_g = knob_gs && knob_gs[0] ? atoi(knob_gs) : 0;
    // the menu, plus 7-row items (exact on planes of 7 * 2^l rows; correlation items only); a
    // shape with a measured preference keeps to it unless a tuning restriction is set
    constexpr int kMenu = (int)(sizeof(kPairShapes) / sizeof(kPairShapes[0]));
    PairSpecPref pref{};
    const char *knob_t = getenv("WTCONV_PAIR_THREADS"), *knob_s = getenv("WTCONV_PAIR_SHAPE");
    const bool tuned = pair_spec_measured(H, W, L, k, dtype, &pref) && !(knob_t && knob_t[0]) && !(knob_s && knob_s[0]);
    for (int si = 0; si <= kMenu; ++si) {
        const PairShape sh = si < kMenu ? kPairShapes[si] : PairShape{2, 7, 2, 7, 2, 7, 1.10};
        if (!pair_shape_allowed(si)) continue;
        if (si == kMenu && H % 7 != 0 && !(knob_s && knob_s[0])) continue;  // 7-row items: planes of 7 * 2^l rows
        if (tuned && pref.dw_shape >= 0 && si != pref.dw_shape) continue;
        for (int T : {64, 128, 256}) {
            if (!pair_threads_allowed(T)) continue;
            if (tuned && pref.dw_threads && T != pref.dw_threads) continue;
            for (int G = 1; G <= std::min(npairs, kPairMaxSlots); ++G) {
                if (knob_g > 0 && G != std::min(knob_g, npairs)) continue;
                PairArgs a{};
                a.B = B; a.C = C; a.H = H; a.W = W; a.L = L; a.K = k;
                a.npairs = npairs;
                a.G = G;
                a.ngroups = (npairs + G - 1) / G;
                a.nthreads = T;
                a.geo = make_pair_geo(H, W, L, k, 1, sh.q0, sh.s0, sh.ql, sh.sl, sh.qd, sh.sd);
                a.spec = -1;
                a.tma = ((size_t)H * W * eb) % 16 == 0;
                a.raw_pair_bytes = (int)(((size_t)4 * H * W * eb + 15) / 16 * 16);
                pair_counts(a);
                const size_t smem = pair_dw_smem_bytes(a, eb);
                if (smem + kStaticSmemMargin > (size_t)kMaxSmem) break;
                const int occ = occupancy_pair_dw(dtype, k, smem, T);
                if (occ <= 0) break;
                // items per signal per group, and the smallest per-thread count that fits T threads
                const PairGeo &g = a.geo;
                long long n[1 + 4 * kMaxLevels];
                double cost[1 + 4 * kMaxLevels];
                for (int s = 0; s < nsig; ++s) {
                    const int l = s == 0 ? 0 : (s - 1) / 4 + 1;
                    n[s] = (long long)G * g.ns[l] * g.ng[l];
                    cost[s] = (double)g.Q[l] * g.S[l] * KK;
                }
                int d = 1;
                for (;; ++d) {
                    long long need = 0;
                    for (int s = 0; s < nsig; ++s) need += (n[s] + d - 1) / d;
                    if (need <= T) break;
                }
                // a warp takes as long as its slowest thread; a warp mixing item shapes runs each
                // shape's code in turn
                double work = 0.0, tmax = 0.0;
                {
                    constexpr int kW = kPairMaxThreads / 32;
                    double tshape[kW][3] = {};  // slowest thread per item shape (S x Q: 3 kinds at most)
                    int t0 = 0;
                    for (int s = 0; s < nsig; ++s) {
                        work += n[s] * cost[s];
                        const int l = s == 0 ? 0 : (s - 1) / 4 + 1;
                        const int kind = l == 0 ? 0 : (l == 1 ? 1 : 2);
                        const int nth = (int)((n[s] + d - 1) / d);
                        const double tt = std::min<double>(d, (double)n[s]) * cost[s];
                        for (int t = t0; t < t0 + nth; ++t) tshape[t / 32][kind] = std::max(tshape[t / 32][kind], tt);
                        t0 += nth;
                    }
                    for (int wi = 0; wi < T / 32; ++wi) {
                        // kinds with the same item shape share their code
                        double tw = tshape[wi][0];
                        tw = (g.Q[1] == g.Q[0] && g.S[1] == g.S[0]) ? std::max(tw, tshape[wi][1]) : tw + tshape[wi][1];
                        if (L >= 2) {
                            const bool same1 = g.Q[2] == g.Q[1] && g.S[2] == g.S[1];
                            tw = same1 ? std::max(tw, tshape[wi][2]) : tw + tshape[wi][2];
                        }
                        tmax = std::max(tmax, tw);
                    }
                }
                const double warps = std::min((double)occ * T / 32.0, 16.0) * (occ >= 2 ? 1.0 : 0.8);
                const double score = work / ((double)T * tmax / sh.eff) * warps;
                if (score > best.score * 1.02) {
                    int t0 = 0;
                    for (int s = 0; s < nsig; ++s) {
                        a.sig_start[s] = t0;
                        t0 += (int)((n[s] + d - 1) / d);
                    }
                    a.sig_start[nsig] = t0;
                    a.per_thread = d;
                    best.status = WTCONV_OK;
                    best.a = a;
                    best.smem = smem;
                    best.occ = occ;
                    best.score = score;
                }
            }
        }
    }
    if (best.status == WTCONV_OK) {
        // units of several groups (one partial each): enough items per thread in a unit that its
        // flush (tap sums to shared memory, the reduction, the partial's store) stays small
        // against its correlations, which matters on small planes (8 x 8: 77 -> 71 us at 8 groups
        // per unit instead of 2), and enough units to keep every resident CTA busy
        PairArgs &a = best.a;
        const long long slots = (long long)sms * best.occ;
        long long items_pair = 0;
        for (int l = 0; l <= L; ++l) items_pair += (l == 0 ? 1 : 4) * (long long)a.geo.ns[l] * a.geo.ng[l];
        const double per_thread_group = (double)a.G * items_pair / a.nthreads;
        int cg = 1;
        while (cg < a.ngroups && cg * per_thread_group < 8.0 &&
               (long long)C * ((a.ngroups + 2 * cg - 1) / (2 * cg)) >= slots)
            cg *= 2;
        const char *kc = getenv("WTCONV_PAIR_CHUNK");  // tuning: groups per work unit
        if (kc && kc[0] && atoi(kc) > 0) cg = std::min(atoi(kc), a.ngroups);
        pair_grid(a, sms, best.occ, cg);
        pair_tma_map_geometry(a, eb);
        best.workspace = ((size_t)a.nchunks * C * nsig * (KK + 1) * sizeof(float) + 255) / 256 * 256;
    }
    return best;
}

PairPlan cached_pair_plan(int kind, int B, int C, int H, int W, int L, int k, int dtype) {
    static std::mutex mu;
    static std::map<std::pair<PlanKey, std::string>, PairPlan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        PairPlan p;
        p.status = WTCONV_ERR_CUDA;
        return p;
    }
    // the tuning restrictions are part of the key: a restricted plan is a different plan
    std::string knobs;
    for (const char *kn : {"WTCONV_PAIR_THREADS", "WTCONV_PAIR_SHAPE", "WTCONV_PAIR_SLOTS", "WTCONV_PAIR_CHUNK",
                           "WTCONV_PAIR_SPLIT", "WTCONV_PAIR_TMAP"}) {
        const char *v = getenv(kn);
        knobs += v ? v : "";
        knobs += ';';
    }
    const auto key = std::make_pair(PlanKey(kind, B, C, H, W, L, k, dtype, dev), knobs);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    PairPlan p = kind == 10 ? plan_pair_fwd_uncached(B, C, H, W, L, k, dtype)
                            : plan_pair_dw_uncached(B, C, H, W, L, k, dtype);
    const char *verbose = getenv("WTCONV_VERBOSE");
    if (verbose && verbose[0] == '1')
        fprintf(stderr, "wtconv plan pair-%s B=%d C=%d H=%d W=%d L=%d k=%d dtype=%d: status %d G=%d items %dx%d/%dx%d "
                        "qd=%d sd=%d spec=%d threads=%d grid=%d units=%d chunk=%d smem=%zu occ=%d tma=%d d=%d score=%.2f\n",
                kind == 10 ? "fwd" : "dw", B, C, H, W, L, k, dtype, p.status, p.a.G, p.a.geo.Q[0], p.a.geo.S[0],
                p.a.geo.Q[1], p.a.geo.S[1], L >= 2 ? p.a.geo.Q[2] : 0, L >= 2 ? p.a.geo.S[2] : 0, p.a.spec,
                p.a.nthreads, p.a.grid, p.a.units, p.a.chunk_groups, p.smem, p.occ,
                p.a.tma, p.a.per_thread, p.score);
    if (p.status == WTCONV_OK || p.status == WTCONV_ERR_UNSUPPORTED) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, p);
    }
    return p;
}

PairPlan plan_pair_fwd(int B, int C, int H, int W, int L, int k, int dtype) {
    return cached_pair_plan(10, B, C, H, W, L, k, dtype);
}
PairPlan plan_pair_dw(int B, int C, int H, int W, int L, int k, int dtype) {
    return cached_pair_plan(11, B, C, H, W, L, k, dtype);
}

// Whether the batch-pair kernels run by default.  For the shapes with a specialised instantiation
// the choice measured on GB300 decides (wtconv_pair_specs.h); elsewhere the generic batch-pair
// forward wins only on the smallest planes (8 x 8: 56 vs 79 us, where the whole-plane kernels'
// per-plane setup does not amortise), the weight gradient up to 28 x 28 planes.  WTCONV_PAIR=0
// turns them off, =1 makes them the default wherever they apply.
bool pair_default(bool weight_gradient, int H, int W, int L, int k, int dtype) {
    const char *v = getenv("WTCONV_PAIR");
    if (v && strcmp(v, "0") == 0) return false;
    if (v && strcmp(v, "1") == 0) return true;
    PairSpecPref pref{};
    if (pair_spec_measured(H, W, L, k, dtype, &pref)) return weight_gradient ? pref.dw_default : pref.fwd_default;
    return (long long)H * W <= (weight_gradient ? 784 : 64);
}

// ------------------------------------------------------- tiled batch-pair weight gradient plan
//
// Launch 0 correlates the base path and levels 1 .. min(L, 2) on tiles of x and dy; while levels
// remain, it writes the level-2 LL bands of x and dy as fp32 planes and launch i + 1 takes the
// next (up to) two levels from them (lvl_off = 2 (i + 1)).  All launches write the same rows of
// partials [nchunks][C][1 + 4L][K*K+1], each its own signals.
struct PtPlan {
    int status = WTCONV_ERR_UNSUPPORTED;
    int nlaunch = 0;
    PtileArgs a[3];
    size_t smem[3] = {0, 0, 0};
    int occ[3] = {0, 0, 0};
    size_t ll_off[3] = {0, 0, 0};     // workspace offset of launch i's LL planes (x, then dy at + ll_half)
    size_t ll_half[3] = {0, 0, 0};
    size_t partial_bytes = 0;
    size_t workspace = 0;
};

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Geometry of one launch on B x C planes of H x W elements (row pitch in_pitch, element size eb)
// with tiles of TH x TW and G pairs per group; false where the bulk tensor copies cannot apply.
bool pt_make(PtileArgs &a, int B, int C, int H, int W, int in_pitch, int eb, int K, int LT, int base, int lvl_off,
             int L_total, int TH, int TW, int G, int nt, bool small) {
    a = PtileArgs{};
    const int P = K / 2, BS = 1 << LT;
    a.B = B; a.C = C; a.H = H; a.W = W; a.K = K; a.LT = LT; a.base = base; a.lvl_off = lvl_off;
    a.L_total = L_total;
    a.TH = TH; a.TW = TW; a.G = G; a.nthreads = nt;
    // a tile that covers the whole plane needs no halo: outside the plane every level is zero,
    // which the zeroed slots already hold
    const bool whole = TH >= H && TW >= W;
    a.HX = whole ? 0 : BS * P;
    const int al = 16 / eb;
    a.HXL = (a.HX + al - 1) / al * al;
    a.RXR = TH + 2 * a.HX;
    a.RXW = TW + 2 * a.HXL;
    a.in_pitch = in_pitch;
    if (TH % BS != 0 || TW % BS != 0 || TH <= 0 || TW <= 0) return false;
    if (((size_t)TW * eb) % 16 != 0 || ((size_t)in_pitch * eb) % 16 != 0) return false;
    if (a.RXW > 256 || a.RXR > 256 || 2 * G > 256 || TW > 256 || TH > 256) return false;
    a.tiles_r = (H + TH - 1) / TH;
    a.tiles_c = (W + TW - 1) / TW;
    a.tiles = a.tiles_r * a.tiles_c;
    int off = 0;
    for (int l = 0; l <= LT; ++l) {
        PtLevel &v = a.lv[l];
        v.h = TH >> l;
        v.w = TW >> l;
        v.Q = small ? 2 : 4;  // one item width per launch (levels narrower than Q round up)
        v.S = v.h >= 8 ? 8 : 4;
        v.ns = (v.w + v.Q - 1) / v.Q;
        v.ng = (v.h + v.S - 1) / v.S;
        v.ipitch = pg_round2(v.Q * v.ns + K - 1);
        v.irows = v.ng * v.S + K - 1;
        v.iimg = v.ipitch * v.irows;
        v.zpitch = pg_round2(v.Q * v.ns);
        v.zrows = v.ng * v.S;
        v.zimg = v.zpitch * v.zrows;
        v.items = v.ns * v.ng;
    }
    if (base) {
        a.lv[0].off_y = off; off += a.lv[0].iimg;
        a.lv[0].off_z = off; off += a.lv[0].zimg;
    }
    for (int l = 1; l <= LT; ++l) { a.lv[l].off_y = off; off += 4 * a.lv[l].iimg; }
    for (int l = 1; l <= LT; ++l) { a.lv[l].off_z = off; off += 4 * a.lv[l].zimg; }
    a.slot = pg_round2(off);
    a.n0 = base ? a.lv[0].items : 0;
    a.n1 = a.lv[1].items;
    a.n2 = LT >= 2 ? a.lv[2].items : 0;
    a.per_pair = a.n0 + 4 * a.n1 + 4 * a.n2;
    a.raw_x_bytes = (int)(((size_t)2 * G * a.RXR * a.RXW * eb + 127) / 128 * 128);
    a.raw_dy_bytes = (int)(((size_t)2 * G * TH * TW * eb + 127) / 128 * 128);
    a.npairs = (B + 1) / 2;
    a.ngroups = (a.npairs + G - 1) / G;
    a.work = a.tiles * a.ngroups;
    a.ll_out = L_total - lvl_off > LT ? 1 : 0;
    if (a.ll_out && LT != 2) return false;
    a.ll_h = H / 4;
    a.ll_w = W / 4;
    a.ll_pitch = (a.ll_w + 3) / 4 * 4;
    a.dv_pp = make_fastdiv(a.per_pair);
    a.dv_n1 = make_fastdiv(std::max(1, a.n1));
    a.dv_n2 = make_fastdiv(std::max(1, a.n2));
    for (int l = 0; l <= kPtMaxLevels; ++l) a.dv_ns[l] = make_fastdiv(l <= LT ? a.lv[l].ns : 1);
    a.dv_tiles = make_fastdiv(a.tiles);
    a.dv_tiles_c = make_fastdiv(a.tiles_c);
    const int xbw = (TW + 2 * a.HX) / BS, xbh = (TH + 2 * a.HX) / BS;
    a.dv_xbw = make_fastdiv(xbw);
    a.dv_xb = make_fastdiv(xbw * xbh);
    a.dv_dbw = make_fastdiv(TW / BS);
    a.dv_db = make_fastdiv((TW / BS) * (TH / BS));
    return true;
}

// Tuning restrictions (0: planner's choice): WTCONV_PTILE=TH,TW,G,threads[,small items 0/1].
void pt_knobs(int &th, int &tw, int &g, int &nt, int &sm) {
    th = tw = g = nt = 0;
    sm = -1;
    const char *v = getenv("WTCONV_PTILE");
    if (v && v[0]) sscanf(v, "%d,%d,%d,%d,%d", &th, &tw, &g, &nt, &sm);
}

// Best geometry of one launch: for each tile and CTA size, the largest G that keeps two CTAs per
// SM resident, scored by how evenly a group's items fill the CTA's threads and by resident warps.
bool pt_choose(PtileArgs &best, size_t &best_smem, int &best_occ, int B, int C, int H, int W, int in_pitch, int eb,
               int dtype, int K, int LT, int base, int lvl_off, int L_total) {
    int kth = 0, ktw = 0, kg = 0, knt = 0, ksm = -1;
    if (base) pt_knobs(kth, ktw, kg, knt, ksm);  // the restrictions apply to the first launch
    const int BS = 1 << LT, al = 16 / eb;
    const int Hr = (H + BS - 1) / BS * BS;
    const int Wr = (W + std::max(BS, al) - 1) / std::max(BS, al) * std::max(BS, al);
    const int sms = device_sms();
    if (sms <= 0) return false;
    double best_score = -1.0;
    for (int th0 : {16, 32, 64}) {
        const int TH = std::min(th0, Hr);
        if (kth && TH != kth) continue;
        for (int tw0 : {32, 64}) {
            const int TW = std::min(tw0, Wr);
            if (ktw && TW != ktw) continue;
            if (th0 > 16 && TH < th0 && TH == std::min(th0 / 2, Hr)) continue;  // same tile as a smaller th0
            if (tw0 > 32 && TW < tw0 && TW == std::min(tw0 / 2, Wr)) continue;
            for (int nt : {128, 256})
            for (int small = 0; small < 2; ++small) {
                if (knt && nt != knt) continue;
                if (ksm >= 0 && small != ksm) continue;
                for (int G = 1; G <= 16; ++G) {
                    if (kg && G != kg) continue;
                    PtileArgs a;
                    if (!pt_make(a, B, C, H, W, in_pitch, eb, K, LT, base, lvl_off, L_total, TH, TW, G, nt, small))
                        break;
                    if (G > a.npairs) break;
                    const size_t smem = ptile_smem_bytes(a, eb);
                    if (smem + kStaticSmemMargin > (size_t)kMaxSmem) break;
                    const int occ = occupancy_ptile_dw(base ? dtype : WTCONV_F32, K, LT, base, smem, nt, a.lv[0].Q);
                    if (occ <= 0) break;
                    // Measured on GB300 (256 x 256 bf16 planes, L = 5): resident threads decide
                    // first (the kernel is latency-bound: 4 x 128 threads ran 1.26x faster than
                    // 3 x 128), CTAs of 128 beat 256 at equal residency (one barrier spans fewer
                    // warps), then how evenly a group's items fill the threads (a group takes as
                    // long as its busiest thread) and the share of the x tile that is halo.
                    const long long items = (long long)a.per_pair * G;
                    const double fill = (double)items / ((double)((items + nt - 1) / nt) * nt);
                    const double resident = std::min(512.0, (double)occ * nt) / 512.0;
                    const double cta = nt == 128 ? 1.0 : 0.7;
                    const double load = small ? 0.9 : 1.0;  // narrower items: more loads per FMA
                    const double halo = (double)(TH * TW) / ((double)a.RXR * (TW + 2 * a.HX));
                    const double tiles_used = (double)H * W / ((double)a.tiles * TH * TW);
                    const double score =
                        resident * cta * std::sqrt(fill) * load * std::sqrt(std::sqrt(halo)) * tiles_used;
                    const char *vb = getenv("WTCONV_VERBOSE");
                    if (vb && vb[0] == '2')
                        fprintf(stderr, "  ptile candidate %dx%d q=%d G=%d nt=%d smem=%zu occ=%d fill=%.3f halo=%.3f score=%.4f\n",
                                TH, TW, a.lv[0].Q, G, nt, smem, occ, fill, halo, score);
                    if (score > best_score) {
                        best_score = score;
                        best = a;
                        best_smem = smem;
                        best_occ = occ;
                    }
                }
            }
        }
    }
    return best_score > 0.0;
}

PtPlan plan_ptile_dw_uncached(int B, int C, int H, int W, int L, int k, int dtype) {
    PtPlan p;
    const int eb = elem_bytes(dtype);
    if (B < 1 || L < 1 || H % (1 << L) != 0 || W % (1 << L) != 0) return p;
    const int sms = device_sms();
    if (sms <= 0) { p.status = WTCONV_ERR_CUDA; return p; }
    int h = H, w = W, pitch = W, e = eb, lvl = 0;
    for (int i = 0; lvl < L; ++i) {
        const int LT = std::min(2, L - lvl);
        if (!pt_choose(p.a[i], p.smem[i], p.occ[i], B, C, h, w, pitch, e, dtype, k, LT, i == 0 ? 1 : 0, lvl, L)) return p;
        lvl += LT;
        if (p.a[i].ll_out) {
            h = p.a[i].ll_h;
            w = p.a[i].ll_w;
            pitch = p.a[i].ll_pitch;
            e = 4;
        }
        p.nlaunch = i + 1;
    }
    // partial rows per channel: enough units to keep every resident CTA of launch 0 busy
    const PtileArgs &a0 = p.a[0];
    const long long slots = (long long)sms * p.occ[0];
    int nchunks = (int)std::min<long long>(a0.work, std::max<long long>(1, (2 * slots + C - 1) / C));
    size_t off = 0;
    const int nsig = 1 + 4 * L, NA = k * k + 1;
    p.partial_bytes = round256((size_t)nchunks * C * nsig * NA * sizeof(float));
    off = p.partial_bytes;
    for (int i = 0; i < p.nlaunch; ++i) {
        PtileArgs &a = p.a[i];
        a.nchunks = nchunks;
        a.units = C * nchunks;
        a.grid = (int)std::min<long long>(a.units, (long long)sms * p.occ[i]);
        if (a.ll_out) {
            p.ll_half[i] = round256((size_t)B * C * a.ll_h * a.ll_pitch * sizeof(float));
            p.ll_off[i] = off;
            off += 2 * p.ll_half[i];
        }
    }
    p.workspace = off;
    p.status = WTCONV_OK;
    return p;
}

PtPlan plan_ptile_dw(int B, int C, int H, int W, int L, int k, int dtype) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, int, int, int, std::string>, PtPlan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        PtPlan p;
        p.status = WTCONV_ERR_CUDA;
        return p;
    }
    const char *kn = getenv("WTCONV_PTILE");
    const auto key = std::make_tuple(B, C, H, W, L, k, dtype, dev, std::string(kn ? kn : ""));
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    PtPlan p = plan_ptile_dw_uncached(B, C, H, W, L, k, dtype);
    const char *verbose = getenv("WTCONV_VERBOSE");
    if (verbose && verbose[0] == '1')
        for (int i = 0; i < p.nlaunch; ++i)
            fprintf(stderr, "wtconv plan ptile-dw[%d] B=%d C=%d H=%d W=%d L=%d k=%d dtype=%d: status %d LT=%d base=%d "
                            "tile=%dx%d halo=%d G=%d threads=%d items/pair=%d (%dx%d) grid=%d units=%d chunks=%d smem=%zu occ=%d\n",
                    i, B, C, p.a[i].H, p.a[i].W, L, k, dtype, p.status, p.a[i].LT, p.a[i].base, p.a[i].TH, p.a[i].TW,
                    p.a[i].HX, p.a[i].G, p.a[i].nthreads, p.a[i].per_pair, p.a[i].lv[1].Q, p.a[i].lv[1].S, p.a[i].grid,
                    p.a[i].units, p.a[i].nchunks, p.smem[i], p.occ[i]);
    if (p.status == WTCONV_OK || p.status == WTCONV_ERR_UNSUPPORTED) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, p);
    }
    return p;
}

// Forward / input-gradient path of a shape (WTCONV_FWD_PATH=pair / fused / plane / ptile / tiles
// selects a path where it applies).  By default the batch-pair whole-plane kernel runs where it
// measured fastest; else the fused whole-plane kernel where it measured fastest on GB300: fp32
// planes with at least 64 output items and three or more resident CTAs per SM; else the
// whole-plane kernel where the pyramid fits; else the deep kernel followed by the tiled batch-pair
// shallow kernel; else the deep kernel followed by the one-warp tiled shallow kernel.
enum FwdPath { FWD_FUSED, FWD_PLANE, FWD_TILES, FWD_PAIR, FWD_PTILE };
struct FwdChoice {
    int status = WTCONV_OK;
    FwdPath path = FWD_PLANE;
    PPlan pp;
    Plan pf;
    PairPlan pr;
    PsPlan ps;
};

FwdChoice choose_fwd(int B, int C, int H, int W, int L, int k, int dtype) {
    FwdChoice f;
    const char *env = getenv("WTCONV_FWD_PATH");
    const bool want_fused = env && strcmp(env, "fused") == 0;
    const bool want_tiles = env && strcmp(env, "tiles") == 0;
    const bool want_plane = env && strcmp(env, "plane") == 0;
    const bool want_pair = env && strcmp(env, "pair") == 0;
    const bool want_ptile = env && strcmp(env, "ptile") == 0;
    if (want_ptile) {
        f.ps = plan_pshallow(B, C, H, W, L, k, dtype);
        if (f.ps.status != WTCONV_OK && f.ps.status != WTCONV_ERR_UNSUPPORTED) { f.status = f.ps.status; return f; }
        if (f.ps.status == WTCONV_OK) {
            f.path = FWD_PTILE;
            return f;
        }
    }
    if (!want_tiles && !want_plane && !want_fused) {
        f.pr = plan_pair_fwd(B, C, H, W, L, k, dtype);
        if (f.pr.status != WTCONV_OK && f.pr.status != WTCONV_ERR_UNSUPPORTED) { f.status = f.pr.status; return f; }
        if (f.pr.status == WTCONV_OK && (want_pair || pair_default(false, H, W, L, k, dtype))) {
            f.path = FWD_PAIR;
            return f;
        }
    }
    if (!want_tiles && !want_plane) {
        f.pp = plan_plane(B, C, H, W, L, k, dtype);
        if (f.pp.status != WTCONV_OK && f.pp.status != WTCONV_ERR_UNSUPPORTED) { f.status = f.pp.status; return f; }
        const bool good = f.pp.status == WTCONV_OK && dtype == WTCONV_F32 && f.pp.occ >= 3 &&
                          f.pp.a.sg.items_r * f.pp.a.sg.items_c >= 64;
        if (f.pp.status == WTCONV_OK && (want_fused || good)) {
            f.path = FWD_FUSED;
            return f;
        }
    }
    f.pf = plan_forward(B, C, H, W, L, k, dtype);
    if (f.pf.status == WTCONV_OK && !want_tiles) {
        f.path = FWD_PLANE;
        return f;
    }
    if (f.pf.status != WTCONV_OK && f.pf.status != WTCONV_ERR_UNSUPPORTED) { f.status = f.pf.status; return f; }
    if (!want_tiles) {
        f.ps = plan_pshallow(B, C, H, W, L, k, dtype);
        if (f.ps.status != WTCONV_OK && f.ps.status != WTCONV_ERR_UNSUPPORTED) { f.status = f.ps.status; return f; }
        if (f.ps.status == WTCONV_OK) {
            f.path = FWD_PTILE;
            return f;
        }
    }
    f.path = FWD_TILES;
    return f;
}

// Which weight-gradient path a call takes: the batch-pair kernel where it measured fastest, the
// fused whole-plane kernel where it applies and measured fastest, else the whole-plane kernel
// where a plane fits, else the tiled batch-pair kernel, else the tiled kernels where they apply,
// else the workspace pyramids.  WTCONV_DW_PATH=pair, =fused, =plane, =ptile, =tiles or =pyramid
// selects a path where it applies (for testing and comparison).
enum DwPath { DW_TILE, DW_PLANE, DW_PYRAMID, DW_FUSED, DW_PAIR, DW_PTILE };
struct DwChoice {
    int status = WTCONV_OK;
    DwPath path = DW_PLANE;
    TPlan t;
    Plan p;
    FPlan f;
    PairPlan pr;
    PtPlan pt;
    size_t workspace = 0;
};

// Where the fused kernel measured faster than the staged whole-plane kernel on GB300: fp32
// planes of at least 64 base items with two resident CTAs per SM (narrow types and larger
// planes ran up to 2x slower).
bool dw_fused_default(const FPlan &f, int dtype) {
    return f.status == WTCONV_OK && dtype == WTCONV_F32 && f.occ >= 2 && f.a.sg.items_r * f.a.sg.items_c >= 64;
}

DwChoice choose_dw(int B, int C, int H, int W, int L, int k, int dtype) {
    DwChoice d;
    const char *env = getenv("WTCONV_DW_PATH");
    const bool want_tiles = env && strcmp(env, "tiles") == 0;
    const bool want_pyramid = env && strcmp(env, "pyramid") == 0;
    const bool want_fused = env && strcmp(env, "fused") == 0;
    const bool want_plane = env && strcmp(env, "plane") == 0;
    const bool want_pair = env && strcmp(env, "pair") == 0;
    const bool want_ptile = env && strcmp(env, "ptile") == 0;
    if (want_ptile) {
        d.pt = plan_ptile_dw(B, C, H, W, L, k, dtype);
        if (d.pt.status != WTCONV_OK && d.pt.status != WTCONV_ERR_UNSUPPORTED) { d.status = d.pt.status; return d; }
        if (d.pt.status == WTCONV_OK) {
            d.path = DW_PTILE;
            d.workspace = d.pt.workspace;
            return d;
        }
    }
    if (!want_tiles && !want_pyramid && !want_plane && !want_fused) {
        d.pr = plan_pair_dw(B, C, H, W, L, k, dtype);
        if (d.pr.status != WTCONV_OK && d.pr.status != WTCONV_ERR_UNSUPPORTED) { d.status = d.pr.status; return d; }
        if (d.pr.status == WTCONV_OK && (want_pair || pair_default(true, H, W, L, k, dtype))) {
            d.path = DW_PAIR;
            d.workspace = d.pr.workspace;
            return d;
        }
    }
    if (!want_tiles && !want_pyramid && !want_plane) {
        d.f = plan_dw_fused(B, C, H, W, L, k, dtype);
        if (d.f.status != WTCONV_OK && d.f.status != WTCONV_ERR_UNSUPPORTED) { d.status = d.f.status; return d; }
        if (d.f.status == WTCONV_OK && (want_fused || dw_fused_default(d.f, dtype))) {
            d.path = DW_FUSED;
            d.workspace = d.f.partial_bytes;
            return d;
        }
    }
    if (!want_tiles && !want_pyramid) {
        d.p = plan_dw(B, C, H, W, L, k, dtype);
        if (d.p.status != WTCONV_OK) { d.status = d.p.status; return d; }
        if (!d.p.dw_pyramid) {
            d.path = DW_PLANE;
            d.workspace = d.p.workspace;
            return d;
        }
    }
    // planes too large for the whole-plane kernels: the tiled batch-pair kernel where its bulk
    // copies apply (256 x 256 bf16 planes, L = 5: 582 vs 882 us), else the tiled kernels
    if (!want_tiles && !want_pyramid) {
        d.pt = plan_ptile_dw(B, C, H, W, L, k, dtype);
        if (d.pt.status != WTCONV_OK && d.pt.status != WTCONV_ERR_UNSUPPORTED) { d.status = d.pt.status; return d; }
        if (d.pt.status == WTCONV_OK) {
            d.path = DW_PTILE;
            d.workspace = d.pt.workspace;
            return d;
        }
    }
    if (!want_pyramid) {
        d.t = plan_dw_tile(B, C, H, W, L, k, dtype);
        if (d.t.status == WTCONV_OK) {
            d.path = DW_TILE;
            d.workspace = d.t.workspace;
            return d;
        }
        if (d.t.status != WTCONV_ERR_UNSUPPORTED) { d.status = d.t.status; return d; }
    }
    d.p = want_pyramid ? plan_dw_pyramid_only(B, C, H, W, L, k, dtype) : plan_dw(B, C, H, W, L, k, dtype);
    if (d.p.status != WTCONV_OK) { d.status = d.p.status; return d; }
    d.path = d.p.dw_pyramid ? DW_PYRAMID : DW_PLANE;
    d.workspace = d.p.workspace;
    return d;
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

// Sticky flag raised by a kernel wait that gave up; read and cleared by wtconv_device_status.
__device__ int g_wait_timeout;

// Device address of g_wait_timeout on the current device (looked up once per device), or nullptr.
int *timeout_flag() {
    static std::mutex mu;
    static std::map<int, int *> addr;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) return it->second;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wait_timeout) != cudaSuccess || p == nullptr) return nullptr;
    addr.emplace(dev, static_cast<int *>(p));
    return static_cast<int *>(p);
}

// Scratch of wtconv_backward_weights_noalloc: the weight-gradient partials of one call, in device
// memory that comes with the library's module instead of from an allocator.
__device__ __align__(256) unsigned char g_noalloc_scratch[WTCONV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up once per device (with
// that device current) and cached; nullptr if the lookup fails.
void *noalloc_scratch() {
    static std::mutex mu;
    static std::map<int, void *> addr;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) return it->second;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    addr.emplace(dev, p);
    return p;
}

}  // namespace

// Workspace of `op` on planes whose sides are multiples of 2^L.
static int workspace_inner(int op, int B, int C, int H, int W, int L, int k, int dtype, size_t *bytes) {
    *bytes = 0;
    if (op != WTCONV_OP_FORWARD && op != WTCONV_OP_BACKWARD_INPUT && op != WTCONV_OP_BACKWARD_WEIGHTS &&
        op != WTCONV_OP_BACKWARD)
        return WTCONV_ERR_INVALID_ARG;
    if (op == WTCONV_OP_FORWARD || op == WTCONV_OP_BACKWARD_INPUT || op == WTCONV_OP_BACKWARD)
        *bytes += deep_bytes(B, C, H, W, L);
    if (op == WTCONV_OP_BACKWARD_WEIGHTS || op == WTCONV_OP_BACKWARD) {
        const DwChoice d = choose_dw(B, C, H, W, L, k, dtype);
        if (d.status != WTCONV_OK) return d.status;
        *bytes += d.workspace;
    }
    return WTCONV_OK;
}

// Padded activation tensors `op` keeps in the workspace when the sides are not multiples of 2^L:
// forward x and y, input gradient dy and dx, weight gradients x and dy, backward x, dy and dx.
static int pad_buffers(int op) { return op == WTCONV_OP_BACKWARD ? 3 : 2; }

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
    case WTCONV_ERR_SCRATCH_LIMIT: return "shape needs more scratch than the no-alloc entry point's fixed array";
    case WTCONV_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait gave up (device status flag)";
    default: return "unknown status";
    }
}

size_t wtconv_workspace_size(int op, int B, int C, int H, int W, int L, int k, int dtype) {
    if (validate_shape(B, C, H, W, L, k, dtype) != WTCONV_OK) return 0;
    const PadDims pd = pad_dims(B, C, H, W, L, dtype);
    size_t bytes = 0;
    if (workspace_inner(op, B, C, pd.Hp, pd.Wp, L, k, dtype, &bytes) != WTCONV_OK) return 0;
    return bytes + (pd.on ? pad_buffers(op) * pd.act_bytes : 0);
}

int wtconv_selftest_wait_timeout(wtconv_stream_t stream) {
    int *flag = timeout_flag();
    if (flag == nullptr) return WTCONV_ERR_CUDA;
    return cuda_status(launch_wait_selftest(flag, reinterpret_cast<cudaStream_t>(stream)));
}

int wtconv_fp32_fma_peak(int iters, double *tflops) {
    if (iters <= 0 || tflops == nullptr) return WTCONV_ERR_INVALID_ARG;
    return cuda_status(measure_fma_peak(iters, tflops));
}

int wtconv_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return WTCONV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_timeout, sizeof(int)) != cudaSuccess) return WTCONV_ERR_CUDA;
    if (v == 0) return WTCONV_OK;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_wait_timeout, &zero, sizeof(int)) != cudaSuccess) return WTCONV_ERR_CUDA;
    return WTCONV_ERR_DEVICE_TIMEOUT;
}

static const char *plan_kernels_inner(int op, int B, int C, int H, int W, int L, int k, int dtype) {
    const bool fwd = op == WTCONV_OP_FORWARD || op == WTCONV_OP_BACKWARD_INPUT;
    const bool dw = op == WTCONV_OP_BACKWARD_WEIGHTS;
    const bool both = op == WTCONV_OP_BACKWARD;
    if (!fwd && !dw && !both) return "";
    const char *f = "";
    if (fwd || both) {
        const FwdChoice fc = choose_fwd(B, C, H, W, L, k, dtype);
        if (fc.status != WTCONV_OK) return "";
        f = fc.path == FWD_PAIR ? "wtconv_pair_fwd_kernel"
            : fc.path == FWD_FUSED ? "wtconv_plane_kernel"
            : fc.path == FWD_PLANE ? "wtconv_fwd_kernel"
            : fc.path == FWD_PTILE ? (L >= 2 ? "wtconv_deep_kernel+wtconv_pshallow_kernel" : "wtconv_pshallow_kernel")
            : (L >= 2 ? "wtconv_deep_kernel+wtconv_shallow_kernel" : "wtconv_shallow_kernel");
        if (fwd) return f;
    }
    const DwChoice d = choose_dw(B, C, H, W, L, k, dtype);
    if (d.status != WTCONV_OK) return "";
    if (dw) {
        return d.path == DW_PTILE ? "wtconv_ptile_dw_kernel+wtconv_dw_finalize_kernel"
             : d.path == DW_PAIR ? "wtconv_pair_dw_kernel+wtconv_dw_finalize_kernel"
             : d.path == DW_FUSED ? "wtconv_dw_plane_kernel+wtconv_dw_finalize_kernel"
             : d.path == DW_PLANE ? "wtconv_dw_kernel+wtconv_dw_finalize_kernel"
             : d.path == DW_TILE ? "wtconv_dw_tile_kernel+wtconv_level2_kernel+wtconv_haar_level_kernel+"
                                   "wtconv_dw_corr_kernel+wtconv_dw_finalize_kernel"
                                 : "wtconv_haar_level_kernel+wtconv_dw_corr_kernel+wtconv_dw_finalize_kernel";
    }
    // BACKWARD: the input gradient's kernels, then the weight gradient's (names built once per
    // combination; static storage)
    static std::mutex mu;
    static std::map<std::string, std::string> names;
    const std::string dws = d.path == DW_PTILE ? "wtconv_ptile_dw_kernel+wtconv_dw_finalize_kernel"
                            : d.path == DW_PAIR ? "wtconv_pair_dw_kernel+wtconv_dw_finalize_kernel"
                            : d.path == DW_FUSED ? "wtconv_dw_plane_kernel+wtconv_dw_finalize_kernel"
                            : d.path == DW_PLANE ? "wtconv_dw_kernel+wtconv_dw_finalize_kernel"
                            : d.path == DW_TILE ? "wtconv_dw_tile_kernel+wtconv_level2_kernel+wtconv_haar_level_kernel+"
                                                  "wtconv_dw_corr_kernel+wtconv_dw_finalize_kernel"
                                                : "wtconv_haar_level_kernel+wtconv_dw_corr_kernel+wtconv_dw_finalize_kernel";
    const std::string key = std::string(f) + "+" + dws;
    std::lock_guard<std::mutex> lock(mu);
    auto it = names.emplace(key, key).first;
    return it->second.c_str();
}

const char *wtconv_plan_kernels(int op, int B, int C, int H, int W, int L, int k, int dtype) {
    if (validate_shape(B, C, H, W, L, k, dtype) != WTCONV_OK) return "";
    const PadDims pd = pad_dims(B, C, H, W, L, dtype);
    const char *inner = plan_kernels_inner(op, B, C, pd.Hp, pd.Wp, L, k, dtype);
    if (!pd.on || inner[0] == 0) return inner;
    // padded planes: the pads before, the crop after
    const bool two_in = op == WTCONV_OP_BACKWARD_WEIGHTS || op == WTCONV_OP_BACKWARD;
    const bool crop = op != WTCONV_OP_BACKWARD_WEIGHTS;
    const std::string key = std::string(two_in ? "wtconv_pad_kernel+wtconv_pad_kernel+" : "wtconv_pad_kernel+") +
                            inner + (crop ? "+wtconv_crop_kernel" : "");
    static std::mutex mu;
    static std::map<std::string, std::string> names;
    std::lock_guard<std::mutex> lock(mu);
    auto it = names.emplace(key, key).first;
    return it->second.c_str();
}

static int launch_count_inner(int op, int B, int C, int H, int W, int L, int k, int dtype);

int wtconv_launch_count(int op, int B, int C, int H, int W, int L, int k, int dtype) {
    if (validate_shape(B, C, H, W, L, k, dtype) != WTCONV_OK) return 0;
    const PadDims pd = pad_dims(B, C, H, W, L, dtype);
    const int n = launch_count_inner(op, B, C, pd.Hp, pd.Wp, L, k, dtype);
    if (!pd.on || n == 0) return n;
    return n + (op == WTCONV_OP_BACKWARD ? 3 : 2);  // pads and crop
}

static int launch_count_inner(int op, int B, int C, int H, int W, int L, int k, int dtype) {
    int n = 0;
    if (op == WTCONV_OP_FORWARD || op == WTCONV_OP_BACKWARD_INPUT || op == WTCONV_OP_BACKWARD) {
        const FwdChoice f = choose_fwd(B, C, H, W, L, k, dtype);
        if (f.status != WTCONV_OK) return 0;
        n += (f.path == FWD_TILES || f.path == FWD_PTILE) ? (L >= 2 ? 2 : 1) : 1;
    }
    if (op == WTCONV_OP_BACKWARD_WEIGHTS || op == WTCONV_OP_BACKWARD) {
        const DwChoice d = choose_dw(B, C, H, W, L, k, dtype);
        if (d.status != WTCONV_OK) return 0;
        if (d.path == DW_TILE) n += 2 + (L >= 2 ? 1 + (L - 2) + (L - 1) : 0);  // tiles, level 2, levels, corr, finalize
        else if (d.path == DW_PTILE) n += d.pt.nlaunch + 1;                       // tile launches, finalize
        else n += d.path == DW_PYRAMID ? 2 * L + 2 : 2;
    }
    return n;
}

// The layer's linear operator on `src` (x -> y, or dy -> dx with rotated kernels and no bias):
// deep kernel (levels >= 2 -> contribution at level-1 resolution, in the workspace), then the
// shallow kernel (base conv + level 1 + synthesis, final outputs).
static int run_operator(int B, int C, int H, int W, int L, int k, int dtype, const void *src, const float *base_w,
                        const float *base_bias, const float *base_scale, const float *wavelet_w,
                        const float *wavelet_scale, void *dst, bool flip, void *workspace, size_t workspace_bytes,
                        cudaStream_t s) {
    const FwdChoice fc = choose_fwd(B, C, H, W, L, k, dtype);
    if (fc.status != WTCONV_OK) return fc.status;
    if (fc.path == FWD_PAIR) {
        PairArgs a = fc.pr.a;
        a.x = src;
        a.out = dst;
        a.base_w = base_w; a.base_bias = base_bias; a.base_scale = base_scale;
        a.wavelet_w = wavelet_w; a.wavelet_scale = wavelet_scale;
        a.flip = flip ? 1 : 0;
        a.with_bias = flip ? 0 : 1;
        a.timeout = timeout_flag();
        if (a.timeout == nullptr) return WTCONV_ERR_CUDA;
        if (a.tma_map && !encode_map(&a.tmap_x, tma_dtype(dtype), elem_bytes(dtype), src, a.tma_rlen, a.tma_rows, C, B,
                                     a.tma_rlen, a.tma_rows, 2 * a.G))
            return WTCONV_ERR_CUDA;
        return cuda_status(launch_pair_fwd(a, dtype, fc.pr.smem, s));
    }
    if (fc.path == FWD_FUSED) {
        PPlan pp = fc.pp;
        PlaneArgs &a = pp.a;
        a.x = src;
        a.out = dst;
        a.base_w = base_w; a.base_bias = base_bias; a.base_scale = base_scale;
        a.wavelet_w = wavelet_w; a.wavelet_scale = wavelet_scale;
        a.flip = flip ? 1 : 0;
        a.with_bias = flip ? 0 : 1;
        a.timeout = timeout_flag();
        if (a.timeout == nullptr) return WTCONV_ERR_CUDA;
        const int eb = elem_bytes(dtype);
        if (!encode_map(&a.tmap_x, tma_dtype(dtype), eb, src, W, H, C, B, a.sg.xw, a.sg.xrows, 1))
            return WTCONV_ERR_CUDA;
        return cuda_status(launch_plane(a, dtype, pp.smem, s));
    }
    if (fc.path == FWD_PLANE) {
        // planes whose whole pyramid fits in shared memory: one kernel, no workspace
        Plan pf = fc.pf;
        pf.a.x = src;
        pf.a.out = dst;
        set_params(pf.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
        pf.a.flip = flip ? 1 : 0;
        pf.a.with_bias = flip ? 0 : 1;
        return cuda_status(launch_forward(pf.a, dtype, pf.smem, s));
    }
    const size_t dbytes = deep_bytes(B, C, H, W, L);
    Plan pd;
    if (L >= 2) {
        pd = plan_deep(B, C, H, W, L, k, dtype);
        if (pd.status != WTCONV_OK) return pd.status;
    }
    SPlan ps;
    if (fc.path == FWD_TILES) {
        ps = plan_shallow(B, C, H, W, L, k, dtype);
        if (ps.status != WTCONV_OK) return ps.status;
    }
    if (workspace_bytes < dbytes || (dbytes > 0 && !aligned16(workspace))) return WTCONV_ERR_WORKSPACE;
    float *deep = L >= 2 ? static_cast<float *>(workspace) : nullptr;
    if (L >= 2) {
        pd.a.x = src;
        set_params(pd.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
        pd.a.flip = flip ? 1 : 0;
        pd.a.with_bias = 0;
        if (launch_deep(pd.a, deep, dtype, pd.smem, s) != cudaSuccess) return WTCONV_ERR_CUDA;
    }
    const int eb = elem_bytes(dtype);
    if (fc.path == FWD_PTILE) {
        PsArgs a = fc.ps.a;
        a.x = src;
        a.deep = deep;
        a.out = dst;
        a.base_w = base_w; a.base_bias = base_bias; a.base_scale = base_scale;
        a.wavelet_w = wavelet_w; a.wavelet_scale = wavelet_scale;
        a.flip = flip ? 1 : 0;
        a.with_bias = flip ? 0 : 1;
        a.timeout = timeout_flag();
        if (a.timeout == nullptr) return WTCONV_ERR_CUDA;
        if (!encode_map(&a.tmap_x, tma_dtype(dtype), eb, src, W, H, C, B, a.RXW, a.RXR, 2 * a.G))
            return WTCONV_ERR_CUDA;
        if (deep != nullptr && !encode_map(&a.tmap_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, deep, W / 2, H / 2, C, B,
                                           a.TW / 2, a.TH / 2, 2 * a.G))
            return WTCONV_ERR_CUDA;
        return cuda_status(launch_pshallow(a, dtype, fc.ps.smem, s));
    }
    ShallowArgs &a = ps.a;
    a.x = src;
    a.deep = deep;
    a.out = dst;
    a.base_w = base_w; a.base_bias = base_bias; a.base_scale = base_scale;
    a.wavelet_w = wavelet_w; a.wavelet_scale = wavelet_scale;
    a.flip = flip ? 1 : 0;
    a.with_bias = flip ? 0 : 1;
    a.timeout = timeout_flag();
    if (a.timeout == nullptr) return WTCONV_ERR_CUDA;
    a.tma_x = shallow_tma_x_ok(a, eb) &&
              encode_map(&a.tmap_x, tma_dtype(dtype), eb, src, W, H, C, B, a.sg.xw, a.sg.xrows, a.sg.G);
    a.tma_d = deep != nullptr && shallow_tma_d_ok(a) &&
              encode_map(&a.tmap_d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, deep, W / 2, H / 2, C, B, a.sg.TW / 2,
                         a.sg.TH / 2, a.sg.G);
    return cuda_status(launch_shallow(a, dtype, ps.smem, s));
}

// The operator on planes padded to multiples of 2^L: pad src into the workspace, run, crop into dst.
static int run_padded_operator(int B, int C, int H, int W, int L, int k, int dtype, const PadDims &pd,
                               const void *src, const float *base_w, const float *base_bias, const float *base_scale,
                               const float *wavelet_w, const float *wavelet_scale, void *dst, bool flip,
                               void *workspace, size_t workspace_bytes, cudaStream_t s) {
    size_t inner = 0;
    int st = workspace_inner(flip ? WTCONV_OP_BACKWARD_INPUT : WTCONV_OP_FORWARD, B, C, pd.Hp, pd.Wp, L, k, dtype,
                             &inner);
    if (st != WTCONV_OK) return st;
    const size_t bufs = 2 * pd.act_bytes;
    if (workspace_bytes < bufs + inner || !aligned16(workspace)) return WTCONV_ERR_WORKSPACE;
    char *w = static_cast<char *>(workspace);
    const int eb = elem_bytes(dtype);
    const long long planes = (long long)B * C;
    if (launch_pad_planes(src, w, planes, H, W, pd.Hp, pd.Wp, eb, s) != cudaSuccess) return WTCONV_ERR_CUDA;
    st = run_operator(B, C, pd.Hp, pd.Wp, L, k, dtype, w, base_w, base_bias, base_scale, wavelet_w, wavelet_scale,
                      w + pd.act_bytes, flip, w + bufs, workspace_bytes - bufs, s);
    if (st != WTCONV_OK) return st;
    return cuda_status(launch_crop_planes(w + pd.act_bytes, dst, planes, H, W, pd.Hp, pd.Wp, eb, s));
}

int wtconv_forward(int B, int C, int H, int W, int L, int k, int dtype, const void *x, const float *base_w,
                   const float *base_bias, const float *base_scale, const float *wavelet_w,
                   const float *wavelet_scale, void *y, void *workspace, size_t workspace_bytes,
                   wtconv_stream_t stream) {
    int st = validate_shape(B, C, H, W, L, k, dtype);
    if (st != WTCONV_OK) return st;
    if (!aligned16(x) || !aligned16(y) || !params_ok(base_w, base_bias, base_scale, wavelet_w, wavelet_scale))
        return WTCONV_ERR_INVALID_ARG;
    if (fault_injected()) return WTCONV_ERR_INJECTED;
    const PadDims pd = pad_dims(B, C, H, W, L, dtype);
    if (pd.on)
        return run_padded_operator(B, C, H, W, L, k, dtype, pd, x, base_w, base_bias, base_scale, wavelet_w,
                                   wavelet_scale, y, false, workspace, workspace_bytes,
                                   reinterpret_cast<cudaStream_t>(stream));
    return run_operator(B, C, H, W, L, k, dtype, x, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, y,
                        false, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int wtconv_backward_input(int B, int C, int H, int W, int L, int k, int dtype, const float *base_w,
                          const float *base_bias, const float *base_scale, const float *wavelet_w,
                          const float *wavelet_scale, const void *dy, void *dx, void *workspace,
                          size_t workspace_bytes, wtconv_stream_t stream) {
    int st = validate_shape(B, C, H, W, L, k, dtype);
    if (st != WTCONV_OK) return st;
    if (!aligned16(dy) || !aligned16(dx) || !params_ok(base_w, base_bias, base_scale, wavelet_w, wavelet_scale))
        return WTCONV_ERR_INVALID_ARG;
    if (fault_injected()) return WTCONV_ERR_INJECTED;
    const PadDims pd = pad_dims(B, C, H, W, L, dtype);
    if (pd.on)
        return run_padded_operator(B, C, H, W, L, k, dtype, pd, dy, base_w, base_bias, base_scale, wavelet_w,
                                   wavelet_scale, dx, true, workspace, workspace_bytes,
                                   reinterpret_cast<cudaStream_t>(stream));
    return run_operator(B, C, H, W, L, k, dtype, dy, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, dx,
                        true, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

// Fused whole-plane weight-gradient kernel into `partials`; fills what the finalize reads.
static int run_dw_fused(FPlan &fp, int dtype, const void *x, const void *dy, float *partials, LayerArgs &fin,
                        cudaStream_t s) {
    DwPlaneArgs &f = fp.a;
    const int eb = elem_bytes(dtype);
    f.partials = partials;
    f.timeout = timeout_flag();
    if (f.timeout == nullptr) return WTCONV_ERR_CUDA;
    if (!encode_map(&f.tmap_x, tma_dtype(dtype), eb, x, f.W, f.H, f.C, f.B, f.sg.xw, f.sg.xrows, 1) ||
        !encode_map(&f.tmap_dy, tma_dtype(dtype), eb, dy, f.W, f.H, f.C, f.B, f.sg.TW, f.sg.TH, 1))
        return WTCONV_ERR_CUDA;
    if (launch_dw_plane(f, dtype, fp.smem, s) != cudaSuccess) return WTCONV_ERR_CUDA;
    fin.B = f.B; fin.C = f.C; fin.H = f.H; fin.W = f.W; fin.L = f.L; fin.K = f.K;
    fin.nb = f.nb;
    fin.partials = partials;
    return WTCONV_OK;
}

// Tiled batch-pair weight-gradient launches: partials at the start of `wsp`, the LL planes of the
// deeper launches after them; fills what the finalize reads.
static int run_dw_ptile(const PtPlan &pt, int dtype, const void *x, const void *dy, char *wsp, LayerArgs &fin,
                        cudaStream_t s) {
    float *partials = reinterpret_cast<float *>(wsp);
    const void *in_x = x, *in_dy = dy;
    int in_dtype = dtype;
    int *timeout = timeout_flag();
    if (timeout == nullptr) return WTCONV_ERR_CUDA;
    for (int i = 0; i < pt.nlaunch; ++i) {
        PtileArgs a = pt.a[i];
        a.x = in_x;
        a.dy = in_dy;
        a.partials = partials;
        a.timeout = timeout;
        if (a.ll_out) {
            a.ll_x = reinterpret_cast<float *>(wsp + pt.ll_off[i]);
            a.ll_dy = reinterpret_cast<float *>(wsp + pt.ll_off[i] + pt.ll_half[i]);
        }
        const int eb = elem_bytes(in_dtype);
        if (!encode_map_pitched(&a.tmap_x, tma_dtype(in_dtype), eb, in_x, a.W, a.H, a.C, a.B, a.in_pitch, a.RXW, a.RXR,
                                2 * a.G) ||
            !encode_map_pitched(&a.tmap_dy, tma_dtype(in_dtype), eb, in_dy, a.W, a.H, a.C, a.B, a.in_pitch, a.TW, a.TH,
                                2 * a.G))
            return WTCONV_ERR_CUDA;
        if (launch_ptile_dw(a, in_dtype, pt.smem[i], s) != cudaSuccess) return WTCONV_ERR_CUDA;
        in_x = a.ll_x;
        in_dy = a.ll_dy;
        in_dtype = WTCONV_F32;
    }
    const PtileArgs &a0 = pt.a[0];
    fin.B = a0.B; fin.C = a0.C; fin.H = a0.H; fin.W = a0.W; fin.L = a0.L_total; fin.K = a0.K;
    fin.nb = a0.nchunks;
    fin.partials = partials;
    return WTCONV_OK;
}

// Batch-pair weight-gradient kernel into `partials`; fills what the finalize reads.
static int run_dw_pair(const PairPlan &pp, int dtype, const void *x, const void *dy, float *partials, LayerArgs &fin,
                       cudaStream_t s) {
    PairArgs a = pp.a;
    a.x = x;
    a.dy = dy;
    a.partials = partials;
    a.timeout = timeout_flag();
    if (a.timeout == nullptr) return WTCONV_ERR_CUDA;
    if (a.tma_map) {
        const int eb = elem_bytes(dtype);
        if (!encode_map(&a.tmap_x, tma_dtype(dtype), eb, x, a.tma_rlen, a.tma_rows, a.C, a.B, a.tma_rlen, a.tma_rows,
                        2 * a.G) ||
            !encode_map(&a.tmap_dy, tma_dtype(dtype), eb, dy, a.tma_rlen, a.tma_rows, a.C, a.B, a.tma_rlen,
                        a.tma_rows, 2 * a.G))
            return WTCONV_ERR_CUDA;
    }
    if (launch_pair_dw(a, dtype, pp.smem, s) != cudaSuccess) return WTCONV_ERR_CUDA;
    fin.B = a.B; fin.C = a.C; fin.H = a.H; fin.W = a.W; fin.L = a.L; fin.K = a.K;
    fin.nb = a.nb;
    fin.partials = partials;
    return WTCONV_OK;
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
    DwChoice dc = choose_dw(B, C, H, W, L, k, dtype);
    if (dc.status != WTCONV_OK) return dc.status;
    const size_t dbytes = want_dx ? deep_bytes(B, C, H, W, L) : 0;
    if (workspace_bytes < dbytes + dc.workspace || (dbytes + dc.workspace > 0 && !aligned16(workspace)))
        return WTCONV_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (want_dx) {
        st = run_operator(B, C, H, W, L, k, dtype, dy, base_w, base_bias, base_scale, wavelet_w, wavelet_scale, dx,
                          true, workspace, dbytes, s);
        if (st != WTCONV_OK) return st;
    }
    char *wsp = static_cast<char *>(workspace) + dbytes;
    LayerArgs fin{};  // what the finalize kernel reads
    if (dc.path == DW_TILE) {
        // base path and level 1 on tiles (signals 0 .. 4), levels >= 2 on their pyramids
        DwTileArgs &t = dc.t.a;
        const int eb = elem_bytes(dtype);
        t.partials = reinterpret_cast<float *>(wsp);
        t.timeout = timeout_flag();
        if (t.timeout == nullptr) return WTCONV_ERR_CUDA;
        if (!encode_map(&t.tmap_x, tma_dtype(dtype), eb, x, W, H, C, B, t.sg.xw, t.sg.xrows, t.sg.G) ||
            !encode_map(&t.tmap_dy, tma_dtype(dtype), eb, dy, W, H, C, B, t.sg.TW, t.sg.TH, t.sg.G))
            return WTCONV_ERR_CUDA;
        if (launch_dw_tile(t, dtype, dc.t.smem, s) != cudaSuccess) return WTCONV_ERR_CUDA;
        if (L >= 2) {
            DwPyramidArgs d{};
            d.B = B; d.C = C; d.H = H; d.W = W; d.L = L; d.K = k;
            d.from_level = 2;
            d.nb = t.nb;
            d.x = x; d.dy = dy;
            char *pw = wsp + dc.t.partial_bytes;
            for (int l = 2; l <= L; ++l) {
                const size_t lb = ((size_t)B * C * (H >> l) * (W >> l) * sizeof(float4) + 255) / 256 * 256;
                d.pyr_x[l] = reinterpret_cast<float4 *>(pw);
                d.pyr_dy[l] = reinterpret_cast<float4 *>(pw + lb);
                pw += 2 * lb;
            }
            d.partials = t.partials;
            if (launch_dw_pyramid(d, dtype, s) != cudaSuccess) return WTCONV_ERR_CUDA;
        }
        fin.B = B; fin.C = C; fin.H = H; fin.W = W; fin.L = L; fin.K = k;
        fin.nb = t.nb;
        fin.partials = t.partials;
    } else if (dc.path == DW_FUSED) {
        st = run_dw_fused(dc.f, dtype, x, dy, reinterpret_cast<float *>(wsp), fin, s);
        if (st != WTCONV_OK) return st;
    } else if (dc.path == DW_PAIR) {
        st = run_dw_pair(dc.pr, dtype, x, dy, reinterpret_cast<float *>(wsp), fin, s);
        if (st != WTCONV_OK) return st;
    } else if (dc.path == DW_PTILE) {
        st = run_dw_ptile(dc.pt, dtype, x, dy, wsp, fin, s);
        if (st != WTCONV_OK) return st;
    } else if (dc.path == DW_PYRAMID) {
        Plan &pw = dc.p;
        DwPyramidArgs d{};
        d.B = B; d.C = C; d.H = H; d.W = W; d.L = L; d.K = k;
        d.from_level = 1;
        d.nb = pw.a.nb;
        d.x = x; d.dy = dy;
        for (int l = 1; l <= L; ++l) {
            const size_t lb = ((size_t)B * C * (H >> l) * (W >> l) * sizeof(float4) + 255) / 256 * 256;
            d.pyr_x[l] = reinterpret_cast<float4 *>(wsp);
            d.pyr_dy[l] = reinterpret_cast<float4 *>(wsp + lb);
            wsp += 2 * lb;
        }
        d.partials = reinterpret_cast<float *>(wsp);
        if (launch_dw_pyramid(d, dtype, s) != cudaSuccess) return WTCONV_ERR_CUDA;
        fin = pw.a;
        fin.partials = d.partials;
    } else {
        Plan &pw = dc.p;
        pw.a.x = x; pw.a.dy = dy;
        set_params(pw.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
        pw.a.partials = reinterpret_cast<float *>(wsp);
        if (launch_dw(pw.a, dtype, pw.smem, s) != cudaSuccess) return WTCONV_ERR_CUDA;
        fin = pw.a;
    }
    set_params(fin, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
    return cuda_status(launch_dw_finalize(fin, d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale, s));
}

// Backward entry points: planes whose sides are multiples of 2^L go straight to backward_common;
// others are padded into the workspace first (x and dy) and dx is cropped back.
static int backward_entry(bool want_dx, int B, int C, int H, int W, int L, int k, int dtype, const void *x,
                          const void *dy, const float *base_w, const float *base_bias, const float *base_scale,
                          const float *wavelet_w, const float *wavelet_scale, void *dx, float *d_base_w,
                          float *d_base_bias, float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale,
                          void *workspace, size_t workspace_bytes, wtconv_stream_t stream) {
    int st = validate_shape(B, C, H, W, L, k, dtype);
    if (st != WTCONV_OK) return st;
    const PadDims pd = pad_dims(B, C, H, W, L, dtype);
    if (!pd.on)
        return backward_common(want_dx, B, C, H, W, L, k, dtype, x, dy, base_w, base_bias, base_scale, wavelet_w,
                               wavelet_scale, dx, d_base_w, d_base_bias, d_base_scale, d_wavelet_w,
                               d_wavelet_scale, workspace, workspace_bytes, stream);
    if (!aligned16(x) || !aligned16(dy) || (want_dx && !aligned16(dx)) ||
        !params_ok(base_w, base_bias, base_scale, wavelet_w, wavelet_scale) ||
        !params_ok(d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale))
        return WTCONV_ERR_INVALID_ARG;
    if (fault_injected()) return WTCONV_ERR_INJECTED;
    const int op = want_dx ? WTCONV_OP_BACKWARD : WTCONV_OP_BACKWARD_WEIGHTS;
    size_t inner = 0;
    st = workspace_inner(op, B, C, pd.Hp, pd.Wp, L, k, dtype, &inner);
    if (st != WTCONV_OK) return st;
    const size_t bufs = pad_buffers(op) * pd.act_bytes;
    if (workspace_bytes < bufs + inner || !aligned16(workspace)) return WTCONV_ERR_WORKSPACE;
    char *w = static_cast<char *>(workspace);
    char *xp = w, *dyp = w + pd.act_bytes, *dxp = want_dx ? w + 2 * pd.act_bytes : nullptr;
    const int eb = elem_bytes(dtype);
    const long long planes = (long long)B * C;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_pad_planes(x, xp, planes, H, W, pd.Hp, pd.Wp, eb, s) != cudaSuccess ||
        launch_pad_planes(dy, dyp, planes, H, W, pd.Hp, pd.Wp, eb, s) != cudaSuccess)
        return WTCONV_ERR_CUDA;
    st = backward_common(want_dx, B, C, pd.Hp, pd.Wp, L, k, dtype, xp, dyp, base_w, base_bias, base_scale,
                         wavelet_w, wavelet_scale, dxp, d_base_w, d_base_bias, d_base_scale, d_wavelet_w,
                         d_wavelet_scale, w + bufs, workspace_bytes - bufs, stream);
    if (st != WTCONV_OK || !want_dx) return st;
    return cuda_status(launch_crop_planes(dxp, dx, planes, H, W, pd.Hp, pd.Wp, eb, s));
}

int wtconv_backward_weights(int B, int C, int H, int W, int L, int k, int dtype, const void *x, const void *dy,
                            const float *base_w, const float *base_bias, const float *base_scale,
                            const float *wavelet_w, const float *wavelet_scale, float *d_base_w,
                            float *d_base_bias, float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale,
                            void *workspace, size_t workspace_bytes, wtconv_stream_t stream) {
    return backward_entry(false, B, C, H, W, L, k, dtype, x, dy, base_w, base_bias, base_scale, wavelet_w,
                          wavelet_scale, nullptr, d_base_w, d_base_bias, d_base_scale, d_wavelet_w,
                          d_wavelet_scale, workspace, workspace_bytes, stream);
}

int wtconv_backward_weights_noalloc(int B, int C, int H, int W, int L, int k, int dtype, const void *x,
                                    const void *dy, const float *base_w, const float *base_bias,
                                    const float *base_scale, const float *wavelet_w, const float *wavelet_scale,
                                    float *d_base_w, float *d_base_bias, float *d_base_scale, float *d_wavelet_w,
                                    float *d_wavelet_scale, wtconv_stream_t stream) {
    int st = validate_shape(B, C, H, W, L, k, dtype);
    if (st != WTCONV_OK) return st;
    if (!aligned16(x) || !aligned16(dy) || !params_ok(base_w, base_bias, base_scale, wavelet_w, wavelet_scale) ||
        !params_ok(d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale))
        return WTCONV_ERR_INVALID_ARG;
    if (fault_injected()) return WTCONV_ERR_INJECTED;
    if (pad_dims(B, C, H, W, L, dtype).on) return WTCONV_ERR_SCRATCH_LIMIT;  // padded planes need buffers
    // the same kernels as wtconv_backward_weights where they need nothing but the partials
    DwChoice dc = choose_dw(B, C, H, W, L, k, dtype);
    if (dc.status != WTCONV_OK) return dc.status;
    if ((dc.path != DW_FUSED && dc.path != DW_PLANE && dc.path != DW_PAIR) || dc.workspace > sizeof(g_noalloc_scratch))
        return WTCONV_ERR_SCRATCH_LIMIT;
    void *scratch = noalloc_scratch();
    if (scratch == nullptr) return WTCONV_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    LayerArgs fin{};
    if (dc.path == DW_FUSED) {
        st = run_dw_fused(dc.f, dtype, x, dy, static_cast<float *>(scratch), fin, s);
        if (st != WTCONV_OK) return st;
    } else if (dc.path == DW_PAIR) {
        st = run_dw_pair(dc.pr, dtype, x, dy, static_cast<float *>(scratch), fin, s);
        if (st != WTCONV_OK) return st;
    } else {
        Plan &pw = dc.p;
        pw.a.x = x; pw.a.dy = dy;
        set_params(pw.a, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
        pw.a.partials = static_cast<float *>(scratch);
        if (launch_dw(pw.a, dtype, pw.smem, s) != cudaSuccess) return WTCONV_ERR_CUDA;
        fin = pw.a;
    }
    set_params(fin, base_w, base_bias, base_scale, wavelet_w, wavelet_scale);
    return cuda_status(launch_dw_finalize(fin, d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale, s));
}

int wtconv_backward(int B, int C, int H, int W, int L, int k, int dtype, const void *x, const void *dy,
                    const float *base_w, const float *base_bias, const float *base_scale, const float *wavelet_w,
                    const float *wavelet_scale, void *dx, float *d_base_w, float *d_base_bias,
                    float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale, void *workspace,
                    size_t workspace_bytes, wtconv_stream_t stream) {
    return backward_entry(true, B, C, H, W, L, k, dtype, x, dy, base_w, base_bias, base_scale, wavelet_w,
                          wavelet_scale, dx, d_base_w, d_base_bias, d_base_scale, d_wavelet_w, d_wavelet_scale,
                          workspace, workspace_bytes, stream);
}

}  // extern "C"
