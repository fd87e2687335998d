// Device building blocks of the WTConv layer for sm_103a (GB300).
//
// The method (paper "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation", Resumo Tecnico / Metodologia):
//   * on-chip Haar analysis: the 2x2 butterflies of every level are recomputed from one read of
//     the input plane and kept in shared memory; no coefficient tensor reaches HBM;
//   * weight folding: each learned scale is multiplied into its conv kernel (and the base scale
//     into the base bias) when the kernels are staged, so no separate scale pass exists;
//   * closed-form synthesis: output pixel (h, w) gathers sum_l 2^-l sum_s sigma_s Z^l_s[h>>l, w>>l]
//     with sigma_s set by bit l-1 of h (row) and w (column) -- one pass, no cascade buffers.
// Power-of-two factors are moved out of the butterflies: the pyramid is kept unnormalised
// (Yhat^l = 2^l Y^l, exact), so the level-l kernels carry 4^-l.
//
// GB300 specifics.  The k x k depthwise convs are not dense contractions, so they run on the
// FP32 pipe, as packed fma.rn.f32x2 (two lanes of work per issue slot) on pairs of adjacent
// output columns.  Each conv item is a vertical sliding window: 8 output rows x 4 columns, the
// window slides down one input row at a time and every loaded row feeds up to k output rows,
// which keeps shared-memory traffic near 0.35 byte per FMA; the item's k x k kernel sits in
// registers as duplicated pairs.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wtconv_internal.h"

namespace wtconv {

// ------------------------------------------------------------------------ packed fp32 pairs

typedef unsigned long long f2_t;  // low half: first element, high half: second element

__device__ __forceinline__ f2_t pk2(float lo, float hi) {
    f2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float lo2(f2_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo;
}
__device__ __forceinline__ float hi2(f2_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return hi;
}
__device__ __forceinline__ f2_t ffma2(f2_t a, f2_t b, f2_t c) {
    f2_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2_t fadd2(f2_t a, f2_t b) {
    f2_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2_t fsub2(f2_t a, f2_t b) {
    f2_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// acc += a * b, in place (keeps the accumulator in its register pair)
__device__ __forceinline__ void ffma2_acc(f2_t &acc, f2_t a, f2_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ f2_t fmul2(f2_t a, f2_t b) {
    f2_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// (hi(a), lo(b)): the pair that starts one element later across two even pairs
__device__ __forceinline__ f2_t shift1(f2_t a, f2_t b) {
    float a0, a1, b0, b1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(b0), "=f"(b1) : "l"(b));
    return pk2(a1, b0);
}

// ------------------------------------------------------------------ activation element types

template <typename T> struct Act;
template <> struct Act<float> {
    static __device__ __forceinline__ float ld(const float *p) { return *p; }
    static __device__ __forceinline__ void st(float *p, float v) { *p = v; }
    static __device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
    static __device__ __forceinline__ void st8(float *p, const float *v) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    static __device__ __forceinline__ void st4(float *p, const float *v) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Act<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
    static __device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
        uint2 u = *reinterpret_cast<const uint2 *>(p);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    static __device__ __forceinline__ void st8(__nv_bfloat16 *p, const float *v) {
        uint4 u;
        uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 t = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&t);
        }
        *reinterpret_cast<uint4 *>(p) = u;
    }
    static __device__ __forceinline__ void st4(__nv_bfloat16 *p, const float *v) {
        __nv_bfloat162 t0 = __floats2bfloat162_rn(v[0], v[1]), t1 = __floats2bfloat162_rn(v[2], v[3]);
        *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<uint32_t *>(&t0), *reinterpret_cast<uint32_t *>(&t1));
    }
};
template <> struct Act<__half> {
    static __device__ __forceinline__ float ld(const __half *p) { return __half2float(*p); }
    static __device__ __forceinline__ void st(__half *p, float v) { *p = __float2half_rn(v); }
    static __device__ __forceinline__ float4 ld4(const __half *p) {
        uint2 u = *reinterpret_cast<const uint2 *>(p);
        float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
        float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    static __device__ __forceinline__ void st8(__half *p, const float *v) {
        uint4 u;
        uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 t = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&t);
        }
        *reinterpret_cast<uint4 *>(p) = u;
    }
    static __device__ __forceinline__ void st4(__half *p, const float *v) {
        __half2 t0 = __floats2half2_rn(v[0], v[1]), t1 = __floats2half2_rn(v[2], v[3]);
        *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<uint32_t *>(&t0), *reinterpret_cast<uint32_t *>(&t1));
    }
};

// Asynchronous 16-byte global -> shared copies (staging of the next planes).
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// every committed group except the most recent one has completed
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// ------------------------------------------------------------------------------ mbarriers

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(bar)), "r"(count)
                 : "memory");
}
// arrive (release semantics at CTA scope: the caller's earlier shared-memory writes, and those of
// the threads it synchronised with, are visible to a thread whose wait observes the phase)
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"((uint32_t)__cvta_generic_to_shared(bar))
                 : "memory");
}
// Make an mbarrier's initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// Arrive on `bar` and add `bytes` to the transaction count its current phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(bar)),
                 "r"(bytes)
                 : "memory");
}
// Bulk tensor copy (TMA) of one box of a 4-D tensor map into shared memory; completion is
// counted in bytes on `bar`.  Coordinates are element indices, innermost first; parts of the box
// outside the tensor are zero-filled.
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"((uint32_t)__cvta_generic_to_shared(bar))
        : "memory");
}

// One arrival on `bar`, made by the hardware once every cp.async this thread issued before has
// completed (the barrier's expected count must include it: .noinc).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"((uint32_t)__cvta_generic_to_shared(bar))
                 : "memory");
}
// Wait until the phase with parity `parity` has completed.  Bounded by elapsed time: after
// kMaxWaitNs of %globaltimer time (half a second; a copy or handshake that takes that long is
// broken, not slow) it raises *timeout (if given) and returns false.  Each try suspends the thread
// for at most kWaitHintNs; kMaxWaitTries is only a backstop should the timer not advance.
constexpr uint64_t kMaxWaitNs = 500000000ull;
constexpr uint32_t kMaxWaitTries = 1u << 24;
constexpr uint32_t kWaitHintNs = 1000;
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *timeout) {
    const uint32_t addr = (uint32_t)__cvta_generic_to_shared(bar);
    uint64_t t0 = 0;
    for (uint32_t i = 0; i < kMaxWaitTries; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(parity), "n"(kWaitHintNs)
            : "memory");
        if (done) return true;
        if ((i & 15) == 0) {
            const uint64_t now = global_ns();
            if (i == 0) t0 = now;
            else if (now - t0 > kMaxWaitNs) break;
        }
    }
    if (timeout) atomicExch(timeout, 1);
    return false;
}

// Copy the raw planes b0 .. b0+G-1 of channel c (those that exist) to the staging area.
template <typename T>
__device__ __forceinline__ void stage_planes(const T *src, T *stg, int B, int C, int c, int b0, int G, size_t HW,
                                             const FastDiv &dn) {
    const int nch = (int)dn.d;
    for (int it = threadIdx.x; it < G * nch; it += blockDim.x) {
        const int g = fdiv(dn, it), ch = it - g * nch;
        const int b = b0 + g;
        if (b < B)
            cp_async16(reinterpret_cast<char *>(stg + g * HW) + 16 * ch,
                       reinterpret_cast<const char *>(src + ((size_t)b * C + c) * HW) + 16 * ch);
    }
}

// Start pulling the next planes into L2 while the current ones are computed.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------------ weight staging

// Stage channel c's kernels into shared memory as packed pairs, scales folded in.  Conv image
// ci = 0 is the base kernel, stored duplicated {w, w} (it pairs two output columns); conv image
// ci = 1 + 2(l-1) + pp holds level l's subbands 2pp and 2pp+1 side by side {w_2pp, w_2pp+1}
// (it pairs the two subbands of a pair image):
//   base            : s_b[c] * w_b[c]
//   level l, subband s: 4^-l * s_l[4c+s] * w_l[4c+s]      (4^-l: unnormalised pyramid)
// `flip` rotates every kernel by 180 degrees (the transposed conv of the input gradient).
template <int K>
__device__ __forceinline__ void stage_weights(const LayerArgs &a, int c, f2_t *wts) {
    constexpr int KK = K * K, WP = wpairs(K);
    const int nimg = 1 + 2 * a.L;
    for (int it = threadIdx.x; it < nimg * KK; it += blockDim.x) {
        const int ci = it / KK, t = it - ci * KK;
        const int tu = t / K, tv = t - tu * K;
        const int src_t = a.flip ? (K - 1 - tu) * K + (K - 1 - tv) : t;
        float v0, v1;
        if (ci == 0) {
            v0 = v1 = a.base_scale[c] * a.base_w[(size_t)c * KK + src_t];
        } else {
            const int l = (ci - 1) / 2 + 1, pp = (ci - 1) & 1;
            const size_t ch = (size_t)(l - 1) * 4 * a.C + 4 * c + 2 * pp;
            v0 = ldexpf(a.wavelet_scale[ch] * a.wavelet_w[ch * KK + src_t], -2 * l);
            v1 = ldexpf(a.wavelet_scale[ch + 1] * a.wavelet_w[(ch + 1) * KK + src_t], -2 * l);
        }
        wts[ci * WP + t] = pk2(v0, v1);
    }
}

template <int K>
__device__ __forceinline__ void load_weights(const f2_t *wsig, f2_t (&w)[K * K]) {
    const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(wsig);
#pragma unroll
    for (int i = 0; i < K * K / 2; ++i) {
        ulonglong2 t = p[i];
        w[2 * i] = t.x;
        w[2 * i + 1] = t.y;
    }
    if constexpr ((K * K) & 1) w[K * K - 1] = wsig[K * K - 1];
}

// -------------------------------------------------------------- sliding-window conv item

// Loads one window row: columns c .. c + 4*NV - 1 of a shared row as even pairs, plus the odd
// (one-element-shifted) pairs.
template <int NV>
__device__ __forceinline__ void load_row(const float *p, f2_t (&e)[2 * NV], f2_t (&o)[2 * NV - 1]) {
    const ulonglong2 *q = reinterpret_cast<const ulonglong2 *>(p);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        ulonglong2 t = q[i];
        e[2 * i] = t.x;
        e[2 * i + 1] = t.y;
    }
#pragma unroll
    for (int i = 0; i < 2 * NV - 1; ++i) o[i] = shift1(e[i], e[i + 1]);
}

// One base conv item: out[r][c] = init + sum_{u,v} w[u][v] * in[r + u][c + v] for r < kRows, c < kCols, where
// `in` points at the padded window origin (= output interior origin) and `out` at the compact
// output.  Weights w are duplicated pairs in registers.  The tap loop runs v-major so that
// consecutive FMAs update different accumulators (rows in flight x column pairs).
template <int K>
__device__ __forceinline__ void conv_item(const float *__restrict__ in, int pitch, const f2_t (&w)[K * K],
                                          float *__restrict__ out, int opitch, f2_t init) {
    constexpr int NV = (kCols + K - 1 + 3) / 4;  // 16-byte loads per window row
    f2_t acc[kRows][2];
#pragma unroll
    for (int i = 0; i < kRows + K - 1; ++i) {
        f2_t e[2 * NV], o[2 * NV - 1];
        load_row<NV>(in + i * pitch, e, o);
#pragma unroll
        for (int v = 0; v < K; ++v) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < kRows) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const f2_t xv = (v & 1) ? o[q + v / 2] : e[q + v / 2];
                        if (u == 0 && v == 0) acc[j][q] = ffma2(w[0], xv, init);
                        else ffma2_acc(acc[j][q], w[u * K + v], xv);
                    }
                }
            }
        }
        const int jd = i - (K - 1);  // output row jd is complete
        if (jd >= 0) {
            ulonglong2 t;
            t.x = acc[jd][0];
            t.y = acc[jd][1];
            *reinterpret_cast<ulonglong2 *>(out + jd * opitch) = t;
        }
    }
}

// One weight-gradient item: acc[u*K+v] (pairs of partial sums) += sum over the kRows x kCols
// interior tile at g of G[r][c] * Ypad[r + u][c + v]; `y` points at the padded window origin of
// the tile, `g` at its interior origin (both in padded buffers of the same pitch).  The loop runs
// column-pair-major so that consecutive FMAs update different taps.
template <int K>
__device__ __forceinline__ void dw_item(const float *__restrict__ y, const float *__restrict__ g, int pitch,
                                        f2_t (&acc)[K * K]) {
    constexpr int NV = (kCols + K - 1 + 3) / 4;
    f2_t gr[kRows][2];
#pragma unroll
    for (int i = 0; i < kRows + K - 1; ++i) {
        if (i < kRows) {
            if constexpr (((K / 2) & 1) == 0) {
                const f2_t *gp = reinterpret_cast<const f2_t *>(g + i * pitch);  // 8-byte aligned (P even)
                gr[i][0] = gp[0];
                gr[i][1] = gp[1];
            } else {
                const float *gf = g + i * pitch;
                gr[i][0] = pk2(gf[0], gf[1]);
                gr[i][1] = pk2(gf[2], gf[3]);
            }
        }
        f2_t e[2 * NV], o[2 * NV - 1];
        load_row<NV>(y + i * pitch, e, o);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < kRows) {
#pragma unroll
                    for (int v = 0; v < K; ++v) {
                        const f2_t xv = (v & 1) ? o[q + v / 2] : e[q + v / 2];
                        ffma2_acc(acc[u * K + v], gr[j][q], xv);
                    }
                }
            }
        }
    }
}

// -------------------------------------------------------- subband-pair items (levels >= 1)

// Window row of a pair image: positions 0 .. 2*NV-1 (each a packed pair of subbands).
template <int NV>
__device__ __forceinline__ void load_pair_row(const float *p, f2_t (&x)[2 * NV]) {
    const ulonglong2 *q = reinterpret_cast<const ulonglong2 *>(p);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const ulonglong2 t = q[i];
        x[2 * i] = t.x;
        x[2 * i + 1] = t.y;
    }
}

// Conv item on a subband-pair image: for kRows x kColsL output positions,
// out[r][c] = sum_{u,v} w[u][v] * in[r + u][c + v] elementwise on the two subbands; `in` points at
// the padded window origin, `out` at the compact pair output; pitches in positions.
template <int K>
__device__ __forceinline__ void conv_item_pair(const float *__restrict__ in, int pitch, const f2_t (&w)[K * K],
                                               float *__restrict__ out, int opitch) {
    constexpr int NV = (kColsL + K - 1 + 1) / 2;  // 16-byte loads (two positions each) per window row
    f2_t acc[kRows][kColsL];
#pragma unroll
    for (int i = 0; i < kRows + K - 1; ++i) {
        f2_t x[2 * NV];
        load_pair_row<NV>(in + 2 * i * pitch, x);
#pragma unroll
        for (int v = 0; v < K; ++v) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < kRows) {
#pragma unroll
                    for (int q = 0; q < kColsL; ++q) {
                        if (u == 0 && v == 0) acc[j][q] = fmul2(w[0], x[q]);
                        else ffma2_acc(acc[j][q], w[u * K + v], x[q + v]);
                    }
                }
            }
        }
        const int jd = i - (K - 1);
        if (jd >= 0) {
            ulonglong2 t;
            t.x = acc[jd][0];
            t.y = acc[jd][1];
            *reinterpret_cast<ulonglong2 *>(out + 2 * jd * opitch) = t;
        }
    }
}

// Weight-gradient item on subband-pair images: acc[u*K+v] = (dW_s0[u][v], dW_s1[u][v]) +=
// sum over the kRows x kColsL interior tile of G[r][c] * Ypad[r + u][c + v] (elementwise on the
// pair); `y` points at the padded window origin, `g` at the tile's interior origin (same pitch).
template <int K>
__device__ __forceinline__ void dw_item_pair(const float *__restrict__ y, const float *__restrict__ g, int pitch,
                                             f2_t (&acc)[K * K]) {
    constexpr int NV = (kColsL + K - 1 + 1) / 2;
    f2_t gr[kRows][kColsL];
#pragma unroll
    for (int i = 0; i < kRows + K - 1; ++i) {
        if (i < kRows) {
            const f2_t *gp = reinterpret_cast<const f2_t *>(g + 2 * i * pitch);
            gr[i][0] = gp[0];
            gr[i][1] = gp[1];
        }
        f2_t x[2 * NV];
        load_pair_row<NV>(y + 2 * i * pitch, x);
#pragma unroll
        for (int q = 0; q < kColsL; ++q) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int j = i - u;
                if (j >= 0 && j < kRows) {
#pragma unroll
                    for (int v = 0; v < K; ++v) ffma2_acc(acc[u * K + v], gr[j][q], x[q + v]);
                }
            }
        }
    }
}

// ------------------------------------------------------------------------- Haar analysis

// Unnormalised 2x2 butterfly of the block [[a, b], [c, d]]:
// LL = a+b+c+d, LH = a-b+c-d, HL = a+b-c-d, HH = a-b-c+d (signs of the page-4 filters).
struct Quad { float ll, lh, hl, hh; };
__device__ __forceinline__ Quad butterfly(float a, float b, float c, float d) {
    const float st = a + b, dt = a - b, sb = c + d, db = c - d;
    return {st + sb, dt + db, st - sb, dt - db};
}

// Store a subband quad at interior position (i, j) of level l's four padded subband images.
__device__ __forceinline__ void put_quad(float *base, int sub, int idx, const Quad &q) {
    base[idx] = q.ll;
    base[sub + idx] = q.lh;
    base[2 * sub + idx] = q.hl;
    base[3 * sub + idx] = q.hh;
}

}  // namespace wtconv
