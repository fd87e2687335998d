/*
 * wtconv.h -- C ABI of the GB300 (sm_103a) WTConv layer library (libwtconv.so).
 *
 * The layer (paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
 * Reformulation", arXiv 2608.10805; its technical summary "Resumo Tecnico", sections Problema
 * and Metodologia) maps an input x of shape (B, C, H, W) to
 *
 *     y = s_b * (conv_k(x, w_b) + b_b)                                      base path
 *       + sum_{l=1..L} Synth_l( s_l * conv_k(Analysis_l(x), w_l) )           wavelet path
 *
 * where Analysis_l is the l-level orthonormal 2-D Haar decomposition (LL, LH, HL, HH subbands of
 * the low band of level l-1), conv_k is a depthwise k x k cross-correlation with zero 'same'
 * padding at each level's resolution, s_l a learned scale per subband channel, and Synth_l the
 * inverse cascade.  The library evaluates it the paper's I/O-aware way: the Haar butterflies are
 * recomputed on chip from one read of x, scales are folded into the conv weights, and the
 * synthesis is the closed form in which output pixel (h, w) gathers its level-l terms at
 * (h >> l, w >> l) with signs set by bit l-1 of h and w.  The backward applies the same
 * reformulation in transpose.
 *
 * Conventions shared by every entry point:
 *   - B, C, H, W > 0; 1 <= L <= WTCONV_MAX_LEVELS; k odd, 1 <= k <= 7 (k in {3, 5, 7} run;
 *     other odd k return WTCONV_ERR_UNSUPPORTED); B*C < 2^31 and Hp*Wp <= 2^30, where Hp, Wp
 *     are H, W rounded up to multiples of 2^L.
 *   - Sides that are not multiples of 2^L: a level whose input has an odd side pads it with one
 *     zero row / column at its end before the analysis (the stride-2 'SAME' Haar conv of the
 *     page-4 snippet), and the synthesis crops that level's reconstruction back to the input's
 *     size.  That equals the layer on the plane zero-padded at its end to Hp x Wp, cropped back
 *     to H x W, which is how it runs: the activations are padded into the workspace (one
 *     Hp x Wp tensor per activation the call reads or writes), and the results cropped out.
 *   - dtype (WTCONV_F32 / WTCONV_BF16 / WTCONV_F16) is the type of the activations x, y, dy,
 *     dx.  Parameters and parameter gradients are always fp32; all arithmetic is fp32 with
 *     round-to-nearest-even on the final store of a bf16 / fp16 activation.
 *   - Layouts are contiguous row-major: x, y, dy, dx [B][C][H][W]; base_w [C][k][k];
 *     base_bias, base_scale [C]; wavelet_w [L][4C][k][k]; wavelet_scale [L][4C], where subband
 *     channel 4c+s holds subband s (0 LL, 1 LH, 2 HL, 3 HH) of input channel c at that level.
 *   - Every pointer is caller-owned DEVICE memory (cudaMalloc or an allocator on top of it).
 *     Activation pointers and the workspace must be 16-byte aligned, parameter and gradient
 *     pointers 4-byte aligned.  The library allocates no device memory; scratch is the
 *     caller's `workspace` of at least wtconv_workspace_size(...) bytes (may be NULL when that
 *     size is 0).  Inputs are never written.  Outputs are fully overwritten (gradients are
 *     not accumulated into).
 *   - Calls are asynchronous on `stream` (NULL: the legacy default stream) and never
 *     synchronise.  Arguments are validated on the host before anything is launched: on any
 *     error no kernel runs and no output is touched.  Faults in a launched kernel surface at
 *     the caller's next synchronisation, as with any CUDA launch.
 *   - No state carries results from one call to the next (the library caches per-shape launch
 *     plans on the host, per device); concurrent calls on different streams with distinct
 *     workspaces are safe.
 *   - The forward and the input gradient run one of five kernel sets: the batch-pair kernel
 *     (two batch entries per packed fp32 pair, whole pyramids of several pairs on chip; small
 *     planes), the fused whole-plane kernel (fp32 planes where it is fastest), the whole-plane
 *     kernel (planes whose pyramid fits in shared memory), or, on larger planes, the deep kernel
 *     (levels >= 2 at level-1 resolution, into the workspace) followed by a tiled shallow kernel:
 *     the batch-pair one (tiles of x with halo and of the deep part by bulk tensor copies; planes
 *     whose rows are a multiple of 16 bytes and of 8 elements) or else the one-warp one.
 *     WTCONV_FWD_PATH=pair, =fused, =plane, =ptile or =tiles selects a set where it applies (same
 *     results within fp32 rounding); WTCONV_PAIR=0 / =1 keeps the batch-pair kernels off / makes
 *     them the default wherever they apply.
 *   - The weight gradients run the batch-pair kernel on small planes, else the fused
 *     whole-plane kernel (x and dy planes moved by bulk tensor copies, both pyramids on chip; fp32
 *     planes of at least 64 base items where both copies fit one box of at most 256 x 256), else a
 *     staged whole-plane kernel where both planes' pyramids fit in shared memory, else the tiled
 *     batch-pair kernel (tiles of x with halo and of dy by bulk tensor copies, two Haar levels per
 *     launch, deeper levels from the level-2 low bands the previous launch writes), else older
 *     tiled kernels (levels >= 2 on their pyramids in the workspace), else workspace pyramids for
 *     every level.  WTCONV_DW_PATH=pair, =fused, =plane, =ptile, =tiles or =pyramid selects a path
 *     where it applies (same results within fp32 rounding).
 *   - Tuning restrictions for measurement runs (the plans they give are valid, only slower or
 *     faster): WTCONV_PAIR_THREADS, WTCONV_PAIR_SHAPE and WTCONV_PAIR_SLOTS fix the batch-pair
 *     kernels' CTA size, item shapes and pair slots per group; WTCONV_PAIR_CHUNK fixes the
 *     batch-pair weight gradient's slot groups per work unit; WTCONV_PAIR_SPLIT=0 keeps every
 *     warp of the batch-pair forward on every level (by default, with L >= 3, the last warp builds
 *     and convolves levels >= 3 while the others convolve levels 1 and 2); WTCONV_PAIR_TMAP=0
 *     brings a group's planes by one bulk copy per plane instead of one tensor copy per input; WTCONV_PTILE=TH,TW,G,threads[,narrow]
 *     fixes the first tiled batch-pair weight-gradient launch's tile, pair slots, CTA size and
 *     item width; WTCONV_PSHALLOW=TH,TW,G,threads[,rows] fixes the tiled batch-pair shallow
 *     kernel's tile, pair slots, CTA size and item rows;
 *     WTCONV_STAGED=G,threads fixes the planes per slot group and CTA size of the whole-plane and
 *     deep kernels.
 *   - Setting the environment variable WTCONV_INJECT_FAULT=1 makes every compute entry point
 *     return WTCONV_ERR_INJECTED before launching anything (host-side fault injection).
 */
#ifndef WTCONV_H
#define WTCONV_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object type as cudaStream_t / CUstream; declared here so this header needs no CUDA
 * header. */
typedef struct CUstream_st *wtconv_stream_t;

enum wtconv_dtype { WTCONV_F32 = 0, WTCONV_BF16 = 1, WTCONV_F16 = 2 };

enum wtconv_status {
    WTCONV_OK = 0,
    WTCONV_ERR_INVALID_ARG = 1, /* bad shape, null or misaligned pointer */
    WTCONV_ERR_UNSUPPORTED = 2, /* valid but not built: dtype, k, or a plane too large */
    WTCONV_ERR_WORKSPACE = 3,   /* workspace smaller than wtconv_workspace_size() */
    WTCONV_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    WTCONV_ERR_INJECTED = 5,    /* WTCONV_INJECT_FAULT is set */
    WTCONV_ERR_SCRATCH_LIMIT = 6, /* shape needs more than WTCONV_NOALLOC_SCRATCH_BYTES of scratch */
    WTCONV_ERR_DEVICE_TIMEOUT = 7 /* a kernel's bounded wait gave up (wtconv_device_status) */
};

/* Operation selector for wtconv_workspace_size. */
enum wtconv_op {
    WTCONV_OP_FORWARD = 0,
    WTCONV_OP_BACKWARD_INPUT = 1,
    WTCONV_OP_BACKWARD_WEIGHTS = 2,
    WTCONV_OP_BACKWARD = 3
};

#define WTCONV_MAX_LEVELS 5

/* Library version, major * 10000 + minor * 100 + patch. */
int wtconv_version(void);

/* Human-readable name of a status code (static storage; never NULL). */
const char *wtconv_strerror(int status);

/* Device-side status of the calls made so far on the current device.  Kernels that wait for
 * their input copies (or hand work between warps) on shared-memory barriers wait at most half a
 * second of elapsed time; a wait that gives up (never expected: it would mean a broken copy or
 * handshake, not a slow GPU) raises a sticky per-device flag and ends its CTA.  The forward and
 * input-gradient outputs of that CTA stay unwritten and the weight gradients it contributes to
 * come out as NaN.  The compute calls themselves cannot report this (they return at launch):
 * a caller that must know its results are valid polls this function after synchronising.  It
 * synchronises the device, returns WTCONV_ERR_DEVICE_TIMEOUT if the flag was raised (and clears
 * it), WTCONV_ERR_CUDA if the synchronisation or the read failed, else WTCONV_OK. */
int wtconv_device_status(void);

/* Diagnostic of the failure path above, with no fault: launches one kernel on `stream` whose
 * single waiting thread waits on a shared-memory barrier that nothing ever completes.  The wait
 * gives up after half a second and raises the flag, so the next wtconv_device_status() returns
 * WTCONV_ERR_DEVICE_TIMEOUT (and clears it).  Returns WTCONV_OK once launched, WTCONV_ERR_CUDA if
 * the launch failed. */
int wtconv_selftest_wait_timeout(wtconv_stream_t stream);

/* Diagnostic: the packed-FMA (fma.rn.f32x2) throughput of the current device in TFLOP/s, the
 * ceiling of the layer's conv arithmetic and the denominator of its ALU roofline.  Runs
 * independent FMA chains of `iters` steps in 8 CTAs of 256 threads per SM on the legacy default
 * stream, timed with CUDA events; synchronises the device.  Writes *tflops; returns WTCONV_OK,
 * WTCONV_ERR_INVALID_ARG (iters <= 0 or tflops NULL) or WTCONV_ERR_CUDA. */
int wtconv_fp32_fma_peak(int iters, double *tflops);

/* Bytes of device workspace `op` needs for this shape on the current device (0 if none).
 * FORWARD and BACKWARD_INPUT need, for L >= 2, one fp32 per level-1 position
 * (B*C*(H/2)*(W/2)*4 bytes, rounded up to 256): the contribution of the Haar levels >= 2, which a
 * first kernel computes per plane and the second kernel adds to every output pixel.  The weight
 * gradients need one fp32 partial per (CTA, channel, subband, tap), and for planes too large
 * for the whole-plane kernels with L >= 3 also the level-2 (and level-4) low bands of x and dy as
 * fp32 planes (2 * B*C*(H/4)*(W/4 rounded up to 4)*4 bytes, then the same for H/16, W/16);
 * BACKWARD needs both.
 * Sides that are not multiples of 2^L add the padded activations (each B*C*Hp*Wp elements,
 * rounded up to 256 bytes): two for FORWARD, BACKWARD_INPUT and BACKWARD_WEIGHTS, three for
 * BACKWARD.
 * Returns 0 for an invalid shape as well; the compute call then reports the error. */
size_t wtconv_workspace_size(int op, int B, int C, int H, int W, int L, int k, int dtype);

/* Names of the kernels `op` launches for this shape on the current device, joined by '+', in
 * launch order ("" for an invalid or unsupported shape).  Static storage; never NULL. */
const char *wtconv_plan_kernels(int op, int B, int C, int H, int W, int L, int k, int dtype);

/* Number of kernel launches `op` makes for this shape on the current device (0 for an invalid
 * or unsupported shape).  Planes whose Haar pyramid fits in shared memory take one launch for
 * the forward and the input gradient and two for the weight gradients (correlations +
 * finalize); larger planes take two for the forward / input gradient (levels >= 2, then the
 * base conv and level 1; one when L = 1) and, for the weight gradients, one tiled launch per two Haar levels
 * plus the finalize (ceil(L / 2) + 1; with WTCONV_DW_PATH=tiles the older tiled chain, 2L + 2).
 * BACKWARD is the sum of BACKWARD_INPUT and BACKWARD_WEIGHTS.  Sides that are not multiples of
 * 2^L add the pads and the crop: two launches for FORWARD, BACKWARD_INPUT and
 * BACKWARD_WEIGHTS, three for BACKWARD. */
int wtconv_launch_count(int op, int B, int C, int H, int W, int L, int k, int dtype);

/* Forward pass (Metodologia: fused on-chip Haar analysis, folded scales, closed-form
 * synthesis).  Writes y [B][C][H][W]. */
int wtconv_forward(int B, int C, int H, int W, int L, int k, int dtype, const void *x,
                   const float *base_w, const float *base_bias, const float *base_scale,
                   const float *wavelet_w, const float *wavelet_scale, void *y, void *workspace,
                   size_t workspace_bytes, wtconv_stream_t stream);

/* Gradient with respect to the input (gist.science pt, Resumo Tecnico / Resultados: the timed
 * training step is forward plus backward; Metodologia: the reformulation leaves the operator
 * unchanged, so its transpose is the same three reformulations run in reverse roles):
 * dx = sum_l Synth_l(s_l * corr(Analysis_l(dy), flip(w_l))) + s_b * corr(dy, flip(w_b)), the
 * transpose of the forward's linear part (the bias drops out), computed by the forward's kernels
 * on dy with every kernel rotated by 180 degrees.  Reads dy, writes dx, both [B][C][H][W]. */
int wtconv_backward_input(int B, int C, int H, int W, int L, int k, int dtype,
                          const float *base_w, const float *base_bias, const float *base_scale,
                          const float *wavelet_w, const float *wavelet_scale, const void *dy,
                          void *dx, void *workspace, size_t workspace_bytes,
                          wtconv_stream_t stream);

/* Gradients of every parameter (Contribuicoes: "all parameter gradients") from x and dy.
 * Writes d_base_w [C][k][k], d_base_bias [C], d_base_scale [C], d_wavelet_w [L][4C][k][k],
 * d_wavelet_scale [L][4C].  Deterministic: the reduction order is fixed for a given device and
 * shape. */
int wtconv_backward_weights(int B, int C, int H, int W, int L, int k, int dtype, const void *x,
                            const void *dy, const float *base_w, const float *base_bias,
                            const float *base_scale, const float *wavelet_w,
                            const float *wavelet_scale, float *d_base_w, float *d_base_bias,
                            float *d_base_scale, float *d_wavelet_w, float *d_wavelet_scale,
                            void *workspace, size_t workspace_bytes, wtconv_stream_t stream);

/* Whole backward in one call (gist.science pt, Resumo Tecnico / Principais Contribuicoes: the
 * reformulated layer is validated on the forward outputs and on all parameter gradients;
 * Resultados: a training step is forward plus backward): dx and every parameter gradient.  It
 * launches the input gradient's kernels and then the weight gradients' on `stream` (each reads
 * dy), with one workspace for both.  Same results as wtconv_backward_input followed by
 * wtconv_backward_weights. */
int wtconv_backward(int B, int C, int H, int W, int L, int k, int dtype, const void *x,
                    const void *dy, const float *base_w, const float *base_bias,
                    const float *base_scale, const float *wavelet_w, const float *wavelet_scale,
                    void *dx, float *d_base_w, float *d_base_bias, float *d_base_scale,
                    float *d_wavelet_w, float *d_wavelet_scale, void *workspace,
                    size_t workspace_bytes, wtconv_stream_t stream);

/* Size of the fixed device scratch behind wtconv_backward_weights_noalloc: 4 MiB per device. */
#define WTCONV_NOALLOC_SCRATCH_BYTES (4u << 20)

/* wtconv_backward_weights without a workspace argument.  The pages describe no such call: it is
 * an addition of this library, for callers that cannot hand it device memory.  Examples are a
 * plain C host program that has no device allocator of its own, a plug-in whose host framework
 * owns all device memory and lends none, and a training step whose memory was budgeted in full
 * beforehand, where a late allocation could fail or stall on the allocator.
 *
 * The per-CTA partial sums of the weight-gradient reduction go to a scratch array that is
 * compiled into the library (WTCONV_NOALLOC_SCRATCH_BYTES bytes of device memory per device,
 * reserved when the library's device code is loaded).  This call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *   - Set-up: the first call on a device, with that device current, looks up the scratch
 *     address (cudaGetSymbolAddress) and plans the shape; later calls reuse both.  Make that
 *     first call for each device and shape before any stream capture begins.
 *   - Limit: if this shape needs more scratch than WTCONV_NOALLOC_SCRATCH_BYTES (many channels
 *     and levels, planes too large for the whole-plane kernel, which need their Haar pyramids
 *     in scratch, or sides that are not multiples of 2^L, which need padded copies of x and
 *     dy), the call returns WTCONV_ERR_SCRATCH_LIMIT and launches nothing; use
 *     wtconv_backward_weights with a workspace then.
 *   - Nothing in the scratch has to start at zero: every partial is written before it is read.
 *   - The scratch is shared by every call on the device.  Calls whose execution overlaps (on
 *     different streams, or issued from different host threads without ordering) race on it
 *     and give wrong gradients; calls ordered on one stream are safe.
 * Arguments, outputs and the other status codes are those of wtconv_backward_weights, whose
 * kernels this call runs; the results equal that call's for the same device and shape. */
int wtconv_backward_weights_noalloc(int B, int C, int H, int W, int L, int k, int dtype,
                                    const void *x, const void *dy, const float *base_w,
                                    const float *base_bias, const float *base_scale,
                                    const float *wavelet_w, const float *wavelet_scale,
                                    float *d_base_w, float *d_base_bias, float *d_base_scale,
                                    float *d_wavelet_w, float *d_wavelet_scale,
                                    wtconv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* WTCONV_H */
