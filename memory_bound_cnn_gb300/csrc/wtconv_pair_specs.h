// Shape-specialised instantiations of the batch-pair kernels: for these layer shapes (the
// workload configurations the library is benchmarked on) the pair geometry is a compile-time
// constant, so pitches and offsets are immediates, level loops unroll and index decodes divide by
// constants.  Every other shape runs the same kernels with the plan's geometry at run time.
//
// Each spec: name, H, W, L, K, activation type, dtype code, q0, s0, ql, sl, qd, sd (item shapes as
// in make_pair_geo), then what measured fastest on GB300 for the layer (B = 128 or 64, k = 5):
// the forward's CTA size and pair slots per group (0: the planner's choice), whether the
// batch-pair forward / weight gradient beat the whole-plane kernels there (1) or not (0), and the
// weight gradient's CTA size and item-shape index (planner menu; 6: 7-row items; -1: the
// planner's choice).
//   64x64 L4 bf16: forward 252 vs 316 us (256 threads, 1 pair; 4-column level-1 items: 261 with
//   2-column, 281 with 4-column level 0, 331 with 4 columns everywhere); weight gradient 424 vs 340 us
//   32x32 L3 bf16: forward 127.6 vs 154 us (256 threads, 4 pairs; 4-column level-1 items);
//   weight gradient 191 vs 176 us
//   16x16 L2 bf16: forward 64.1 vs 84.6 us (128 threads, 4 pairs; window rows outside the plane
//   skipped); weight gradient 106 vs 122 us
//   8x8 L1 bf16: forward 43.6 vs 78.5 us (64 threads, 8 pairs; window rows outside the plane
//   skipped); weight gradient 74 vs 134 us
//   28x28 L2 bf16 (14-row output items, 7-row conv items: no rows past the plane): forward
//   60.1 vs 74.4 us (76.4 with 8-row items); weight gradient 76 us with 7-row items on
//   128 threads, against 82.5 on 64 threads, 80 with 8-row items on 128 threads and 94 on the
//   whole-plane kernel
//   56x56 L3 fp32: forward 113 us with 7-row items at levels >= 1 on 256 threads (136 with
//   8-row items) vs 118 on the fused whole-plane kernel, since the last warp builds and
//   convolves level 3 beside levels 1-2 (131 before); weight gradient 167 vs 159 us
#define WTCONV_SPEC_b64l4 b64l4, 64, 64, 4, 5, __nv_bfloat16, 1, 2, 8, 4, 8, 2, 8, 256, 1, 1, 0, 0, -1
#define WTCONV_SPEC_b32l3 b32l3, 32, 32, 3, 5, __nv_bfloat16, 1, 2, 8, 4, 8, 2, 8, 256, 4, 1, 0, 0, -1
#define WTCONV_SPEC_b16l2 b16l2, 16, 16, 2, 5, __nv_bfloat16, 1, 2, 8, 2, 8, 2, 8, 128, 4, 1, 1, 0, -1
#define WTCONV_SPEC_b8l1 b8l1, 8, 8, 1, 5, __nv_bfloat16, 1, 2, 8, 2, 8, 2, 8, 64, 8, 1, 1, 0, -1
#define WTCONV_SPEC_b28l2 b28l2, 28, 28, 2, 5, __nv_bfloat16, 1, 2, 14, 2, 7, 2, 7, 0, 0, 1, 1, 128, 6
#define WTCONV_SPEC_f56l3 f56l3, 56, 56, 3, 5, float, 0, 2, 8, 2, 7, 2, 7, 256, 1, 1, 0, 0, -1

#define WTCONV_PAIR_SPEC_LIST(X)                                                                    \
    X(WTCONV_SPEC_b64l4) X(WTCONV_SPEC_b32l3) X(WTCONV_SPEC_b16l2) X(WTCONV_SPEC_b8l1)             \
    X(WTCONV_SPEC_b28l2) X(WTCONV_SPEC_f56l3)

// M(spec fields...): the spec macro's fields are expanded before M sees them.
#define WTCONV_CALL(M, ...) M(__VA_ARGS__)

// The functions one specialised translation unit defines.
#define WTCONV_PAIR_SPEC_DECL(name, H, W, L, K, T, dt, q0, s0, ql, sl, qd, sd, nt, g, fd, dd, dnt, dsh)                      \
    cudaError_t launch_pair_fwd_spec_##name(const PairArgs &a, size_t smem, cudaStream_t st);       \
    int occupancy_pair_fwd_spec_##name(size_t smem, int nthreads);

#define WTCONV_PAIR_SPEC_DEF(name, H, W, L, K, T, dt, q0, s0, ql, sl, qd, sd, nt, g, fd, dd, dnt, dsh)                       \
    cudaError_t launch_pair_fwd_spec_##name(const PairArgs &a, size_t smem, cudaStream_t st) {      \
        return launch_pair_fwd_t<K, T, PairShapeSpec<H, W, L, q0, s0, ql, sl, qd, sd>>(a, smem, st); \
    }                                                                                               \
    int occupancy_pair_fwd_spec_##name(size_t smem, int nthreads) {                                 \
        return occ_pair_fwd_t<K, T, PairShapeSpec<H, W, L, q0, s0, ql, sl, qd, sd>>(smem, nthreads); \
    }
