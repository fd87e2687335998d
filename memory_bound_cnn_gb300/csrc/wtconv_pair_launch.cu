// Host side of the batch-pair kernels: shared-memory sizes, and the dispatch on the activation
// type to the per-type translation units.
#include "wtconv_pair_dw.cuh"
#include "wtconv_pair_fwd.cuh"
#include "wtconv_pair_specs.h"
#include "wtconv_pshallow.cuh"
#include "wtconv_ptile_dw.cuh"

namespace wtconv {

#define WTCONV_DECL_ONE(spec) WTCONV_CALL(WTCONV_PAIR_SPEC_DECL, spec)
WTCONV_PAIR_SPEC_LIST(WTCONV_DECL_ONE)

namespace {

struct PairSpecEntry {
    int H, W, L, K, dtype, shape[6];
    int fwd_threads, fwd_slots, fwd_default, dw_default, dw_threads, dw_shape;
    cudaError_t (*launch_fwd)(const PairArgs &, size_t, cudaStream_t);
    int (*occ_fwd)(size_t, int);
};

#define WTCONV_ENTRY(name, H, W, L, K, T, dt, q0, s0, ql, sl, qd, sd, nt, g, fd, dd, dnt, dsh)        \
    {H, W, L, K, dt, {q0, s0, ql, sl, qd, sd}, nt, g, fd, dd, dnt, dsh, launch_pair_fwd_spec_##name, \
     occupancy_pair_fwd_spec_##name},
#define WTCONV_ENTRY_ONE(spec) WTCONV_CALL(WTCONV_ENTRY, spec)
const PairSpecEntry kSpecs[] = {WTCONV_PAIR_SPEC_LIST(WTCONV_ENTRY_ONE)};

}  // namespace

int pair_spec_index(int H, int W, int L, int K, int dtype, const int (&shape)[6]) {
    for (int i = 0; i < (int)(sizeof(kSpecs) / sizeof(kSpecs[0])); ++i) {
        const PairSpecEntry &e = kSpecs[i];
        if (e.H == H && e.W == W && e.L == L && e.K == K && e.dtype == dtype) {
            bool same = true;
            for (int j = 0; j < 6; ++j) same = same && e.shape[j] == shape[j];
            if (same) return i;
        }
    }
    return -1;
}

int occupancy_pair_fwd_spec(int spec, size_t smem, int nthreads) { return kSpecs[spec].occ_fwd(smem, nthreads); }

bool pair_spec_measured(int H, int W, int L, int K, int dtype, PairSpecPref *pref) {
    for (const PairSpecEntry &e : kSpecs) {
        if (e.H == H && e.W == W && e.L == L && e.K == K && e.dtype == dtype) {
            for (int j = 0; j < 6; ++j) pref->shape[j] = e.shape[j];
            pref->threads = e.fwd_threads;
            pref->slots = e.fwd_slots;
            pref->fwd_default = e.fwd_default;
            pref->dw_default = e.dw_default;
            pref->dw_threads = e.dw_threads;
            pref->dw_shape = e.dw_shape;
            return true;
        }
    }
    return false;
}

size_t pair_fwd_smem_bytes(const PairArgs &a, int elem_bytes) {
    (void)elem_bytes;
    return pair_fwd_layout(a).total;
}

size_t pair_dw_smem_bytes(const PairArgs &a, int elem_bytes) {
    (void)elem_bytes;
    return pair_dw_layout(a).total;
}

cudaError_t launch_pair_fwd(const PairArgs &a, int dtype, size_t smem, cudaStream_t st) {
    if (a.spec >= 0) return kSpecs[a.spec].launch_fwd(a, smem, st);
    switch (dtype) {
    case 0: return launch_pair_fwd_typed<float>(a, smem, st);
    case 1: return launch_pair_fwd_typed<__nv_bfloat16>(a, smem, st);
    case 2: return launch_pair_fwd_typed<__half>(a, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

int occupancy_pair_fwd(int dtype, int K, size_t smem, int nthreads) {
    switch (dtype) {
    case 0: return occupancy_pair_fwd_typed<float>(K, smem, nthreads);
    case 1: return occupancy_pair_fwd_typed<__nv_bfloat16>(K, smem, nthreads);
    case 2: return occupancy_pair_fwd_typed<__half>(K, smem, nthreads);
    default: return 0;
    }
}

cudaError_t launch_pair_dw(const PairArgs &a, int dtype, size_t smem, cudaStream_t st) {
    switch (dtype) {
    case 0: return launch_pair_dw_typed<float>(a, smem, st);
    case 1: return launch_pair_dw_typed<__nv_bfloat16>(a, smem, st);
    case 2: return launch_pair_dw_typed<__half>(a, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

int occupancy_pair_dw(int dtype, int K, size_t smem, int nthreads) {
    switch (dtype) {
    case 0: return occupancy_pair_dw_typed<float>(K, smem, nthreads);
    case 1: return occupancy_pair_dw_typed<__nv_bfloat16>(K, smem, nthreads);
    case 2: return occupancy_pair_dw_typed<__half>(K, smem, nthreads);
    default: return 0;
    }
}

// ---------------------------------------------------------------- tiled batch-pair weight gradient

cudaError_t launch_ptile_dw_f32(const PtileArgs &a, size_t smem, cudaStream_t st);
cudaError_t launch_ptile_dw_bf16(const PtileArgs &a, size_t smem, cudaStream_t st);
cudaError_t launch_ptile_dw_f16(const PtileArgs &a, size_t smem, cudaStream_t st);
int occupancy_ptile_dw_f32(int K, int LT, int base, size_t smem, int nthreads, int iq);
int occupancy_ptile_dw_bf16(int K, int LT, int base, size_t smem, int nthreads, int iq);
int occupancy_ptile_dw_f16(int K, int LT, int base, size_t smem, int nthreads, int iq);

size_t ptile_smem_bytes(const PtileArgs &a, int elem_bytes) {
    (void)elem_bytes;  // the raw tile sizes already count the element size
    return ptile_layout(a).total;
}

cudaError_t launch_ptile_dw(const PtileArgs &a, int dtype, size_t smem, cudaStream_t st) {
    switch (dtype) {
    case 0: return launch_ptile_dw_f32(a, smem, st);
    case 1: return launch_ptile_dw_bf16(a, smem, st);
    case 2: return launch_ptile_dw_f16(a, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

int occupancy_ptile_dw(int dtype, int K, int LT, int base, size_t smem, int nthreads, int iq) {
    switch (dtype) {
    case 0: return occupancy_ptile_dw_f32(K, LT, base, smem, nthreads, iq);
    case 1: return occupancy_ptile_dw_bf16(K, LT, base, smem, nthreads, iq);
    case 2: return occupancy_ptile_dw_f16(K, LT, base, smem, nthreads, iq);
    default: return 0;
    }
}

// ---------------------------------------------------------------- tiled batch-pair shallow kernel

cudaError_t launch_pshallow_f32(const PsArgs &a, size_t smem, cudaStream_t st);
cudaError_t launch_pshallow_bf16(const PsArgs &a, size_t smem, cudaStream_t st);
cudaError_t launch_pshallow_f16(const PsArgs &a, size_t smem, cudaStream_t st);
int occupancy_pshallow_f32(int K, size_t smem, int nthreads, int s);
int occupancy_pshallow_bf16(int K, size_t smem, int nthreads, int s);
int occupancy_pshallow_f16(int K, size_t smem, int nthreads, int s);

size_t pshallow_smem_bytes(const PsArgs &a) { return pshallow_layout(a).total; }

cudaError_t launch_pshallow(const PsArgs &a, int dtype, size_t smem, cudaStream_t st) {
    switch (dtype) {
    case 0: return launch_pshallow_f32(a, smem, st);
    case 1: return launch_pshallow_bf16(a, smem, st);
    case 2: return launch_pshallow_f16(a, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

int occupancy_pshallow(int dtype, int K, size_t smem, int nthreads, int s) {
    switch (dtype) {
    case 0: return occupancy_pshallow_f32(K, smem, nthreads, s);
    case 1: return occupancy_pshallow_bf16(K, smem, nthreads, s);
    case 2: return occupancy_pshallow_f16(K, smem, nthreads, s);
    default: return 0;
    }
}

}  // namespace wtconv
