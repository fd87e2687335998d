/*
 * WTConv CPU oracle -- TEST INFRASTRUCTURE, not part of the product.
 *
 * Only the test suite, the package's smoke check and the benchmark's CPU-baseline leg may load
 * this library.  It is a plain, slow, fp64 restatement of what the WTConv layer computes, written
 * from the paper "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware Reformulation"
 * (arXiv 2608.10805) as summarised on its web pages.  It shares no code with the CUDA library.
 *
 * It follows the *reference* pipeline the paper describes (Resumo Tecnico -- Problema and
 * Metodologia on the gist.science Portuguese page): an explicit Haar analysis per level that
 * materialises the coefficient tensor Y^(l), a depthwise conv per subband, the learned
 * per-channel scale as a separate elementwise pass, the L-step sequential synthesis cascade in
 * which each step adds the previous reconstruction to the low-pass subband and applies the
 * inverse transform, and the base depthwise conv with bias times its scale.  None of the
 * paper's three reformulations (on-chip analysis, closed-form synthesis, weight folding) is
 * used here.  The backward pass reverses every step with the literal transpose of its loop.
 *
 * Readings taken where the pages are silent:
 *   - Haar filters: the four 2x2 sign patterns LL [[1,1],[1,1]], LH [[1,-1],[1,-1]],
 *     HL [[1,1],[-1,-1]], HH [[1,-1],[-1,1]] times 1/2 with stride 2 (page 4, section 3, the
 *     TensorFlow Haar snippet; "fixed power-of-two scaling" in the Metodologia section).
 *   - Subband channel order 4c+s with s = 0 LL, 1 LH, 2 HL, 3 HH.
 *   - Level l analyses the raw low band LL_(l-1) of level l-1 (LL_0 = x).
 *   - Conv: cross-correlation, stride 1, zero 'same' padding of k/2 at each level's resolution,
 *     odd k, no wavelet bias.
 *   - The synthesis adds the previous reconstruction to the *scaled conv output* of the LL
 *     subband, then inverts the transform.
 *   - Base path: y_base = base_scale * (conv(x, base_w) + base_bias): the bias is scaled too
 *     ("folded into the weights, and into the bias for the base path").
 *   - Odd sides: a level whose input has an odd number of rows (columns) pads it with one zero
 *     row (column) at the end before the analysis, as the stride-2 'SAME' Haar conv of the page-4
 *     snippet does, so level l has ceil(n_(l-1) / 2) positions per side; the synthesis crops each
 *     level's reconstruction back to the size of that level's input.
 *
 * Parity status: the pages print no worked example, so nothing here is pinned to printed
 * values.  Every function is pinned by the tests to mathematics instead (perfect
 * reconstruction, Parseval, library convolution, closed forms, dense-matrix brute force,
 * finite differences, Euler identities).
 *
 * All arrays are row-major.  Threads (pthreads) split the work over channels; each channel's
 * planes are processed in batch order, so results do not depend on the thread count.
 */
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* Haar 2x2 sign patterns (page 4, section 3), indexed [subband][row offset a][col offset b]. */
static const double HAAR_SIGN[4][2][2] = {
    {{1.0, 1.0}, {1.0, 1.0}},   /* LL */
    {{1.0, -1.0}, {1.0, -1.0}}, /* LH */
    {{1.0, 1.0}, {-1.0, -1.0}}, /* HL */
    {{1.0, -1.0}, {-1.0, 1.0}}, /* HH */
};

/* ---------------------------------------------------------------- building blocks ------- */

/* One level of the 2-D Haar analysis: a stride-2 conv of the H x W plane `in` with the four
 * 2x2 filters.  out is [4][H/2][W/2]. */
void oracle_haar_analysis(const double *in, int H, int W, double *out)
{
    int h = H / 2, w = W / 2;
    for (int s = 0; s < 4; ++s)
        for (int i = 0; i < h; ++i)
            for (int j = 0; j < w; ++j) {
                double acc = 0.0;
                for (int a = 0; a < 2; ++a)
                    for (int b = 0; b < 2; ++b)
                        acc += 0.5 * HAAR_SIGN[s][a][b] * in[(2 * i + a) * W + (2 * j + b)];
                out[(s * h + i) * w + j] = acc;
            }
}

/* One level of the inverse transform: the transposed stride-2 conv with the same four filters.
 * in is [4][h][w]; out is the 2h x 2w plane. */
void oracle_haar_synthesis(const double *in, int h, int w, double *out)
{
    int W = 2 * w;
    for (int i = 0; i < h; ++i)
        for (int j = 0; j < w; ++j)
            for (int a = 0; a < 2; ++a)
                for (int b = 0; b < 2; ++b) {
                    double acc = 0.0;
                    for (int s = 0; s < 4; ++s)
                        acc += 0.5 * HAAR_SIGN[s][a][b] * in[(s * h + i) * w + j];
                    out[(2 * i + a) * W + (2 * j + b)] = acc;
                }
}

/* Depthwise k x k cross-correlation of one H x W plane, zero 'same' padding, stride 1:
 * out[i][j] = sum_{u,v} ker[u][v] * in[i+u-p][j+v-p], p = k/2. */
void oracle_dwconv(const double *in, int H, int W, const double *ker, int k, double *out)
{
    int p = k / 2;
    for (int i = 0; i < H; ++i)
        for (int j = 0; j < W; ++j) {
            double acc = 0.0;
            for (int u = 0; u < k; ++u)
                for (int v = 0; v < k; ++v) {
                    int r = i + u - p, c = j + v - p;
                    if (r >= 0 && r < H && c >= 0 && c < W)
                        acc += ker[u * k + v] * in[r * W + c];
                }
            out[i * W + j] = acc;
        }
}

/* --- transposes (adjoints) of the building blocks, each the literal transpose of the loop
 *     above: every multiply-add `out += m * in` becomes `d_in += m * d_out`. */

/* Adjoint of oracle_haar_analysis: d_in (H x W) += A^T d_out ([4][H/2][W/2]). */
static void haar_analysis_adjoint(const double *d_out, int H, int W, double *d_in)
{
    int h = H / 2, w = W / 2;
    for (int s = 0; s < 4; ++s)
        for (int i = 0; i < h; ++i)
            for (int j = 0; j < w; ++j)
                for (int a = 0; a < 2; ++a)
                    for (int b = 0; b < 2; ++b)
                        d_in[(2 * i + a) * W + (2 * j + b)] +=
                            0.5 * HAAR_SIGN[s][a][b] * d_out[(s * h + i) * w + j];
}

/* Adjoint of oracle_haar_synthesis: d_in ([4][h][w]) += S^T d_out (2h x 2w). */
static void haar_synthesis_adjoint(const double *d_out, int h, int w, double *d_in)
{
    int W = 2 * w;
    for (int i = 0; i < h; ++i)
        for (int j = 0; j < w; ++j)
            for (int a = 0; a < 2; ++a)
                for (int b = 0; b < 2; ++b)
                    for (int s = 0; s < 4; ++s)
                        d_in[(s * h + i) * w + j] +=
                            0.5 * HAAR_SIGN[s][a][b] * d_out[(2 * i + a) * W + (2 * j + b)];
}

/* Adjoint of oracle_dwconv with respect to its input: d_in += K^T d_out. */
static void dwconv_adjoint_input(const double *d_out, int H, int W, const double *ker, int k,
                                 double *d_in)
{
    int p = k / 2;
    for (int i = 0; i < H; ++i)
        for (int j = 0; j < W; ++j)
            for (int u = 0; u < k; ++u)
                for (int v = 0; v < k; ++v) {
                    int r = i + u - p, c = j + v - p;
                    if (r >= 0 && r < H && c >= 0 && c < W)
                        d_in[r * W + c] += ker[u * k + v] * d_out[i * W + j];
                }
}

/* Adjoint of oracle_dwconv with respect to its kernel: d_ker += sum over outputs. */
static void dwconv_adjoint_kernel(const double *d_out, int H, int W, const double *in, int k,
                                  double *d_ker)
{
    int p = k / 2;
    for (int i = 0; i < H; ++i)
        for (int j = 0; j < W; ++j)
            for (int u = 0; u < k; ++u)
                for (int v = 0; v < k; ++v) {
                    int r = i + u - p, c = j + v - p;
                    if (r >= 0 && r < H && c >= 0 && c < W)
                        d_ker[u * k + v] += in[r * W + c] * d_out[i * W + j];
                }
}

/* ------------------------------------------------------------ per-plane pipeline -------- */

#define ORACLE_MAX_LEVELS 16

/* Side lengths of every level: hs[0] = H, hs[l] = ceil(hs[l-1] / 2) (odd sides padded with one
 * zero at the end before the analysis); likewise ws. */
static void level_sizes(int H, int W, int L, int *hs, int *ws)
{
    hs[0] = H;
    ws[0] = W;
    for (int l = 1; l <= L; ++l) {
        hs[l] = (hs[l - 1] + 1) / 2;
        ws[l] = (ws[l - 1] + 1) / 2;
    }
}

typedef struct {
    int B, C, H, W, L, k;
    const double *x, *dy;
    const double *base_w, *base_bias, *base_scale, *wavelet_w, *wavelet_scale;
    double *y, *dx;
    double *d_base_w, *d_base_bias, *d_base_scale, *d_wavelet_w, *d_wavelet_scale;
    int backward;
    int nthreads, tid;
    int status;
} job_t;

/* Scratch for one plane: the materialised tensors of the reference pipeline. */
typedef struct {
    double **Y;     /* Y[l]: [4][H_l][W_l], analysis coefficients of level l (1-based) */
    double **T;     /* T[l]: conv outputs before the scale */
    double **Z;     /* Z[l]: scaled conv outputs (LL later receives the reconstruction) */
    double *R, *R2; /* reconstruction buffers, up to 2*hs[1] x 2*ws[1] */
    double *Pd;     /* a level's input padded to even sides */
    double *base;   /* conv(x, base_w) */
    double **dZ, **dT, **dY;
    double *dR, *dR2, *dbase;
} scratch_t;

static int scratch_alloc(scratch_t *s, int H, int W, int L)
{
    memset(s, 0, sizeof(*s));
    int hs[ORACLE_MAX_LEVELS + 1], ws[ORACLE_MAX_LEVELS + 1];
    level_sizes(H, W, L, hs, ws);
    size_t HW = (size_t)H * W, HW2 = (size_t)(2 * hs[1]) * (2 * ws[1]);
    s->Y = calloc((size_t)L + 1, sizeof(double *));
    s->T = calloc((size_t)L + 1, sizeof(double *));
    s->Z = calloc((size_t)L + 1, sizeof(double *));
    s->dZ = calloc((size_t)L + 1, sizeof(double *));
    s->dT = calloc((size_t)L + 1, sizeof(double *));
    s->dY = calloc((size_t)L + 1, sizeof(double *));
    if (!s->Y || !s->T || !s->Z || !s->dZ || !s->dT || !s->dY)
        return -1;
    for (int l = 1; l <= L; ++l) {
        size_t n = 4 * (size_t)hs[l] * (size_t)ws[l];
        s->Y[l] = malloc(n * sizeof(double));
        s->T[l] = malloc(n * sizeof(double));
        s->Z[l] = malloc(n * sizeof(double));
        s->dZ[l] = malloc(n * sizeof(double));
        s->dT[l] = malloc(n * sizeof(double));
        s->dY[l] = malloc(n * sizeof(double));
        if (!s->Y[l] || !s->T[l] || !s->Z[l] || !s->dZ[l] || !s->dT[l] || !s->dY[l])
            return -1;
    }
    s->R = malloc(HW2 * sizeof(double));
    s->R2 = malloc(HW2 * sizeof(double));
    s->Pd = malloc(HW2 * sizeof(double));
    s->base = malloc(HW * sizeof(double));
    s->dR = malloc(HW2 * sizeof(double));
    s->dR2 = malloc(HW2 * sizeof(double));
    s->dbase = malloc(HW * sizeof(double));
    if (!s->R || !s->R2 || !s->Pd || !s->base || !s->dR || !s->dR2 || !s->dbase)
        return -1;
    return 0;
}

static void scratch_free(scratch_t *s, int L)
{
    for (int l = 1; l <= L; ++l) {
        if (s->Y) free(s->Y[l]);
        if (s->T) free(s->T[l]);
        if (s->Z) free(s->Z[l]);
        if (s->dZ) free(s->dZ[l]);
        if (s->dT) free(s->dT[l]);
        if (s->dY) free(s->dY[l]);
    }
    free(s->Y); free(s->T); free(s->Z); free(s->dZ); free(s->dT); free(s->dY);
    free(s->R); free(s->R2); free(s->Pd); free(s->base); free(s->dR); free(s->dR2); free(s->dbase);
}

/* Forward of one (b, c) plane through the reference pipeline. Leaves the materialised
 * intermediates in `s` for the backward. */
static void plane_forward(const job_t *J, int c, const double *x, double *y, scratch_t *s)
{
    int H = J->H, W = J->W, L = J->L, k = J->k, C = J->C;
    size_t kk = (size_t)k * k;
    int hs[ORACLE_MAX_LEVELS + 1], ws[ORACLE_MAX_LEVELS + 1];
    level_sizes(H, W, L, hs, ws);

    /* (1) analysis cascade: Y^(l) = WT(LL_(l-1)), LL_0 = x, LL_l = subband 0 of Y^(l); an odd
     *     side of LL_(l-1) gets one zero row / column at its end first */
    const double *LL = x;
    for (int l = 1; l <= L; ++l) {
        int hi = hs[l - 1], wi = ws[l - 1], h = hs[l], w = ws[l];
        if (hi == 2 * h && wi == 2 * w) {
            oracle_haar_analysis(LL, hi, wi, s->Y[l]);
        } else {
            memset(s->Pd, 0, (size_t)(2 * h) * (2 * w) * sizeof(double));
            for (int i = 0; i < hi; ++i)
                for (int j = 0; j < wi; ++j)
                    s->Pd[i * (2 * w) + j] = LL[i * wi + j];
            oracle_haar_analysis(s->Pd, 2 * h, 2 * w, s->Y[l]);
        }
        LL = s->Y[l]; /* subband 0 is the first [h_l][w_l] block */
    }

    /* (2) depthwise conv per subband, (3) the learned scale as its own pass */
    for (int l = 1; l <= L; ++l) {
        int h = hs[l], w = ws[l];
        size_t n = (size_t)h * w;
        for (int sb = 0; sb < 4; ++sb) {
            const double *ker = J->wavelet_w + ((size_t)(l - 1) * 4 * C + 4 * c + sb) * kk;
            oracle_dwconv(s->Y[l] + sb * n, h, w, ker, k, s->T[l] + sb * n);
        }
        for (int sb = 0; sb < 4; ++sb) {
            double sc = J->wavelet_scale[(size_t)(l - 1) * 4 * C + 4 * c + sb];
            for (size_t i = 0; i < n; ++i)
                s->Z[l][sb * n + i] = sc * s->T[l][sb * n + i];
        }
    }

    /* (4) synthesis cascade, levels L..1: add the previous reconstruction to the LL subband,
     *     then invert the transform. R holds the reconstruction at the current resolution. */
    {
        memset(s->R, 0, (size_t)hs[L] * ws[L] * sizeof(double));
        for (int l = L; l >= 1; --l) {
            int h = hs[l], w = ws[l], ho = hs[l - 1], wo = ws[l - 1];
            for (int i = 0; i < h * w; ++i)
                s->Z[l][i] += s->R[i]; /* subband 0 = LL */
            oracle_haar_synthesis(s->Z[l], h, w, s->R2);
            /* back to the size of this level's input (drops a padded row / column) */
            for (int i = 0; i < ho; ++i)
                for (int j = 0; j < wo; ++j)
                    s->R[i * wo + j] = s->R2[i * (2 * w) + j];
        }
    }

    /* (5) base path: y = base_scale * (conv(x, base_w) + base_bias) + R */
    oracle_dwconv(x, H, W, J->base_w + (size_t)c * kk, k, s->base);
    double sb_ = J->base_scale[c], bb = J->base_bias[c];
    for (int i = 0; i < H * W; ++i)
        y[i] = sb_ * (s->base[i] + bb) + s->R[i];
}

/* Backward of one (b, c) plane: reverse every forward step in turn.  Requires the
 * intermediates from plane_forward on the same plane. */
static void plane_backward(const job_t *J, int c, const double *x, const double *dy, double *dx,
                           scratch_t *s, double *g_base_w, double *g_base_bias,
                           double *g_base_scale, double *g_wavelet_w, double *g_wavelet_scale)
{
    int H = J->H, W = J->W, L = J->L, k = J->k, C = J->C;
    size_t kk = (size_t)k * k, HW = (size_t)H * W;
    double sb_ = J->base_scale[c], bb = J->base_bias[c];
    int hs[ORACLE_MAX_LEVELS + 1], ws[ORACLE_MAX_LEVELS + 1];
    level_sizes(H, W, L, hs, ws);

    /* (5) base path.  y = sb * (base + bb) + R. */
    double acc_scale = 0.0, acc_bias = 0.0;
    for (size_t i = 0; i < HW; ++i) {
        acc_scale += dy[i] * (s->base[i] + bb);
        acc_bias += dy[i];
        s->dbase[i] = sb_ * dy[i];
    }
    g_base_scale[c] += acc_scale;
    g_base_bias[c] += sb_ * acc_bias;
    dwconv_adjoint_kernel(s->dbase, H, W, x, k, g_base_w + (size_t)c * kk);
    memset(dx, 0, HW * sizeof(double));
    dwconv_adjoint_input(s->dbase, H, W, J->base_w + (size_t)c * kk, k, dx);

    /* (4) synthesis cascade in reverse, levels 1..L.  The forward step at level l was
     *     Z[l].LL += R_(l+1); R_l = crop(IWT(Z[l])).  Reversed: the crop's transpose pads dR_l
     *     with zeros to 2h x 2w, dZ[l] = IWT^T of that, then dR_(l+1) = dZ[l].LL (the
     *     reconstruction entered the LL subband with weight 1). */
    memcpy(s->dR, dy, HW * sizeof(double)); /* y = ... + R_1 */
    for (int l = 1; l <= L; ++l) {
        int h = hs[l], w = ws[l], ho = hs[l - 1], wo = ws[l - 1];
        size_t n = 4 * (size_t)h * w;
        memset(s->dR2, 0, (size_t)(2 * h) * (2 * w) * sizeof(double));
        for (int i = 0; i < ho; ++i)
            for (int j = 0; j < wo; ++j)
                s->dR2[i * (2 * w) + j] = s->dR[i * wo + j];
        memset(s->dZ[l], 0, n * sizeof(double));
        haar_synthesis_adjoint(s->dR2, h, w, s->dZ[l]);
        memcpy(s->dR, s->dZ[l], (size_t)h * w * sizeof(double)); /* LL block */
    }

    /* (3) scale pass and (2) conv, per level and subband */
    for (int l = 1; l <= L; ++l) {
        int h = hs[l], w = ws[l];
        size_t n = (size_t)h * w;
        memset(s->dY[l], 0, 4 * n * sizeof(double));
        for (int sb = 0; sb < 4; ++sb) {
            size_t ch = (size_t)(l - 1) * 4 * C + 4 * c + sb;
            double sc = J->wavelet_scale[ch];
            double acc = 0.0;
            for (size_t i = 0; i < n; ++i) {
                acc += s->dZ[l][sb * n + i] * s->T[l][sb * n + i];
                s->dT[l][sb * n + i] = sc * s->dZ[l][sb * n + i];
            }
            g_wavelet_scale[ch] += acc;
            const double *ker = J->wavelet_w + ch * kk;
            dwconv_adjoint_kernel(s->dT[l] + sb * n, h, w, s->Y[l] + sb * n, k,
                                  g_wavelet_w + ch * kk);
            dwconv_adjoint_input(s->dT[l] + sb * n, h, w, ker, k, s->dY[l] + sb * n);
        }
    }

    /* (1) analysis cascade in reverse, levels L..1: LL_l = Y^(l).LL feeds level l+1, so its
     *     gradient collects from there before flowing through WT^T into the padded LL_(l-1);
     *     the padding's transpose then drops the padded row / column. */
    {
        memset(s->dR2, 0, (size_t)hs[L] * ws[L] * sizeof(double)); /* dLL_L = 0 */
        for (int l = L; l >= 1; --l) {
            int h = hs[l], w = ws[l], hi = hs[l - 1], wi = ws[l - 1];
            for (int i = 0; i < h * w; ++i)
                s->dY[l][i] += s->dR2[i];
            memset(s->Pd, 0, (size_t)(2 * h) * (2 * w) * sizeof(double));
            haar_analysis_adjoint(s->dY[l], 2 * h, 2 * w, s->Pd);
            for (int i = 0; i < hi; ++i)
                for (int j = 0; j < wi; ++j)
                    s->dR2[i * wi + j] = s->Pd[i * (2 * w) + j];
        }
        for (size_t i = 0; i < HW; ++i)
            dx[i] += s->dR2[i]; /* LL_0 = x */
    }
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    int B = J->B, C = J->C, H = J->H, W = J->W, L = J->L;
    size_t HW = (size_t)H * W;
    scratch_t s;
    if (scratch_alloc(&s, H, W, L) != 0) {
        scratch_free(&s, L);
        J->status = -2;
        return NULL;
    }
    double *y_tmp = J->backward ? malloc(HW * sizeof(double)) : NULL;
    if (J->backward && !y_tmp) {
        scratch_free(&s, L);
        J->status = -2;
        return NULL;
    }
    for (int c = J->tid; c < C; c += J->nthreads) {
        for (int b = 0; b < B; ++b) {
            size_t off = ((size_t)b * C + c) * HW;
            if (!J->backward) {
                plane_forward(J, c, J->x + off, J->y + off, &s);
            } else {
                plane_forward(J, c, J->x + off, y_tmp, &s);
                plane_backward(J, c, J->x + off, J->dy + off, J->dx + off, &s, J->d_base_w,
                               J->d_base_bias, J->d_base_scale, J->d_wavelet_w,
                               J->d_wavelet_scale);
            }
        }
    }
    free(y_tmp);
    scratch_free(&s, L);
    J->status = 0;
    return NULL;
}

static int check_shape(int B, int C, int H, int W, int L, int k)
{
    if (B <= 0 || C <= 0 || H <= 0 || W <= 0 || L < 1 || L > ORACLE_MAX_LEVELS || k < 1 || (k % 2) == 0)
        return -1;
    return 0;
}

static int run_jobs(job_t *proto, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > proto->C)
        nthreads = proto->C;
    job_t *jobs = calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs); free(th);
        return -2;
    }
    int status = 0, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].tid = t;
        jobs[t].nthreads = nthreads;
        jobs[t].status = -3;
        if (t == 0)
            continue; /* thread 0's share runs on the calling thread */
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) {
            status = -3;
            break;
        }
        started = t;
    }
    if (status == 0)
        worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads && status == 0; ++t)
        if (jobs[t].status != 0)
            status = jobs[t].status;
    free(jobs); free(th);
    return status;
}

/* ------------------------------------------------------------------- entry points ------- */

/* Forward: y = s_b (conv(x, base_w) + base_bias) + cascade synthesis of the scaled per-level
 * subband convs.  Shapes: x, y [B][C][H][W]; base_w [C][k][k]; base_bias, base_scale [C];
 * wavelet_w [L][4C][k][k]; wavelet_scale [L][4C].  Returns 0, -1 (bad shape), -2 (no memory),
 * -3 (threads). */
int oracle_forward(int B, int C, int H, int W, int L, int k, const double *x,
                   const double *base_w, const double *base_bias, const double *base_scale,
                   const double *wavelet_w, const double *wavelet_scale, double *y, int nthreads)
{
    if (check_shape(B, C, H, W, L, k) != 0)
        return -1;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.B = B; J.C = C; J.H = H; J.W = W; J.L = L; J.k = k;
    J.x = x; J.base_w = base_w; J.base_bias = base_bias; J.base_scale = base_scale;
    J.wavelet_w = wavelet_w; J.wavelet_scale = wavelet_scale; J.y = y;
    J.backward = 0;
    return run_jobs(&J, nthreads);
}

/* Backward: dx and every parameter gradient for upstream gradient dy.  Gradient arrays are
 * overwritten (zeroed first).  Same shapes as the forward; grads match their parameters. */
int oracle_backward(int B, int C, int H, int W, int L, int k, const double *x, const double *dy,
                    const double *base_w, const double *base_bias, const double *base_scale,
                    const double *wavelet_w, const double *wavelet_scale, double *dx,
                    double *d_base_w, double *d_base_bias, double *d_base_scale,
                    double *d_wavelet_w, double *d_wavelet_scale, int nthreads)
{
    if (check_shape(B, C, H, W, L, k) != 0)
        return -1;
    size_t kk = (size_t)k * k;
    memset(d_base_w, 0, (size_t)C * kk * sizeof(double));
    memset(d_base_bias, 0, (size_t)C * sizeof(double));
    memset(d_base_scale, 0, (size_t)C * sizeof(double));
    memset(d_wavelet_w, 0, (size_t)L * 4 * C * kk * sizeof(double));
    memset(d_wavelet_scale, 0, (size_t)L * 4 * C * sizeof(double));
    job_t J;
    memset(&J, 0, sizeof(J));
    J.B = B; J.C = C; J.H = H; J.W = W; J.L = L; J.k = k;
    J.x = x; J.dy = dy; J.base_w = base_w; J.base_bias = base_bias; J.base_scale = base_scale;
    J.wavelet_w = wavelet_w; J.wavelet_scale = wavelet_scale; J.dx = dx;
    J.d_base_w = d_base_w; J.d_base_bias = d_base_bias; J.d_base_scale = d_base_scale;
    J.d_wavelet_w = d_wavelet_w; J.d_wavelet_scale = d_wavelet_scale;
    J.backward = 1;
    return run_jobs(&J, nthreads);
}
