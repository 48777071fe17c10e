/*
 * CPU reference for 2-D convolution forward -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg use this file.  It shares no code with the CUDA implementation.
 *
 * What it computes (the plain definition, with no blocking or reordering):
 * the direct convolution that burn keeps as its baseline strategy
 * ("Direct" in docs.rs burn-cubecl 0.20.0 burn_cubecl/kernel/conv/base.rs,
 * ConvStrategy / conv_forward_nhwc; "Direct" rows of burn PR #2287,
 * Benchmarking / Conv2d).  The im2col and implicit-GEMM algorithms of the same
 * pages compute this same quantity (burn PR #2287, Changes; burn PR #2545,
 * Changes), so it is the result the GPU path has to reproduce.
 *
 *   y[n][p][q][k] = bias[k]
 *                 + sum_{r,s,c} x[n][p*sh - ph + r*dh][q*sw - pw + s*dw][c] * w[k][r][s][c]
 *
 * with out-of-image input positions contributing zero (symmetric zero padding),
 * cross-correlation (no filter flip), NHWC input, KRSC weight and the bias
 * added once per output channel ("The bias added to each channel",
 * conv_forward's doc comment on the same page).  With `groups` = G (the
 * ConvOptions field of the same page; burn's conv_forward_nhwc sends G != 1 to
 * the direct strategy) the channels split into G equal consecutive groups:
 * output channel k belongs to group g = k / (K/G) and sums only over the input
 * channels g*C/G .. (g+1)*C/G - 1, its weight row holding C/G channels per tap
 * (weight [K][R][S][C/G]):
 *
 *   y[n][p][q][k] = bias[k] + sum_{r,s,c < C/G} x[n][ih][iw][g*C/G + c] * w[k][r][s][c]
 *
 * G = 1 is the formula above.  Output extents:
 *
 *   P = floor((H + 2*ph - dh*(R-1) - 1) / sh) + 1   (0 if the window does not fit)
 *
 * Arithmetic is IEEE fp64 in loop order (r, s, c) after the bias; inputs are
 * bf16 bit patterns widened exactly to double, the bias is fp32 widened to
 * double.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t n, h, w, c, k, r, s;
    int64_t sh, sw, ph, pw, dh, dw;
    int64_t g;       /* groups */
    int64_t p, q;
} oracle_shape;

/* Output extent along one spatial axis, from the definition above. */
int64_t oracle_out_extent(int64_t in, int64_t pad, int64_t dil, int64_t ker, int64_t stride)
{
    int64_t span = dil * (ker - 1) + 1;
    int64_t room = in + 2 * pad - span;
    if (room < 0) return 0;
    return room / stride + 1;
}

/* Exact widening of a bf16 bit pattern: the upper half of an fp32. */
static double bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* One output element y[n][p][q][k]: the seven-loop body, for fixed (n,p,q,k). */
static double conv_point(const oracle_shape* sp, const double* x, const double* w,
                         const float* bias, int64_t n, int64_t p, int64_t q, int64_t k)
{
    const int64_t cg = sp->c / sp->g;          /* input channels per group */
    const int64_t group = k / (sp->k / sp->g); /* the group of output channel k */
    double acc = bias ? (double)bias[k] : 0.0;
    for (int64_t r = 0; r < sp->r; ++r) {
        int64_t ih = p * sp->sh - sp->ph + r * sp->dh;
        if (ih < 0 || ih >= sp->h) continue;
        for (int64_t s = 0; s < sp->s; ++s) {
            int64_t iw = q * sp->sw - sp->pw + s * sp->dw;
            if (iw < 0 || iw >= sp->w) continue;
            const double* xv = x + ((n * sp->h + ih) * sp->w + iw) * sp->c + group * cg;
            const double* wv = w + ((k * sp->r + r) * sp->s + s) * cg;
            for (int64_t c = 0; c < cg; ++c) acc += xv[c] * wv[c];
        }
    }
    return acc;
}

typedef struct {
    const oracle_shape* sp;
    const double* x;
    const double* w;
    const float* bias;
    double* y;
    int64_t row_begin, row_end; /* rows are (n, p) pairs */
} conv_job;

static void* conv_rows(void* arg)
{
    conv_job* j = (conv_job*)arg;
    const oracle_shape* sp = j->sp;
    for (int64_t row = j->row_begin; row < j->row_end; ++row) {
        int64_t n = row / sp->p;
        int64_t p = row % sp->p;
        for (int64_t q = 0; q < sp->q; ++q)
            for (int64_t k = 0; k < sp->k; ++k)
                j->y[((n * sp->p + p) * sp->q + q) * sp->k + k] =
                    conv_point(sp, j->x, j->w, j->bias, n, p, q, k);
    }
    return NULL;
}

static int make_shape(oracle_shape* sp, const int64_t dims[7], const int64_t opts[7])
{
    sp->n = dims[0]; sp->h = dims[1]; sp->w = dims[2]; sp->c = dims[3];
    sp->k = dims[4]; sp->r = dims[5]; sp->s = dims[6];
    sp->sh = opts[0]; sp->sw = opts[1]; sp->ph = opts[2]; sp->pw = opts[3];
    sp->dh = opts[4]; sp->dw = opts[5]; sp->g = opts[6];
    for (int i = 0; i < 7; ++i) if (dims[i] < 0) return 1;
    if (sp->sh < 1 || sp->sw < 1 || sp->dh < 1 || sp->dw < 1 || sp->ph < 0 || sp->pw < 0) return 1;
    if (sp->r < 1 || sp->s < 1) return 1;
    if (sp->g < 1 || sp->c % sp->g != 0 || sp->k % sp->g != 0) return 1;
    sp->p = oracle_out_extent(sp->h, sp->ph, sp->dh, sp->r, sp->sh);
    sp->q = oracle_out_extent(sp->w, sp->pw, sp->dw, sp->s, sp->sw);
    return 0;
}

/*
 * Full convolution over double inputs.
 *   dims = {N, H, W, C, K, R, S}; opts = {stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, groups}
 *   x: N*H*W*C doubles (NHWC); w: K*R*S*(C/groups) doubles (KRSC); bias: K floats or NULL
 *   y: N*P*Q*K doubles (NHWC), P and Q from oracle_out_extent.
 * Rows (n, p) are split statically over `threads` POSIX threads.
 * Returns 0 on success, 1 on invalid arguments, 2 if a thread could not start.
 */
int oracle_conv2d_f64(const int64_t dims[7], const int64_t opts[7], const double* x,
                      const double* w, const float* bias, double* y, int threads)
{
    oracle_shape sp;
    if (make_shape(&sp, dims, opts)) return 1;
    int64_t rows = sp.n * sp.p;
    if (rows == 0 || sp.q == 0 || sp.k == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > rows) threads = (int)rows;
    pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)threads);
    conv_job* jobs = (conv_job*)malloc(sizeof(conv_job) * (size_t)threads);
    if (!tid || !jobs) { free(tid); free(jobs); return 2; }
    char* started = (char*)calloc((size_t)threads, 1);
    if (!started) { free(tid); free(jobs); return 2; }
    for (int t = 0; t < threads; ++t) {
        jobs[t].sp = &sp; jobs[t].x = x; jobs[t].w = w; jobs[t].bias = bias; jobs[t].y = y;
        jobs[t].row_begin = rows * t / threads;
        jobs[t].row_end = rows * (t + 1) / threads;
    }
    /* Threads 1..T-1 run on their own; the calling thread takes block 0. */
    for (int t = 1; t < threads; ++t)
        started[t] = pthread_create(&tid[t], NULL, conv_rows, &jobs[t]) == 0;
    conv_rows(&jobs[0]);
    for (int t = 1; t < threads; ++t) {
        if (started[t]) pthread_join(tid[t], NULL);
        else conv_rows(&jobs[t]);
    }
    free(started);
    free(tid);
    free(jobs);
    return 0;
}

static double* widen_bf16(const uint16_t* v, int64_t count)
{
    double* out = (double*)malloc(sizeof(double) * (size_t)(count > 0 ? count : 1));
    if (!out) return NULL;
    for (int64_t i = 0; i < count; ++i) out[i] = bf16_to_double(v[i]);
    return out;
}

/* Same as oracle_conv2d_f64 with bf16 (bit pattern) input and weight. */
int oracle_conv2d_bf16(const int64_t dims[7], const int64_t opts[7], const uint16_t* x,
                       const uint16_t* w, const float* bias, double* y, int threads)
{
    if (opts[6] < 1 || dims[3] % opts[6] != 0) return 1;
    int64_t nx = dims[0] * dims[1] * dims[2] * dims[3];
    int64_t nw = dims[4] * dims[5] * dims[6] * (dims[3] / opts[6]);
    double* xd = widen_bf16(x, nx);
    double* wd = widen_bf16(w, nw);
    int rc = 2;
    if (xd && wd) rc = oracle_conv2d_f64(dims, opts, xd, wd, bias, y, threads);
    free(xd);
    free(wd);
    return rc;
}

/* Selected output elements y[m_idx[i]][k_idx[i]] over already-widened inputs. */
static void points_f64(const oracle_shape* sp, const double* x, const double* w, const float* bias,
                       const int64_t* m_idx, const int64_t* k_idx, int64_t npts, double* out)
{
    for (int64_t i = 0; i < npts; ++i) {
        int64_t m = m_idx[i];
        int64_t q = m % sp->q;
        int64_t p = (m / sp->q) % sp->p;
        int64_t n = m / (sp->q * sp->p);
        out[i] = conv_point(sp, x, w, bias, n, p, q, k_idx[i]);
    }
}

static int check_points(const oracle_shape* sp, const int64_t* m_idx, const int64_t* k_idx, int64_t npts)
{
    int64_t mtot = sp->n * sp->p * sp->q;
    for (int64_t i = 0; i < npts; ++i)
        if (m_idx[i] < 0 || m_idx[i] >= mtot || k_idx[i] < 0 || k_idx[i] >= sp->k) return 1;
    return 0;
}

/*
 * Selected output elements only: for each i, out[i] = y[m_idx[i]][k_idx[i]] where
 * m = (n*P + p)*Q + q is the row of the NHWC output viewed as [N*P*Q][K].
 * Returns 0, 1 on invalid arguments / out-of-range indices, 2 on allocation failure.
 */
int oracle_conv2d_points_bf16(const int64_t dims[7], const int64_t opts[7], const uint16_t* x,
                              const uint16_t* w, const float* bias, const int64_t* m_idx,
                              const int64_t* k_idx, int64_t npts, double* out)
{
    oracle_shape sp;
    if (make_shape(&sp, dims, opts) || check_points(&sp, m_idx, k_idx, npts)) return 1;
    double* xd = widen_bf16(x, sp.n * sp.h * sp.w * sp.c);
    double* wd = widen_bf16(w, sp.k * sp.r * sp.s * (sp.c / sp.g));
    if (!xd || !wd) { free(xd); free(wd); return 2; }
    points_f64(&sp, xd, wd, bias, m_idx, k_idx, npts, out);
    free(xd);
    free(wd);
    return 0;
}

/* As oracle_conv2d_points_bf16 over double inputs (for repeated sampling of one problem). */
int oracle_conv2d_points_f64(const int64_t dims[7], const int64_t opts[7], const double* x,
                             const double* w, const float* bias, const int64_t* m_idx,
                             const int64_t* k_idx, int64_t npts, double* out)
{
    oracle_shape sp;
    if (make_shape(&sp, dims, opts) || check_points(&sp, m_idx, k_idx, npts)) return 1;
    points_f64(&sp, x, w, bias, m_idx, k_idx, npts, out);
    return 0;
}
