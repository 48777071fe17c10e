/*
 * CPU reference for the weight gradient of 2-D convolution -- TEST
 * INFRASTRUCTURE ONLY.
 *
 * Only the tests and the benchmark's CPU-baseline leg use this file.  It shares
 * no code with the CUDA implementation (nor with conv2d_direct.c).
 *
 * What it computes: the backward pass with regard to the weight that burn runs
 * as conv_weight_backward (docs.rs burn-cubecl 0.20.0,
 * burn_cubecl/kernel/conv/base.rs: from the input feature map and the output
 * gradient, both permuted to NHWC, to a weight gradient of the weight's shape
 * permuted the same way, i.e. [K][R][S][C/groups]).  The forward sum
 *
 *   y[n][p][q][k] = bias[k] + sum_{r,s,c} x[n][ih][iw][g*C/G + c] * w[k][r][s][c],
 *   ih = p*sh - ph + r*dh,  iw = q*sw - pw + s*dw,  g = k / (K/G),
 *
 * is linear in w, so the derivative of a loss L with respect to w[k][r][s][c]
 * collects, over every output element that weight touches, dL/dy times the
 * input it multiplies:
 *
 *   dw[k][r][s][c] = sum_{n,p,q} dy[n][p][q][k] * x[n][ih][iw][g*C/G + c]
 *
 * with out-of-image positions contributing zero, exactly as in the forward
 * sum.  Arithmetic is IEEE fp64 in loop order (n, p, q); inputs are bf16 bit
 * patterns widened exactly.  Alongside each element it can return the sum of
 * the absolute values of its terms (used to scale test tolerances).
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t n, h, w, c, k, r, s;
    int64_t sh, sw, ph, pw, dh, dw;
    int64_t g;
    int64_t p, q;
} wgrad_shape;

static int64_t extent(int64_t in, int64_t pad, int64_t dil, int64_t ker, int64_t stride)
{
    int64_t room = in + 2 * pad - (dil * (ker - 1) + 1);
    return room < 0 ? 0 : room / stride + 1;
}

static int wgrad_make_shape(wgrad_shape* sp, const int64_t dims[7], const int64_t opts[7])
{
    sp->n = dims[0]; sp->h = dims[1]; sp->w = dims[2]; sp->c = dims[3];
    sp->k = dims[4]; sp->r = dims[5]; sp->s = dims[6];
    sp->sh = opts[0]; sp->sw = opts[1]; sp->ph = opts[2]; sp->pw = opts[3];
    sp->dh = opts[4]; sp->dw = opts[5]; sp->g = opts[6];
    for (int i = 0; i < 7; ++i) if (dims[i] < 0) return 1;
    if (sp->sh < 1 || sp->sw < 1 || sp->dh < 1 || sp->dw < 1 || sp->ph < 0 || sp->pw < 0) return 1;
    if (sp->r < 1 || sp->s < 1) return 1;
    if (sp->g < 1 || sp->c % sp->g != 0 || sp->k % sp->g != 0) return 1;
    sp->p = extent(sp->h, sp->ph, sp->dh, sp->r, sp->sh);
    sp->q = extent(sp->w, sp->pw, sp->dw, sp->s, sp->sw);
    return 0;
}

static double widen(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* One gradient element dw[k][r][s][c] (c within the group) and the sum of |terms|. */
static double wgrad_point(const wgrad_shape* sp, const double* x, const double* dy, int64_t k, int64_t r,
                          int64_t s, int64_t c, double* abs_sum)
{
    const int64_t cin = (k / (sp->k / sp->g)) * (sp->c / sp->g) + c; /* input channel */
    double acc = 0.0, mass = 0.0;
    for (int64_t n = 0; n < sp->n; ++n)
        for (int64_t p = 0; p < sp->p; ++p) {
            const int64_t ih = p * sp->sh - sp->ph + r * sp->dh;
            if (ih < 0 || ih >= sp->h) continue;
            for (int64_t q = 0; q < sp->q; ++q) {
                const int64_t iw = q * sp->sw - sp->pw + s * sp->dw;
                if (iw < 0 || iw >= sp->w) continue;
                const double t = dy[((n * sp->p + p) * sp->q + q) * sp->k + k] *
                                 x[((n * sp->h + ih) * sp->w + iw) * sp->c + cin];
                acc += t;
                mass += t < 0 ? -t : t;
            }
        }
    if (abs_sum) *abs_sum = mass;
    return acc;
}

typedef struct {
    const wgrad_shape* sp;
    const double* x;
    const double* dy;
    double* dw;
    double* mass; /* may be NULL */
    int64_t k_begin, k_end;
} wgrad_job;

static void* wgrad_rows(void* arg)
{
    wgrad_job* j = (wgrad_job*)arg;
    const wgrad_shape* sp = j->sp;
    const int64_t cg = sp->c / sp->g;
    for (int64_t k = j->k_begin; k < j->k_end; ++k)
        for (int64_t r = 0; r < sp->r; ++r)
            for (int64_t s = 0; s < sp->s; ++s)
                for (int64_t c = 0; c < cg; ++c) {
                    const int64_t at = ((k * sp->r + r) * sp->s + s) * cg + c;
                    double m = 0.0;
                    j->dw[at] = wgrad_point(sp, j->x, j->dy, k, r, s, c, &m);
                    if (j->mass) j->mass[at] = m;
                }
    return NULL;
}

/*
 * Full weight gradient over double inputs.
 *   dims = {N, H, W, C, K, R, S}; opts = {stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, groups}
 *   x: N*H*W*C doubles (NHWC); dy: N*P*Q*K doubles (NHWC)
 *   dw: K*R*S*(C/groups) doubles (KRSC); mass: the same shape or NULL (sum of |terms|)
 * Output channels are split statically over `threads` POSIX threads.
 * Returns 0 on success, 1 on invalid arguments, 2 if memory ran out.
 */
int oracle_wgrad_f64(const int64_t dims[7], const int64_t opts[7], const double* x, const double* dy, double* dw,
                     double* mass, int threads)
{
    wgrad_shape sp;
    if (wgrad_make_shape(&sp, dims, opts)) return 1;
    if (sp.k == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > sp.k) threads = (int)sp.k;
    pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)threads);
    wgrad_job* jobs = (wgrad_job*)malloc(sizeof(wgrad_job) * (size_t)threads);
    char* started = (char*)calloc((size_t)threads, 1);
    if (!tid || !jobs || !started) { free(tid); free(jobs); free(started); return 2; }
    for (int t = 0; t < threads; ++t) {
        jobs[t].sp = &sp; jobs[t].x = x; jobs[t].dy = dy; jobs[t].dw = dw; jobs[t].mass = mass;
        jobs[t].k_begin = sp.k * t / threads;
        jobs[t].k_end = sp.k * (t + 1) / threads;
    }
    for (int t = 1; t < threads; ++t) started[t] = pthread_create(&tid[t], NULL, wgrad_rows, &jobs[t]) == 0;
    wgrad_rows(&jobs[0]);
    for (int t = 1; t < threads; ++t) {
        if (started[t]) pthread_join(tid[t], NULL);
        else wgrad_rows(&jobs[t]);
    }
    free(started);
    free(tid);
    free(jobs);
    return 0;
}

static double* widen_all(const uint16_t* v, int64_t count)
{
    double* out = (double*)malloc(sizeof(double) * (size_t)(count > 0 ? count : 1));
    if (!out) return NULL;
    for (int64_t i = 0; i < count; ++i) out[i] = widen(v[i]);
    return out;
}

/* As oracle_wgrad_f64 with bf16 (bit pattern) x and dy. */
int oracle_wgrad_bf16(const int64_t dims[7], const int64_t opts[7], const uint16_t* x, const uint16_t* dy,
                      double* dw, double* mass, int threads)
{
    wgrad_shape sp;
    if (wgrad_make_shape(&sp, dims, opts)) return 1;
    double* xd = widen_all(x, sp.n * sp.h * sp.w * sp.c);
    double* dyd = widen_all(dy, sp.n * sp.p * sp.q * sp.k);
    int rc = 2;
    if (xd && dyd) rc = oracle_wgrad_f64(dims, opts, xd, dyd, dw, mass, threads);
    free(xd);
    free(dyd);
    return rc;
}

/*
 * Selected elements only: out[i] = dw[k_idx[i]][j_idx[i]] of the gradient viewed as
 * [K][R*S*(C/groups)], j = (r*S + s)*(C/groups) + c; mass[i] (may be NULL) the sum of
 * |terms|.  Double inputs.  Returns 0, or 1 on invalid arguments / indices.
 */
int oracle_wgrad_points_f64(const int64_t dims[7], const int64_t opts[7], const double* x, const double* dy,
                            const int64_t* k_idx, const int64_t* j_idx, int64_t npts, double* out, double* mass)
{
    wgrad_shape sp;
    if (wgrad_make_shape(&sp, dims, opts)) return 1;
    const int64_t cg = sp.c / sp.g;
    const int64_t cols = sp.r * sp.s * cg;
    for (int64_t i = 0; i < npts; ++i)
        if (k_idx[i] < 0 || k_idx[i] >= sp.k || j_idx[i] < 0 || j_idx[i] >= cols) return 1;
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t j = j_idx[i];
        const int64_t c = j % cg;
        const int64_t rs = j / cg;
        double m = 0.0;
        out[i] = wgrad_point(&sp, x, dy, k_idx[i], rs / sp.s, rs % sp.s, c, &m);
        if (mass) mass[i] = m;
    }
    return 0;
}
