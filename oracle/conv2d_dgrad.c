/*
 * CPU reference for the data gradient of 2-D convolution -- TEST
 * INFRASTRUCTURE ONLY.
 *
 * Only the tests and the benchmark's CPU-baseline leg use this file.  It shares
 * no code with the CUDA implementation (nor with the other oracle files).
 *
 * What it computes: the backward pass with regard to the input that burn runs
 * as conv_data_backward (docs.rs burn-cubecl 0.20.0,
 * burn_cubecl/kernel/conv/base.rs: from the output gradient and the weights,
 * both permuted to NHWC / KRSC, to a gradient of the input's shape, NHWC).
 * The forward sum
 *
 *   y[n][p][q][k] = bias[k] + sum_{r,s,c} x[n][p*sh - ph + r*dh][q*sw - pw + s*dw][g*C/G + c] * w[k][r][s][c]
 *
 * is linear in x, so the derivative of a loss with respect to x[n][h][w][ci]
 * collects dL/dy times the weight over every (output element, tap) whose
 * window reads that input position:
 *
 *   dx[n][h][w][ci] = sum_{r,s} sum_{k in group(ci)} dy[n][p][q][k] * w[k][r][s][ci - g*C/G]
 *       over the taps with h + ph - r*dh = p*sh and w + pw - s*dw = q*sw for
 *       integers 0 <= p < P, 0 <= q < Q (g = ci / (C/G); group(ci) = the
 *       output channels g*K/G .. (g+1)*K/G - 1).
 *
 * This is conv_transpose2d's definition as well (conv_transpose2d of dy with
 * the weight read as [in = K][R][S][out = C]).  Arithmetic is IEEE fp64 in loop
 * order (r, s, k); inputs are bf16 bit patterns widened exactly.  Alongside
 * each element it can return the sum of |terms|.
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
} dgrad_shape;

static int64_t dgrad_extent(int64_t in, int64_t pad, int64_t dil, int64_t ker, int64_t stride)
{
    int64_t room = in + 2 * pad - (dil * (ker - 1) + 1);
    return room < 0 ? 0 : room / stride + 1;
}

static int dgrad_make_shape(dgrad_shape* sp, const int64_t dims[7], const int64_t opts[7])
{
    sp->n = dims[0]; sp->h = dims[1]; sp->w = dims[2]; sp->c = dims[3];
    sp->k = dims[4]; sp->r = dims[5]; sp->s = dims[6];
    sp->sh = opts[0]; sp->sw = opts[1]; sp->ph = opts[2]; sp->pw = opts[3];
    sp->dh = opts[4]; sp->dw = opts[5]; sp->g = opts[6];
    for (int i = 0; i < 7; ++i) if (dims[i] < 0) return 1;
    if (sp->sh < 1 || sp->sw < 1 || sp->dh < 1 || sp->dw < 1 || sp->ph < 0 || sp->pw < 0) return 1;
    if (sp->r < 1 || sp->s < 1) return 1;
    if (sp->g < 1 || sp->c % sp->g != 0 || sp->k % sp->g != 0) return 1;
    sp->p = dgrad_extent(sp->h, sp->ph, sp->dh, sp->r, sp->sh);
    sp->q = dgrad_extent(sp->w, sp->pw, sp->dw, sp->s, sp->sw);
    return 0;
}

static double widen16(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* One input-gradient element dx[n][h][w][ci] and the sum of |terms|. */
static double dgrad_point(const dgrad_shape* sp, const double* dy, const double* wt, int64_t n, int64_t h,
                          int64_t w, int64_t ci, double* abs_sum)
{
    const int64_t cg = sp->c / sp->g, kg = sp->k / sp->g;
    const int64_t grp = ci / cg;
    const int64_t cw = ci - grp * cg; /* channel within the weight row */
    double acc = 0.0, mass = 0.0;
    for (int64_t r = 0; r < sp->r; ++r) {
        const int64_t th = h + sp->ph - r * sp->dh;
        if (th < 0 || th % sp->sh != 0) continue;
        const int64_t p = th / sp->sh;
        if (p >= sp->p) continue;
        for (int64_t s = 0; s < sp->s; ++s) {
            const int64_t tw = w + sp->pw - s * sp->dw;
            if (tw < 0 || tw % sp->sw != 0) continue;
            const int64_t q = tw / sp->sw;
            if (q >= sp->q) continue;
            const double* g = dy + ((n * sp->p + p) * sp->q + q) * sp->k;
            for (int64_t kk = grp * kg; kk < (grp + 1) * kg; ++kk) {
                const double t = g[kk] * wt[((kk * sp->r + r) * sp->s + s) * cg + cw];
                acc += t;
                mass += t < 0 ? -t : t;
            }
        }
    }
    if (abs_sum) *abs_sum = mass;
    return acc;
}

typedef struct {
    const dgrad_shape* sp;
    const double* dy;
    const double* wt;
    double* dx;
    double* mass; /* may be NULL */
    int64_t row_begin, row_end; /* rows are (n, h) pairs */
} dgrad_job;

static void* dgrad_rows(void* arg)
{
    dgrad_job* j = (dgrad_job*)arg;
    const dgrad_shape* sp = j->sp;
    for (int64_t row = j->row_begin; row < j->row_end; ++row) {
        const int64_t n = row / sp->h, h = row % sp->h;
        for (int64_t w = 0; w < sp->w; ++w)
            for (int64_t ci = 0; ci < sp->c; ++ci) {
                const int64_t at = ((n * sp->h + h) * sp->w + w) * sp->c + ci;
                double m = 0.0;
                j->dx[at] = dgrad_point(sp, j->dy, j->wt, n, h, w, ci, &m);
                if (j->mass) j->mass[at] = m;
            }
    }
    return NULL;
}

/*
 * Full input gradient over double inputs.
 *   dims = {N, H, W, C, K, R, S} of the forward convolution; opts = {stride_h, stride_w, pad_h, pad_w,
 *   dil_h, dil_w, groups}; dy: N*P*Q*K doubles (NHWC); wt: K*R*S*(C/groups) doubles (KRSC)
 *   dx: N*H*W*C doubles (NHWC); mass: the same shape or NULL (sum of |terms|)
 * Rows (n, h) are split statically over `threads` POSIX threads.
 * Returns 0 on success, 1 on invalid arguments, 2 if memory ran out.
 */
int oracle_dgrad_f64(const int64_t dims[7], const int64_t opts[7], const double* dy, const double* wt, double* dx,
                     double* mass, int threads)
{
    dgrad_shape sp;
    if (dgrad_make_shape(&sp, dims, opts)) return 1;
    const int64_t rows = sp.n * sp.h;
    if (rows == 0 || sp.c == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > rows) threads = (int)rows;
    pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)threads);
    dgrad_job* jobs = (dgrad_job*)malloc(sizeof(dgrad_job) * (size_t)threads);
    char* started = (char*)calloc((size_t)threads, 1);
    if (!tid || !jobs || !started) { free(tid); free(jobs); free(started); return 2; }
    for (int t = 0; t < threads; ++t) {
        jobs[t].sp = &sp; jobs[t].dy = dy; jobs[t].wt = wt; jobs[t].dx = dx; jobs[t].mass = mass;
        jobs[t].row_begin = rows * t / threads;
        jobs[t].row_end = rows * (t + 1) / threads;
    }
    for (int t = 1; t < threads; ++t) started[t] = pthread_create(&tid[t], NULL, dgrad_rows, &jobs[t]) == 0;
    dgrad_rows(&jobs[0]);
    for (int t = 1; t < threads; ++t) {
        if (started[t]) pthread_join(tid[t], NULL);
        else dgrad_rows(&jobs[t]);
    }
    free(started);
    free(tid);
    free(jobs);
    return 0;
}

static double* widen16_all(const uint16_t* v, int64_t count)
{
    double* out = (double*)malloc(sizeof(double) * (size_t)(count > 0 ? count : 1));
    if (!out) return NULL;
    for (int64_t i = 0; i < count; ++i) out[i] = widen16(v[i]);
    return out;
}

/* As oracle_dgrad_f64 with bf16 (bit pattern) dy and weights. */
int oracle_dgrad_bf16(const int64_t dims[7], const int64_t opts[7], const uint16_t* dy, const uint16_t* wt,
                      double* dx, double* mass, int threads)
{
    dgrad_shape sp;
    if (dgrad_make_shape(&sp, dims, opts)) return 1;
    double* dyd = widen16_all(dy, sp.n * sp.p * sp.q * sp.k);
    double* wd = widen16_all(wt, sp.k * sp.r * sp.s * (sp.c / sp.g));
    int rc = 2;
    if (dyd && wd) rc = oracle_dgrad_f64(dims, opts, dyd, wd, dx, mass, threads);
    free(dyd);
    free(wd);
    return rc;
}

/*
 * Selected elements only: out[i] = dx[m_idx[i]][c_idx[i]] of the gradient viewed as
 * [N*H*W][C] (m = (n*H + h)*W + w); mass[i] (may be NULL) the sum of |terms|.  Double
 * inputs.  Returns 0, or 1 on invalid arguments / indices.
 */
int oracle_dgrad_points_f64(const int64_t dims[7], const int64_t opts[7], const double* dy, const double* wt,
                            const int64_t* m_idx, const int64_t* c_idx, int64_t npts, double* out, double* mass)
{
    dgrad_shape sp;
    if (dgrad_make_shape(&sp, dims, opts)) return 1;
    const int64_t rows = sp.n * sp.h * sp.w;
    for (int64_t i = 0; i < npts; ++i)
        if (m_idx[i] < 0 || m_idx[i] >= rows || c_idx[i] < 0 || c_idx[i] >= sp.c) return 1;
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t m = m_idx[i];
        const int64_t w = m % sp.w, h = (m / sp.w) % sp.h, n = m / (sp.w * sp.h);
        double a = 0.0;
        out[i] = dgrad_point(&sp, dy, wt, n, h, w, c_idx[i], &a);
        if (mass) mass[i] = a;
    }
    return 0;
}
