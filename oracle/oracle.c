/*
 * oracle.c -- plain fp64 CPU oracle for differentiable Fourier-slice projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file: only the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header or constant with the CUDA library.
 *
 * Source of the method: the web summaries of "torch-projectors: A High-Performance
 * Differentiable Projection Library for PyTorch" (gist.science; Spanish, Dutch, French
 * and Hindi pages of the same preprint).  The sections cited below are:
 *   [Method/RFFT]     the pages' Method section, bullet on PyTorch's RFFT format with
 *                     FFTW conventions (half spectrum, no intermediate format change);
 *   [Method/Interp]   Method section, interpolation bullet: linear (bilinear/trilinear)
 *                     and Catmull-Rom cubic with a = -0.5, C1 and exact at control points;
 *   [Method/Friedel]  Method section, Friedel bullet: F(-k) = conj F(k) for real
 *                     functions, no double counting on the zero-frequency axis;
 *   [Method/Ops]      Method section, operations list: 2D->2D forward/backward, 3D->2D
 *                     forward (central slice theorem), 2D->3D backward (accumulation);
 *                     each op supports rotation, translation by phase modulation and
 *                     weight accumulation;
 *   [Method/Shifts]   Method section (Dutch page), shifts by Fourier phase modulation;
 *   [Method/Grad]     Method section, differentiation bullet: gradients for inputs,
 *                     rotation matrices and shifts, without stored intermediates.
 *
 * The pages give no formulas.  The readings taken where they are silent are:
 *   - layout: full (non-half) axes are either FFTW order (index i holds frequency i for
 *     i < D/2, else i - D) or centered (index i holds i - D/2); the half axis x holds
 *     frequencies 0..D/2 in both;
 *   - output pixel (i, j) has kx = j and ky = frequency of row i; it is kept iff
 *     kx^2 + ky^2 <= rc^2 (rc = Do/2 when cutoff < 0), else it is zero;
 *   - sample coordinate c = o * R * q with q = (kx, ky, 0) in 3D or (kx, ky) in 2D,
 *     R row-major, vector order (x, y, z) <-> tensor axes (last, middle, first);
 *   - v(c) = sum_t w(c - t) V_ext(t) with separable kernel weights over the taps
 *     floor(c) + {0, 1} (linear) or floor(c) + {-1, 0, 1, 2} (cubic);
 *   - V_ext(t) = V[t] if t_x >= 0, conj(V[-t]) if t_x < 0, and zero where the stored
 *     frequency lies outside x in [0, Dv/2], y, z in [-Dv/2, Dv/2 - 1];
 *   - output y = v * exp(-2 pi i (kx sx + ky sy) / Do);
 *   - gradients follow PyTorch's convention for complex tensors
 *     (dL/dRe + i dL/dIm); a real parameter's gradient is Re(conj(g) dy/dtheta);
 *   - the linear kernel's derivative at a kink is taken from the cell
 *     [floor(c), floor(c) + 1] that holds the sample.
 *
 * Arrays are C-contiguous fp64 (complex = interleaved re, im = C99 double complex):
 *   rec     [n_rec][Dv][Dv][Dv/2+1] (3D) or [n_rec][Dv][Dv/2+1] (2D)
 *   images  [n_rec][n_pose][Do][Do/2+1]
 *   rot     [n_rot][n_pose][k][k], n_rot in {1, n_rec} (1 = shared by every rec)
 *   shift   [n_sh][n_pose][2] = (sx, sy), n_sh in {1, n_rec}; may be NULL
 */
#include <complex.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_LINEAR 0
#define ORC_CUBIC 1
#define ORC_FFTW 0
#define ORC_CENTERED 1

typedef struct {
    int ndim;           /* 2 or 3 */
    int n_rec, n_pose;  /* items are (rec, pose) pairs */
    int n_rot, n_sh;    /* 1 (shared) or n_rec */
    long Dv, Do;        /* box sizes of the reconstruction and of the images */
    int interp, layout;
    double o;           /* oversampling: coordinate scale */
    double rc2;         /* squared cutoff radius in image frequency units */
} geom;

/* ---------------------------------------------------------------- indexing ---- */

/* Frequency held at storage index i of a full axis of length D ([Method/RFFT]). */
static long freq_of_index(long i, long D, int layout)
{
    if (layout == ORC_CENTERED) return i - D / 2;
    return i < D / 2 ? i : i - D;
}

/* Storage index of frequency f on a full axis of length D; -1 when f is not stored. */
static long index_of_freq(long f, long D, int layout)
{
    if (f < -D / 2 || f > D / 2 - 1) return -1;
    if (layout == ORC_CENTERED) return f + D / 2;
    return f >= 0 ? f : f + D;
}

/* Where the extended spectrum value V_ext(t) is stored ([Method/Friedel]).  Returns the
 * element offset within one reconstruction, or -1 when V_ext(t) is zero; *mirror is set
 * to 1 when the stored value must be conjugated (t_x < 0 reads conj V[-t]). */
static long locate(const geom* g, long tx, long ty, long tz, int* mirror)
{
    long H = g->Dv / 2 + 1, iy, iz;
    *mirror = tx < 0;
    if (*mirror) {
        tx = -tx;
        ty = -ty;
        tz = -tz;
    }
    if (tx > g->Dv / 2) return -1;
    iy = index_of_freq(ty, g->Dv, g->layout);
    if (iy < 0) return -1;
    if (g->ndim == 2) return iy * H + tx;
    iz = index_of_freq(tz, g->Dv, g->layout);
    if (iz < 0) return -1;
    return (iz * g->Dv + iy) * H + tx;
}

/* ------------------------------------------------------------ interpolation ---- */

/* Interpolation kernel ([Method/Interp]): the tent 1 - |d| for linear, and Keys' cubic
 * convolution kernel with a = -1/2 (Catmull-Rom) for cubic. */
static double kernel(double d, int interp)
{
    const double a = -0.5;
    double u = fabs(d);
    if (interp == ORC_LINEAR) return u < 1.0 ? 1.0 - u : 0.0;
    if (u <= 1.0) return (a + 2.0) * u * u * u - (a + 3.0) * u * u + 1.0;
    if (u < 2.0) return a * u * u * u - 5.0 * a * u * u + 8.0 * a * u - 4.0 * a;
    return 0.0;
}

/* d kernel / d d.  For the tent the value at a kink is the one of the cell that holds
 * the sample: d in [0, 1) (tap floor(c)) gives -1, d in [-1, 0) (tap floor(c)+1) gives +1. */
static double kernel_deriv(double d, int interp)
{
    const double a = -0.5;
    double u = fabs(d), s = d < 0.0 ? -1.0 : 1.0;
    if (interp == ORC_LINEAR) {
        if (d >= 0.0 && d < 1.0) return -1.0;
        if (d >= -1.0 && d < 0.0) return 1.0;
        return 0.0;
    }
    if (u <= 1.0) return s * (3.0 * (a + 2.0) * u * u - 2.0 * (a + 3.0) * u);
    if (u < 2.0) return s * (3.0 * a * u * u - 10.0 * a * u + 8.0 * a);
    return 0.0;
}

/* Taps of one axis for coordinate c: t[k], w[k] = kernel(c - t[k]), dw[k] = kernel'(c - t[k]). */
static int axis_taps(double c, int interp, long t[4], double w[4], double dw[4])
{
    long b = (long)floor(c);
    int n = interp == ORC_LINEAR ? 2 : 4;
    long first = interp == ORC_LINEAR ? b : b - 1;
    for (int k = 0; k < n; ++k) {
        t[k] = first + k;
        w[k] = kernel(c - (double)t[k], interp);
        dw[k] = kernel_deriv(c - (double)t[k], interp);
    }
    return n;
}

/* v(c) = sum_t w(c - t) V_ext(t); when dv != NULL also dv[a] = dv/dc_a. */
static double complex sample(const geom* g, const double complex* V, const double c[3],
                             double complex dv[3])
{
    long tx[4], ty[4], tz[4] = {0, 0, 0, 0};
    double wx[4], wy[4], wz[4] = {1, 0, 0, 0}, dwx[4], dwy[4], dwz[4] = {0, 0, 0, 0};
    int nx = axis_taps(c[0], g->interp, tx, wx, dwx);
    int ny = axis_taps(c[1], g->interp, ty, wy, dwy);
    int nz = g->ndim == 3 ? axis_taps(c[2], g->interp, tz, wz, dwz) : 1;
    double complex v = 0.0;
    if (dv) dv[0] = dv[1] = dv[2] = 0.0;
    for (int a = 0; a < nz; ++a)
        for (int b = 0; b < ny; ++b)
            for (int k = 0; k < nx; ++k) {
                int mirror;
                long off = locate(g, tx[k], ty[b], tz[a], &mirror);
                double complex val;
                if (off < 0) continue;
                val = mirror ? conj(V[off]) : V[off];
                v += wz[a] * wy[b] * wx[k] * val;
                if (dv) {
                    dv[0] += wz[a] * wy[b] * dwx[k] * val;
                    dv[1] += wz[a] * dwy[b] * wx[k] * val;
                    dv[2] += dwz[a] * wy[b] * wx[k] * val;
                }
            }
    return v;
}

/* Adjoint of sample(): for every tap, R[t] += w(c - t) * val when t_x >= 0, and
 * R[-t] += conj(w(c - t) * val) when t_x < 0.  When W != NULL the real weight volume
 * receives W[t or -t] += w(c - t) * wt (no conjugation: the weight is real). */
static void scatter(const geom* g, double complex* R, double* W, const double c[3],
                    double complex val, double wt)
{
    long tx[4], ty[4], tz[4] = {0, 0, 0, 0};
    double wx[4], wy[4], wz[4] = {1, 0, 0, 0}, dwx[4], dwy[4], dwz[4];
    int nx = axis_taps(c[0], g->interp, tx, wx, dwx);
    int ny = axis_taps(c[1], g->interp, ty, wy, dwy);
    int nz = g->ndim == 3 ? axis_taps(c[2], g->interp, tz, wz, dwz) : 1;
    for (int a = 0; a < nz; ++a)
        for (int b = 0; b < ny; ++b)
            for (int k = 0; k < nx; ++k) {
                int mirror;
                long off = locate(g, tx[k], ty[b], tz[a], &mirror);
                double w = wz[a] * wy[b] * wx[k];
                if (off < 0) continue;
                if (R) R[off] += mirror ? conj(w * val) : w * val;
                if (W) W[off] += w * wt;
            }
}

/* ------------------------------------------------------------- per pixel ---- */

typedef struct {
    long kx, ky;
    int kept;
    double c[3];
    double complex phase; /* exp(-2 pi i (kx sx + ky sy) / Do) */
} pixel;

/* Pixel (i, j) of an image of item (r, p): frequencies, cutoff, rotated coordinate
 * c = o R q ([Method/Ops], central slice theorem) and the shift phase ([Method/Shifts]). */
static pixel make_pixel(const geom* g, const double* R, const double* s, long i, long j)
{
    pixel px;
    int k = g->ndim;
    double q[3];
    px.kx = j;
    px.ky = freq_of_index(i, g->Do, g->layout);
    px.kept = (double)(px.kx * px.kx + px.ky * px.ky) <= g->rc2;
    q[0] = (double)px.kx;
    q[1] = (double)px.ky;
    q[2] = 0.0;
    for (int a = 0; a < 3; ++a) {
        px.c[a] = 0.0;
        if (a < k)
            for (int b = 0; b < k; ++b) px.c[a] += g->o * R[a * k + b] * q[b];
    }
    px.phase = 1.0;
    if (s) {
        double turns = ((double)px.kx * s[0] + (double)px.ky * s[1]) / (double)g->Do;
        px.phase = cexp(-2.0 * M_PI * I * turns);
    }
    return px;
}

static const double* item_rot(const geom* g, const double* rot, long r, long p)
{
    long k = g->ndim;
    return rot + ((g->n_rot == 1 ? 0 : r) * g->n_pose + p) * k * k;
}

static const double* item_shift(const geom* g, const double* shift, long r, long p)
{
    if (!shift) return NULL;
    return shift + ((g->n_sh == 1 ? 0 : r) * g->n_pose + p) * 2;
}

static long rec_size(const geom* g)
{
    long H = g->Dv / 2 + 1;
    return g->ndim == 3 ? g->Dv * g->Dv * H : g->Dv * H;
}

static int make_geom(geom* g, int ndim, int n_rec, int Dv, int n_rot, int n_pose, int n_sh,
                     int Do, int interp, int layout, double oversampling, double cutoff)
{
    if (ndim != 2 && ndim != 3) return 1;
    if (n_rec < 0 || n_pose < 0 || Dv < 2 || Do < 2 || (Dv & 1) || (Do & 1)) return 2;
    if (n_rot != 1 && n_rot != n_rec) return 2;
    if (n_sh != 1 && n_sh != n_rec) return 2;
    if (interp != ORC_LINEAR && interp != ORC_CUBIC) return 3;
    if (layout != ORC_FFTW && layout != ORC_CENTERED) return 3;
    if (!(oversampling > 0.0)) return 3;
    g->ndim = ndim;
    g->n_rec = n_rec;
    g->n_pose = n_pose;
    g->n_rot = n_rot;
    g->n_sh = n_sh;
    g->Dv = Dv;
    g->Do = Do;
    g->interp = interp;
    g->layout = layout;
    g->o = oversampling;
    cutoff = cutoff < 0.0 ? 0.5 * Do : cutoff;
    g->rc2 = cutoff * cutoff;
    return 0;
}

/* ------------------------------------------------------------ public API ---- */

/* Forward projection ([Method/Ops]): 3D->2D central slices (ndim = 3) or 2D->2D rotation
 * (ndim = 2).  out [n_rec][n_pose][Do][Do/2+1] is overwritten.  Returns 0 or an error. */
int orc_project(int ndim, const double complex* rec, int n_rec, int Dv, const double* rot,
                int n_rot, int n_pose, const double* shift, int n_sh, double complex* out,
                int Do, int interp, int layout, double oversampling, double cutoff,
                int nthreads)
{
    geom g;
    int err = make_geom(&g, ndim, n_rec, Dv, n_rot, n_pose, n_sh, Do, interp, layout,
                        oversampling, cutoff);
    long H = g.Do / 2 + 1, n_items = (long)n_rec * n_pose;
    if (err) return err;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (long it = 0; it < n_items; ++it) {
        long r = it / n_pose, p = it % n_pose;
        const double* R = item_rot(&g, rot, r, p);
        const double* s = item_shift(&g, shift, r, p);
        const double complex* V = rec + r * rec_size(&g);
        double complex* y = out + it * g.Do * H;
        for (long i = 0; i < g.Do; ++i)
            for (long j = 0; j < H; ++j) {
                pixel px = make_pixel(&g, R, s, i, j);
                y[i * H + j] = px.kept ? sample(&g, V, px.c, NULL) * px.phase : 0.0;
            }
    }
    return 0;
}

/* Forward projection at a list of pixels only: for each n, item = items[n] (= r * n_pose
 * + p) and pixel index pix[n] (= i * (Do/2+1) + j).  vals[n] receives the output value. */
int orc_project_samples(int ndim, const double complex* rec, int n_rec, int Dv,
                        const double* rot, int n_rot, int n_pose, const double* shift,
                        int n_sh, int Do, int interp, int layout, double oversampling,
                        double cutoff, long n, const long* items, const long* pix,
                        double complex* vals, int nthreads)
{
    geom g;
    int err = make_geom(&g, ndim, n_rec, Dv, n_rot, n_pose, n_sh, Do, interp, layout,
                        oversampling, cutoff);
    long H = g.Do / 2 + 1;
    if (err) return err;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads > 0 ? nthreads : 1)
    for (long m = 0; m < n; ++m) {
        long r = items[m] / n_pose, p = items[m] % n_pose;
        pixel px = make_pixel(&g, item_rot(&g, rot, r, p), item_shift(&g, shift, r, p),
                              pix[m] / H, pix[m] % H);
        vals[m] = px.kept ? sample(&g, rec + r * rec_size(&g), px.c, NULL) * px.phase : 0.0;
    }
    return 0;
}

/* Per-thread private accumulators for the scatters, summed at the end: the sum is the
 * same as a serial scatter up to the order of fp64 additions. */
static int scatter_threads(int nthreads, long elems)
{
    long cap = (2L << 30) / (long)(elems * (sizeof(double complex) + sizeof(double)) + 1);
    int t = nthreads > 0 ? nthreads : 1;
    if (cap < 1) cap = 1;
    return t < cap ? t : (int)cap;
}

/* Back-projection ([Method/Ops]): 2D->3D insertion (ndim = 3) or 2D->2D accumulation
 * (ndim = 2), the adjoint of orc_project, plus the weight accumulation.  ADDS into
 * rec_out (complex) and wrec_out (real; both nullable).  The data receive
 * proj * conj(phase) with the scatter rule; the weights receive the real per-pixel
 * weight (1 when weights == NULL) with the same interpolation weights and no phase. */
int orc_backproject(int ndim, const double complex* proj, const double* weights, int n_rec,
                    int Do, const double* rot, int n_rot, int n_pose, const double* shift,
                    int n_sh, double complex* rec_out, double* wrec_out, int Dv, int interp,
                    int layout, double oversampling, double cutoff, int nthreads)
{
    geom g;
    int err = make_geom(&g, ndim, n_rec, Dv, n_rot, n_pose, n_sh, Do, interp, layout,
                        oversampling, cutoff);
    long H = g.Do / 2 + 1, n_items = (long)n_rec * n_pose, rs;
    int nt;
    double complex* accR;
    double* accW;
    if (err) return err;
    rs = rec_size(&g);
    nt = scatter_threads(nthreads, rs * n_rec);
    accR = calloc((size_t)nt * rs * n_rec, sizeof(double complex));
    accW = calloc((size_t)nt * rs * n_rec, sizeof(double));
    if (!accR || !accW) {
        free(accR);
        free(accW);
        return 4;
    }
#pragma omp parallel num_threads(nt)
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
#pragma omp for schedule(dynamic, 1)
        for (long it = 0; it < n_items; ++it) {
            long r = it / n_pose, p = it % n_pose;
            const double* R = item_rot(&g, rot, r, p);
            const double* s = item_shift(&g, shift, r, p);
            double complex* aR = accR + ((long)tid * n_rec + r) * rs;
            double* aW = accW + ((long)tid * n_rec + r) * rs;
            for (long i = 0; i < g.Do; ++i)
                for (long j = 0; j < H; ++j) {
                    long e = it * g.Do * H + i * H + j;
                    pixel px = make_pixel(&g, R, s, i, j);
                    if (!px.kept) continue;
                    scatter(&g, aR, aW, px.c, proj[e] * conj(px.phase),
                            weights ? weights[e] : 1.0);
                }
        }
    }
    for (int t = 0; t < nt; ++t)
        for (long e = 0; e < rs * n_rec; ++e) {
            if (rec_out) rec_out[e] += accR[(long)t * rs * n_rec + e];
            if (wrec_out) wrec_out[e] += accW[(long)t * rs * n_rec + e];
        }
    free(accR);
    free(accW);
    return 0;
}

/* Backward of orc_project ([Method/Grad]) for the upstream gradient grad_out:
 *   grad_rec   = the real-linear transpose of the projection applied to grad_out,
 *   grad_rot   [n_rot][n_pose][k][k]: dL/dR[a][b] = o q_b Re(conj(g') dv/dc_a),
 *              g' = g conj(phase); summed over recs when n_rot = 1,
 *   grad_shift [n_sh][n_pose][2]: dL/ds = Re(conj(g) y (-2 pi i k / Do)), k = (kx, ky).
 * Every output is nullable and, when given, overwritten. */
int orc_project_backward(int ndim, const double complex* rec, int n_rec, int Dv,
                         const double* rot, int n_rot, int n_pose, const double* shift,
                         int n_sh, const double complex* grad_out, int Do,
                         double complex* grad_rec, double* grad_rot, double* grad_shift,
                         int interp, int layout, double oversampling, double cutoff,
                         int nthreads)
{
    geom g;
    int err = make_geom(&g, ndim, n_rec, Dv, n_rot, n_pose, n_sh, Do, interp, layout,
                        oversampling, cutoff);
    long H = g.Do / 2 + 1, n_items = (long)n_rec * n_pose, k = ndim;
    double *item_grot, *item_gsh;
    if (err) return err;
    if (grad_rec) {
        memset(grad_rec, 0, sizeof(double complex) * (size_t)(rec_size(&g) * n_rec));
        err = orc_backproject(ndim, grad_out, NULL, n_rec, Do, rot, n_rot, n_pose, shift,
                              n_sh, grad_rec, NULL, Dv, interp, layout, oversampling, cutoff,
                              nthreads);
        if (err) return err;
    }
    if (!grad_rot && !grad_shift) return 0;
    /* per-item gradients first, then the sum over recs for shared parameters */
    item_grot = calloc((size_t)(n_items * k * k + 1), sizeof(double));
    item_gsh = calloc((size_t)(n_items * 2 + 1), sizeof(double));
    if (!item_grot || !item_gsh) {
        free(item_grot);
        free(item_gsh);
        return 4;
    }
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (long it = 0; it < n_items; ++it) {
        long r = it / n_pose, p = it % n_pose;
        const double* R = item_rot(&g, rot, r, p);
        const double* s = item_shift(&g, shift, r, p);
        const double complex* V = rec + r * rec_size(&g);
        for (long i = 0; i < g.Do; ++i)
            for (long j = 0; j < H; ++j) {
                double complex gy = grad_out[it * g.Do * H + i * H + j], dv[3], v, gp;
                double q[2];
                pixel px = make_pixel(&g, R, s, i, j);
                if (!px.kept) continue;
                v = sample(&g, V, px.c, dv);
                gp = gy * conj(px.phase);
                q[0] = (double)px.kx;
                q[1] = (double)px.ky;
                for (long a = 0; a < k; ++a)
                    for (long b = 0; b < 2; ++b)
                        item_grot[it * k * k + a * k + b] += g.o * q[b] * creal(conj(gp) * dv[a]);
                if (s) {
                    double complex y = v * px.phase;
                    for (long b = 0; b < 2; ++b)
                        item_gsh[it * 2 + b] +=
                            creal(conj(gy) * y * (-2.0 * M_PI * I * q[b] / (double)g.Do));
                }
            }
    }
    if (grad_rot) {
        memset(grad_rot, 0, sizeof(double) * (size_t)(n_rot * (long)n_pose * k * k));
        for (long it = 0; it < n_items; ++it) {
            long r = it / n_pose, p = it % n_pose, dst = (n_rot == 1 ? 0 : r) * n_pose + p;
            for (long e = 0; e < k * k; ++e) grad_rot[dst * k * k + e] += item_grot[it * k * k + e];
        }
    }
    if (grad_shift) {
        memset(grad_shift, 0, sizeof(double) * (size_t)(n_sh * (long)n_pose * 2));
        if (shift)
            for (long it = 0; it < n_items; ++it) {
                long r = it / n_pose, p = it % n_pose, dst = (n_sh == 1 ? 0 : r) * n_pose + p;
                for (long e = 0; e < 2; ++e) grad_shift[dst * 2 + e] += item_gsh[it * 2 + e];
            }
    }
    free(item_grot);
    free(item_gsh);
    return 0;
}

/* Interpolation weights and their derivatives for one coordinate, exposed for the
 * tests that pin the kernel itself (control points, partition of unity, C1). */
int orc_axis_weights(double c, int interp, long* t, double* w, double* dw)
{
    return axis_taps(c, interp, t, w, dw);
}
