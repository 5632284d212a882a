/*
 * Float64 CPU oracle for the ray-driven Siddon projector pair.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, header
 * or constant with the CUDA library; both are fed from the seeded input
 * generators only.
 *
 * What it computes (diffct release pages, my.diffend.io):
 *   - forward: p(R) = sum over cells of |R n cell| * f(cell), the exact line
 *     integral of the cell-constant image ("exact adjoint pair for the
 *     cell-constant Siddon model", diffct 2.1.0 -> 2.2.1, README "Matched
 *     operators"; "Siddon path sum; matched adjoint", diffct 2.4.1 -> 2.4.2,
 *     docs/video/README.md, shot "Autograd");
 *   - backward: g(cell) = sum over rays of |R n cell| * y(R), the transpose;
 *   - lengths in physical units with per-axis spacing (diffct 2.4.3 -> 2.4.4,
 *     CHANGELOG 2.4.4 "Added": per-axis voxel spacing, physical length units).
 *
 * Method: the textbook parametric Siddon traversal in float64 -- clip the ray to
 * the box, merge the plane-crossing parameters of the three axes, and give each
 * positive-length piece to the cell that contains its midpoint.  A second,
 * independent brute-force path clips the ray against every cell's box.  A third
 * path (voxel-driven) evaluates the transpose at chosen voxels by clipping every
 * candidate ray of every view against that voxel's box.
 *
 * Readings where the pages are silent:
 *   - pixel centre: det_centre + (iu - (n_u-1)/2 + offset_u) * pitch_u * u
 *                              + (iv - (n_v-1)/2 + offset_v) * pitch_v * v;
 *   - divergent ray: the segment source -> pixel centre (t in [0, 1]);
 *     parallel ray: the full line through the pixel centre along src (t free);
 *   - cell (i, j, k) is [o + i d, o + (i+1) d) per axis; a ray lying exactly in a
 *     face plane belongs to the cell on the + side of that plane.
 * Every floating-point value is a double; inputs are float32 promoted exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int beam;            /* 0 = parallel, 1 = divergent (fan / cone) */
    int n_views, n_u, n_v;
    const float *src;    /* (n_views, 3): source, or unit ray direction (parallel) */
    const float *det_centre;
    const float *det_u;
    const float *det_v;
    double pitch_u, pitch_v, offset_u, offset_v;
    int n[3];            /* cells along x, y, z */
    int pad_;
    double d[3];         /* spacing along x, y, z */
    double o[3];         /* world position of the min corner of cell (0, 0, 0) */
    const float *offsets;  /* NULL (flat detector) or per-pixel offsets (t, s, e): */
    int offsets_per_view;  /* 0: (n_v, n_u, 3) shared by all views; 1: (n_views, n_v, n_u, 3) */
    int pad2_;
} ora_ctx;

static int ora_threads(int requested)
{
#ifdef _OPENMP
    if (requested > 0) return requested;
    return omp_get_max_threads();
#else
    (void)requested;
    return 1;
#endif
}

/* The ray of detector sample `ray` (view-major, then v, then u).  Flat
 * detector: pixel = centre + a u + b v with a, b the pitch grid.  Curved
 * (per-pixel offsets (t, s, e), shared by all views or one table per view; the
 * pages' surface composition, diffct 2.4.1 -> 2.4.2, kernels/surface_geometry.py
 * `compose_surface`: point = centre + tangent u + vertical v + depth n, with
 * view and pixel batches of offsets): pixel = centre + t u + s v + e n,
 * n = (u x v) / |u x v|. */
static void ora_ray(const ora_ctx *c, long ray, double X0[3], double r[3],
                    double *tlo, double *thi)
{
    long per_view = (long)c->n_u * c->n_v;
    long view = ray / per_view;
    long pix = ray % per_view;
    long iv = pix / c->n_u, iu = pix % c->n_u;
    const float *S = c->src + 3 * view, *C = c->det_centre + 3 * view;
    const float *U = c->det_u + 3 * view, *V = c->det_v + 3 * view;
    double P[3];
    if (c->offsets) {
        const float *q = c->offsets + 3 * (c->offsets_per_view ? ray : pix);
        double u[3] = {U[0], U[1], U[2]}, v[3] = {V[0], V[1], V[2]};
        double n[3] = {u[1] * v[2] - u[2] * v[1], u[2] * v[0] - u[0] * v[2],
                       u[0] * v[1] - u[1] * v[0]};
        double nn = sqrt(n[0] * n[0] + n[1] * n[1] + n[2] * n[2]);
        for (int ax = 0; ax < 3; ++ax)
            P[ax] = (double)C[ax] + (double)q[0] * u[ax] + (double)q[1] * v[ax] +
                    (double)q[2] * (n[ax] / nn);
    } else {
        double a = ((double)iu - 0.5 * (double)(c->n_u - 1) + c->offset_u) * c->pitch_u;
        double b = ((double)iv - 0.5 * (double)(c->n_v - 1) + c->offset_v) * c->pitch_v;
        for (int ax = 0; ax < 3; ++ax)
            P[ax] = (double)C[ax] + a * (double)U[ax] + b * (double)V[ax];
    }
    if (c->beam == 1) {
        for (int ax = 0; ax < 3; ++ax) {
            X0[ax] = (double)S[ax];
            r[ax] = P[ax] - (double)S[ax];
        }
        *tlo = 0.0;
        *thi = 1.0;
    } else {
        for (int ax = 0; ax < 3; ++ax) {
            X0[ax] = P[ax];
            r[ax] = (double)S[ax];
        }
        *tlo = -INFINITY;
        *thi = INFINITY;
    }
}

static double ora_norm(const double r[3])
{
    return sqrt(r[0] * r[0] + r[1] * r[1] + r[2] * r[2]);
}

/* Parameter interval of the line X0 + t r inside the cell box [lo, hi) (in cell
 * indices), intersected with [tlo, thi].  Returns 0 when empty. */
static int ora_clip_cells(const ora_ctx *c, const double X0[3], const double r[3],
                          double tlo, double thi, const int lo[3], const int hi[3],
                          double *amin, double *amax)
{
    double a0 = tlo, a1 = thi;
    for (int ax = 0; ax < 3; ++ax) {
        double p0 = c->o[ax] + (double)lo[ax] * c->d[ax];
        double p1 = c->o[ax] + (double)hi[ax] * c->d[ax];
        if (r[ax] == 0.0) {
            if (!(X0[ax] >= p0 && X0[ax] < p1)) return 0;
        } else {
            double t0 = (p0 - X0[ax]) / r[ax], t1 = (p1 - X0[ax]) / r[ax];
            a0 = fmax(a0, fmin(t0, t1));
            a1 = fmin(a1, fmax(t0, t1));
        }
    }
    *amin = a0;
    *amax = a1;
    return a0 < a1;
}

/*
 * Siddon traversal of one ray inside the cell box [lo, hi).  Writes the linear
 * cell index ((k * ny + j) * nx + i) and the physical length of every
 * positive-length piece; returns the number of pieces.  `buf` must hold
 * (hi-lo summed over axes) + 6 doubles; cells/lens the same count.
 */
static int ora_trace(const ora_ctx *c, const double X0[3], const double r[3],
                     double tlo, double thi, const int lo[3], const int hi[3],
                     double *buf, long *cells, double *lens)
{
    double amin, amax;
    if (!ora_clip_cells(c, X0, r, tlo, thi, lo, hi, &amin, &amax)) return 0;

    /* Per-axis crossing parameters strictly inside (amin, amax), each in
     * increasing order, then a three-way merge. */
    double *seq[3];
    int len[3], pos[3];
    double *next = buf;
    for (int ax = 0; ax < 3; ++ax) {
        seq[ax] = next;
        len[ax] = 0;
        pos[ax] = 0;
        if (r[ax] == 0.0) continue;
        int count = hi[ax] - lo[ax] + 1;
        for (int m = 0; m < count; ++m) {
            int k = r[ax] > 0.0 ? lo[ax] + m : hi[ax] - m;
            double t = (c->o[ax] + (double)k * c->d[ax] - X0[ax]) / r[ax];
            if (t > amin && t < amax) seq[ax][len[ax]++] = t;
        }
        next += len[ax];
    }
    double norm = ora_norm(r);
    double prev = amin;
    int out = 0;
    for (;;) {
        double t = amax;
        int which = -1;
        for (int ax = 0; ax < 3; ++ax)
            if (pos[ax] < len[ax] && seq[ax][pos[ax]] < t) {
                t = seq[ax][pos[ax]];
                which = ax;
            }
        if (t > prev) {
            double mid = 0.5 * (prev + t);
            long idx[3];
            for (int ax = 0; ax < 3; ++ax) {
                long q = (long)floor((X0[ax] + mid * r[ax] - c->o[ax]) / c->d[ax]);
                if (q < lo[ax]) q = lo[ax];
                if (q > hi[ax] - 1) q = hi[ax] - 1;
                idx[ax] = q;
            }
            cells[out] = (idx[2] * c->n[1] + idx[1]) * c->n[0] + idx[0];
            lens[out] = (t - prev) * norm;
            ++out;
            prev = t;
        }
        if (which < 0) break;
        pos[which]++;
    }
    return out;
}

static long ora_n_rays(const ora_ctx *c)
{
    return (long)c->n_views * c->n_u * c->n_v;
}

static int ora_buf_len(const ora_ctx *c)
{
    return c->n[0] + c->n[1] + c->n[2] + 8;
}

/* Forward projection of rays [ray0, ray1): sino[ray - ray0] = sum len * vol. */
int ora_forward(const ora_ctx *c, const float *vol, double *sino, long ray0, long ray1,
                int nthreads)
{
    int T = ora_threads(nthreads);
    int B = ora_buf_len(c);
    int err = 0;
#pragma omp parallel num_threads(T)
    {
        double *buf = (double *)malloc(sizeof(double) * B);
        long *cells = (long *)malloc(sizeof(long) * B);
        double *lens = (double *)malloc(sizeof(double) * B);
        if (!buf || !cells || !lens) {
#pragma omp atomic write
            err = 1;
        } else {
            int lo[3] = {0, 0, 0};
#pragma omp for schedule(dynamic, 64)
            for (long ray = ray0; ray < ray1; ++ray) {
                double X0[3], r[3], tlo, thi;
                ora_ray(c, ray, X0, r, &tlo, &thi);
                int n = ora_trace(c, X0, r, tlo, thi, lo, c->n, buf, cells, lens);
                double acc = 0.0;
                for (int s = 0; s < n; ++s) acc += lens[s] * (double)vol[cells[s]];
                sino[ray - ray0] = acc;
            }
        }
        free(buf);
        free(cells);
        free(lens);
    }
    return err;
}

/* Forward projection of an explicit list of rays. */
int ora_forward_rays(const ora_ctx *c, const float *vol, const long *rays, long count,
                     double *out, int nthreads)
{
    int T = ora_threads(nthreads);
    int B = ora_buf_len(c);
    int err = 0;
#pragma omp parallel num_threads(T)
    {
        double *buf = (double *)malloc(sizeof(double) * B);
        long *cells = (long *)malloc(sizeof(long) * B);
        double *lens = (double *)malloc(sizeof(double) * B);
        if (!buf || !cells || !lens) {
#pragma omp atomic write
            err = 1;
        } else {
            int lo[3] = {0, 0, 0};
#pragma omp for schedule(dynamic, 16)
            for (long q = 0; q < count; ++q) {
                double X0[3], r[3], tlo, thi;
                ora_ray(c, rays[q], X0, r, &tlo, &thi);
                int n = ora_trace(c, X0, r, tlo, thi, lo, c->n, buf, cells, lens);
                double acc = 0.0;
                for (int s = 0; s < n; ++s) acc += lens[s] * (double)vol[cells[s]];
                out[q] = acc;
            }
        }
        free(buf);
        free(cells);
        free(lens);
    }
    return err;
}

/*
 * Backprojection (transpose) of rays [ray0, ray1) into vol (zeroed first).
 * Deterministic without atomics: each thread owns a band of cells along one
 * axis (z when there are enough z cells, else y) and walks every ray clipped
 * to its band.  sino is indexed by ray - ray0.
 */
int ora_backward(const ora_ctx *c, const float *sino, double *vol, long ray0, long ray1,
                 int nthreads)
{
    int T = ora_threads(nthreads);
    int B = ora_buf_len(c);
    long nvox = (long)c->n[0] * c->n[1] * c->n[2];
    memset(vol, 0, sizeof(double) * nvox);
    int own = c->n[2] >= T ? 2 : (c->n[1] >= T ? 1 : 0);
    int bands = c->n[own] < T ? c->n[own] : T;
    int err = 0;
#pragma omp parallel num_threads(bands)
    {
        int t = 0;
#ifdef _OPENMP
        t = omp_get_thread_num();
#endif
        double *buf = (double *)malloc(sizeof(double) * B);
        long *cells = (long *)malloc(sizeof(long) * B);
        double *lens = (double *)malloc(sizeof(double) * B);
        if (!buf || !cells || !lens) {
#pragma omp atomic write
            err = 1;
        } else {
            int lo[3] = {0, 0, 0}, hi[3] = {c->n[0], c->n[1], c->n[2]};
            lo[own] = (int)((long)c->n[own] * t / bands);
            hi[own] = (int)((long)c->n[own] * (t + 1) / bands);
            for (long ray = ray0; ray < ray1 && hi[own] > lo[own]; ++ray) {
                double y = (double)sino[ray - ray0];
                double X0[3], r[3], tlo, thi;
                ora_ray(c, ray, X0, r, &tlo, &thi);
                int n = ora_trace(c, X0, r, tlo, thi, lo, hi, buf, cells, lens);
                for (int s = 0; s < n; ++s) vol[cells[s]] += lens[s] * y;
            }
        }
        free(buf);
        free(cells);
        free(lens);
    }
    return err;
}

/* Number of (ray, cell) pieces longer than min_len over rays [ray0, ray1).
 * min_len = 0 counts every positive-length piece; a small positive min_len
 * drops the numerically degenerate pieces of rays that cross a cell edge or
 * corner exactly (length 0 in exact arithmetic, rounding-sized here). */
int ora_segment_count(const ora_ctx *c, long ray0, long ray1, int nthreads, double min_len,
                      unsigned long long *out)
{
    int T = ora_threads(nthreads);
    int B = ora_buf_len(c);
    unsigned long long total = 0;
    int err = 0;
#pragma omp parallel num_threads(T) reduction(+ : total)
    {
        double *buf = (double *)malloc(sizeof(double) * B);
        long *cells = (long *)malloc(sizeof(long) * B);
        double *lens = (double *)malloc(sizeof(double) * B);
        if (!buf || !cells || !lens) {
#pragma omp atomic write
            err = 1;
        } else {
            int lo[3] = {0, 0, 0};
#pragma omp for schedule(dynamic, 256)
            for (long ray = ray0; ray < ray1; ++ray) {
                double X0[3], r[3], tlo, thi;
                ora_ray(c, ray, X0, r, &tlo, &thi);
                int n = ora_trace(c, X0, r, tlo, thi, lo, c->n, buf, cells, lens);
                for (int s = 0; s < n; ++s) total += lens[s] > min_len ? 1u : 0u;
            }
        }
        free(buf);
        free(cells);
        free(lens);
    }
    *out = total;
    return err;
}

/* Length of the line X0 + t r, t in [tlo, thi], inside the box [blo, bhi)
 * (half-open in the sense of the face-plane rule above). */
static double ora_clip_box(const double X0[3], const double r[3], double tlo, double thi,
                           const double blo[3], const double bhi[3])
{
    double a0 = tlo, a1 = thi;
    for (int ax = 0; ax < 3; ++ax) {
        if (r[ax] == 0.0) {
            if (!(X0[ax] >= blo[ax] && X0[ax] < bhi[ax])) return 0.0;
        } else {
            double t0 = (blo[ax] - X0[ax]) / r[ax], t1 = (bhi[ax] - X0[ax]) / r[ax];
            a0 = fmax(a0, fmin(t0, t1));
            a1 = fmin(a1, fmax(t0, t1));
        }
    }
    return a1 > a0 ? (a1 - a0) * ora_norm(r) : 0.0;
}

static void ora_cell_box(const ora_ctx *c, long i, long j, long k, double blo[3], double bhi[3])
{
    long idx[3] = {i, j, k};
    for (int ax = 0; ax < 3; ++ax) {
        blo[ax] = c->o[ax] + (double)idx[ax] * c->d[ax];
        bhi[ax] = c->o[ax] + (double)(idx[ax] + 1) * c->d[ax];
    }
}

/* Brute force forward: every ray clipped against every cell box.  O(cells) per
 * ray; tiny volumes only.  Shares no traversal logic with ora_trace. */
int ora_brute_forward(const ora_ctx *c, const float *vol, double *sino, int nthreads)
{
    int T = ora_threads(nthreads);
    long nr = ora_n_rays(c);
#pragma omp parallel for num_threads(T) schedule(dynamic, 16)
    for (long ray = 0; ray < nr; ++ray) {
        double X0[3], r[3], tlo, thi;
        ora_ray(c, ray, X0, r, &tlo, &thi);
        double acc = 0.0;
        for (long k = 0; k < c->n[2]; ++k)
            for (long j = 0; j < c->n[1]; ++j)
                for (long i = 0; i < c->n[0]; ++i) {
                    double blo[3], bhi[3];
                    ora_cell_box(c, i, j, k, blo, bhi);
                    double L = ora_clip_box(X0, r, tlo, thi, blo, bhi);
                    if (L > 0.0) acc += L * (double)vol[(k * c->n[1] + j) * c->n[0] + i];
                }
        sino[ray] = acc;
    }
    return 0;
}

/* Brute-force segment count: cells whose clipped length exceeds min_len. */
int ora_brute_count(const ora_ctx *c, double min_len, unsigned long long *out, int nthreads)
{
    int T = ora_threads(nthreads);
    long nr = ora_n_rays(c);
    unsigned long long total = 0;
#pragma omp parallel for num_threads(T) schedule(dynamic, 16) reduction(+ : total)
    for (long ray = 0; ray < nr; ++ray) {
        double X0[3], r[3], tlo, thi;
        ora_ray(c, ray, X0, r, &tlo, &thi);
        for (long k = 0; k < c->n[2]; ++k)
            for (long j = 0; j < c->n[1]; ++j)
                for (long i = 0; i < c->n[0]; ++i) {
                    double blo[3], bhi[3];
                    ora_cell_box(c, i, j, k, blo, bhi);
                    if (ora_clip_box(X0, r, tlo, thi, blo, bhi) > min_len) total++;
                }
    }
    *out = total;
    return 0;
}

/* Solve the 3x3 system M x = rhs (columns m0, m1, m2) by Cramer's rule. */
static int ora_solve3(const double m0[3], const double m1[3], const double m2[3],
                      const double rhs[3], double x[3])
{
    double det = m0[0] * (m1[1] * m2[2] - m1[2] * m2[1])
               - m1[0] * (m0[1] * m2[2] - m0[2] * m2[1])
               + m2[0] * (m0[1] * m1[2] - m0[2] * m1[1]);
    if (!(fabs(det) > 0.0)) return 0;
    double d0 = rhs[0] * (m1[1] * m2[2] - m1[2] * m2[1])
              - m1[0] * (rhs[1] * m2[2] - rhs[2] * m2[1])
              + m2[0] * (rhs[1] * m1[2] - rhs[2] * m1[1]);
    double d1 = m0[0] * (rhs[1] * m2[2] - rhs[2] * m2[1])
              - rhs[0] * (m0[1] * m2[2] - m0[2] * m2[1])
              + m2[0] * (m0[1] * rhs[2] - m0[2] * rhs[1]);
    double d2 = m0[0] * (m1[1] * rhs[2] - m1[2] * rhs[1])
              - m1[0] * (m0[1] * rhs[2] - m0[2] * rhs[1])
              + rhs[0] * (m0[1] * m1[2] - m0[2] * m1[1]);
    x[0] = d0 / det;
    x[1] = d1 / det;
    x[2] = d2 / det;
    return 1;
}

/*
 * Voxel-driven transpose at chosen voxels: out[q] = sum over every ray of
 * |ray n box(voxel q)| * sino(ray).  For each view the voxel's 8 corners are
 * projected onto the detector plane to bound the candidate pixels (with one
 * pixel of margin); every candidate ray is clipped against the voxel box.
 * voxels[q] is the linear index (k * ny + j) * nx + i.
 */
int ora_backward_voxels(const ora_ctx *c, const float *sino, const long *voxels, long count,
                        double *out, int nthreads)
{
    if (c->offsets) return 2;  /* the candidate-ray solve assumes a flat detector */
    int T = ora_threads(nthreads);
#pragma omp parallel for num_threads(T) schedule(dynamic, 1)
    for (long q = 0; q < count; ++q) {
        long v = voxels[q];
        long i = v % c->n[0], j = (v / c->n[0]) % c->n[1], k = v / ((long)c->n[0] * c->n[1]);
        double blo[3], bhi[3];
        ora_cell_box(c, i, j, k, blo, bhi);
        double acc = 0.0;
        for (long view = 0; view < c->n_views; ++view) {
            const float *S = c->src + 3 * view, *C = c->det_centre + 3 * view;
            const float *U = c->det_u + 3 * view, *V = c->det_v + 3 * view;
            double Ud[3], Vd[3], Sd[3], Cd[3];
            for (int ax = 0; ax < 3; ++ax) {
                Ud[ax] = U[ax];
                Vd[ax] = V[ax];
                Sd[ax] = S[ax];
                Cd[ax] = C[ax];
            }
            double umin = INFINITY, umax = -INFINITY, vmin = INFINITY, vmax = -INFINITY;
            int full = 0;
            for (int corner = 0; corner < 8 && !full; ++corner) {
                double X[3] = {(corner & 1) ? bhi[0] : blo[0], (corner & 2) ? bhi[1] : blo[1],
                               (corner & 4) ? bhi[2] : blo[2]};
                double m2[3], rhs[3], sol[3];
                for (int ax = 0; ax < 3; ++ax) {
                    if (c->beam == 1) {
                        m2[ax] = -(X[ax] - Sd[ax]);
                        rhs[ax] = Sd[ax] - Cd[ax];
                    } else {
                        m2[ax] = -Sd[ax];
                        rhs[ax] = X[ax] - Cd[ax];
                    }
                }
                if (!ora_solve3(Ud, Vd, m2, rhs, sol) || (c->beam == 1 && !(sol[2] > 0.0))) {
                    full = 1;
                    break;
                }
                double iu = sol[0] / c->pitch_u + 0.5 * (c->n_u - 1) - c->offset_u;
                double iv = sol[1] / c->pitch_v + 0.5 * (c->n_v - 1) - c->offset_v;
                umin = fmin(umin, iu);
                umax = fmax(umax, iu);
                vmin = fmin(vmin, iv);
                vmax = fmax(vmax, iv);
            }
            long u0 = 0, u1 = c->n_u - 1, v0 = 0, v1 = c->n_v - 1;
            if (!full) {
                u0 = (long)floor(umin) - 1;
                u1 = (long)ceil(umax) + 1;
                v0 = (long)floor(vmin) - 1;
                v1 = (long)ceil(vmax) + 1;
                if (u0 < 0) u0 = 0;
                if (v0 < 0) v0 = 0;
                if (u1 > c->n_u - 1) u1 = c->n_u - 1;
                if (v1 > c->n_v - 1) v1 = c->n_v - 1;
            }
            for (long iv = v0; iv <= v1; ++iv)
                for (long iu = u0; iu <= u1; ++iu) {
                    long ray = (view * c->n_v + iv) * c->n_u + iu;
                    double X0[3], r[3], tlo, thi;
                    ora_ray(c, ray, X0, r, &tlo, &thi);
                    double L = ora_clip_box(X0, r, tlo, thi, blo, bhi);
                    if (L > 0.0) acc += L * (double)sino[ray];
                }
        }
        out[q] = acc;
    }
    return 0;
}

/*
 * Face-plane ambiguity flag per ray: 1 when, over its chord through the closed
 * volume box, the ray stays within tol * d of one cell-face plane of some axis
 * (it lies in, or numerically on, a face, where the two neighbouring cells
 * both contain it).  Such rays are assigned by the + side rule above, which any
 * other finite-precision traversal can only reproduce up to rounding.
 */
int ora_ambiguous(const ora_ctx *c, double tol, unsigned char *flags, int nthreads)
{
    int T = ora_threads(nthreads);
    long nr = ora_n_rays(c);
#pragma omp parallel for num_threads(T) schedule(dynamic, 256)
    for (long ray = 0; ray < nr; ++ray) {
        double X0[3], r[3], tlo, thi;
        ora_ray(c, ray, X0, r, &tlo, &thi);
        double a0 = tlo, a1 = thi;
        int miss = 0;
        for (int ax = 0; ax < 3; ++ax) {
            double p0 = c->o[ax], p1 = c->o[ax] + (double)c->n[ax] * c->d[ax];
            double slack = tol * c->d[ax];
            if (r[ax] == 0.0) {
                if (X0[ax] < p0 - slack || X0[ax] > p1 + slack) miss = 1;
            } else {
                double t0 = (p0 - slack - X0[ax]) / r[ax], t1 = (p1 + slack - X0[ax]) / r[ax];
                a0 = fmax(a0, fmin(t0, t1));
                a1 = fmin(a1, fmax(t0, t1));
            }
        }
        unsigned char flag = 0;
        if (!miss && a0 <= a1) {
            for (int ax = 0; ax < 3 && !flag; ++ax) {
                double e0 = X0[ax] + (r[ax] == 0.0 ? 0.0 : a0 * r[ax]);
                double e1 = X0[ax] + (r[ax] == 0.0 ? 0.0 : a1 * r[ax]);
                double slack = tol * c->d[ax];
                if (fabs(e1 - e0) > slack) continue;
                double q = (0.5 * (e0 + e1) - c->o[ax]) / c->d[ax];
                double nearest = floor(q + 0.5);
                if (nearest >= 0.0 && nearest <= (double)c->n[ax] &&
                    fabs(q - nearest) * c->d[ax] <= slack)
                    flag = 1;
            }
        }
        flags[ray] = flag;
    }
    return 0;
}

/* Midpoint-rule line integral with M samples along the chord through the
 * volume (nearest-cell lookup), for convergence checks of ora_forward. */
int ora_supersampled(const ora_ctx *c, const float *vol, const long *rays, long count,
                     long M, double *out, int nthreads)
{
    int T = ora_threads(nthreads);
#pragma omp parallel for num_threads(T) schedule(dynamic, 1)
    for (long q = 0; q < count; ++q) {
        double X0[3], r[3], tlo, thi, amin, amax;
        int lo[3] = {0, 0, 0};
        ora_ray(c, rays[q], X0, r, &tlo, &thi);
        double acc = 0.0;
        if (ora_clip_cells(c, X0, r, tlo, thi, lo, c->n, &amin, &amax)) {
            double h = (amax - amin) / (double)M;
            for (long m = 0; m < M; ++m) {
                double t = amin + ((double)m + 0.5) * h;
                long idx[3];
                int inside = 1;
                for (int ax = 0; ax < 3; ++ax) {
                    idx[ax] = (long)floor((X0[ax] + t * r[ax] - c->o[ax]) / c->d[ax]);
                    if (idx[ax] < 0 || idx[ax] >= c->n[ax]) inside = 0;
                }
                if (inside) acc += (double)vol[(idx[2] * c->n[1] + idx[1]) * c->n[0] + idx[0]];
            }
            acc *= h * ora_norm(r);
        }
        out[q] = acc;
    }
    return 0;
}

/* The pieces of one ray: linear cell index and physical length of every
 * positive-length piece, in traversal order.  cells / lens must hold
 * nx + ny + nz + 8 entries.  Returns the number of pieces. */
int ora_trace_ray(const ora_ctx *c, long ray, long *cells, double *lens)
{
    int B = ora_buf_len(c);
    double *buf = (double *)malloc(sizeof(double) * B);
    if (!buf) return -1;
    double X0[3], r[3], tlo, thi;
    int lo[3] = {0, 0, 0};
    ora_ray(c, ray, X0, r, &tlo, &thi);
    int n = ora_trace(c, X0, r, tlo, thi, lo, c->n, buf, cells, lens);
    free(buf);
    return n;
}

/*
 * Geometry vector-Jacobian product: first-order gradients of the path sums
 * with respect to each view's frame ("first-order source / centre / axis
 * gradients", diffct 2.4.1 -> 2.4.2, docs/video/README.md, shot "Geometry";
 * trajectory tensors that require gradients receive geometry gradients,
 * diffct 2.1.0 -> 2.2.1, README "Arbitrary trajectories").
 *
 *     out[view * 12 + m] = sum over rays R of the view of w[R] * d p(R) / d theta_m,
 *     theta = (src[3], det_centre[3], det_u[3], det_v[3]).
 *
 * For the line X0 + t r, t in [tlo, thi] (divergent: X0 = source, r = pixel -
 * source, t in [0, 1]; parallel: X0 = pixel, r = src, t free), the path sum of
 * the cell-constant image is p = |r| sum_j (t_{j+1} - t_j) f_j.  Its pieces end
 * where the line crosses a plane x_a = const of the grid (or the ray's own end
 * point, which does not move with the planes).  A crossing at t_k moves by
 * dt_k = -(dX0_a + t_k dr_a) / r_a, so
 *     dp/dX0_a = -|r| sum_{k on axis a} (f_before - f_after)_k / r_a,
 *     dp/dr_a  = -|r| sum_{k on axis a} (f_before - f_after)_k t_k / r_a + p r_a / |r|^2,
 * with the value outside the volume 0 at the box faces.
 */
/* Gradient of one ray's path sum with respect to the ray's start X0 and its
 * direction r (the crossing sums above, written out for ray `ray`): dsrc and
 * dpix are dp/d source and dp/d pixel (divergent: X0 = source, r = pixel -
 * source; parallel: X0 = pixel, r = src, so dsrc is dp/d src).  Returns 0 when
 * the ray misses the grid (both zero).  buf: ora_buf_len(c) doubles. */
static int ora_ray_gradient(const ora_ctx *c, const float *vol, long ray, double *buf,
                            double dsrc[3], double dpix[3])
{
    for (int ax = 0; ax < 3; ++ax) dsrc[ax] = dpix[ax] = 0.0;
    double X0[3], r[3], tlo, thi;
    ora_ray(c, ray, X0, r, &tlo, &thi);
    /* clip to the grid, remembering which face plane bounds it */
    double amin = tlo, amax = thi;
    int ain = -1, aout = -1, empty = 0;
    for (int ax = 0; ax < 3; ++ax) {
        double p0 = c->o[ax], p1 = c->o[ax] + (double)c->n[ax] * c->d[ax];
        if (r[ax] == 0.0) {
            if (!(X0[ax] >= p0 && X0[ax] < p1)) empty = 1;
            continue;
        }
        double t0 = (p0 - X0[ax]) / r[ax], t1 = (p1 - X0[ax]) / r[ax];
        double e0 = fmin(t0, t1), e1 = fmax(t0, t1);
        if (e0 > amin) { amin = e0; ain = ax; }
        if (e1 < amax) { amax = e1; aout = ax; }
    }
    if (empty || !(amin < amax)) return 0;
    /* interior crossings per axis, merged in increasing t */
    double *seq[3];
    int len[3], pos[3];
    double *next = buf;
    for (int ax = 0; ax < 3; ++ax) {
        seq[ax] = next;
        len[ax] = 0;
        pos[ax] = 0;
        if (r[ax] == 0.0) continue;
        for (int m = 0; m <= c->n[ax]; ++m) {
            int k = r[ax] > 0.0 ? m : c->n[ax] - m;
            double t = (c->o[ax] + (double)k * c->d[ax] - X0[ax]) / r[ax];
            if (t > amin && t < amax) seq[ax][len[ax]++] = t;
        }
        next += len[ax];
    }
    double norm = ora_norm(r);
    double sum_df[3] = {0, 0, 0}, sum_dft[3] = {0, 0, 0};
    double p = 0.0, prev = amin, f_prev = 0.0;
    int first = 1;
    for (;;) {
        double t = amax;
        int which = -1;
        for (int ax = 0; ax < 3; ++ax)
            if (pos[ax] < len[ax] && seq[ax][pos[ax]] < t) {
                t = seq[ax][pos[ax]];
                which = ax;
            }
        /* the piece [prev, t) and its value (midpoint cell) */
        double mid = 0.5 * (prev + t), f = 0.0;
        if (t > prev) {
            long idx[3];
            for (int ax = 0; ax < 3; ++ax) {
                long q = (long)floor((X0[ax] + mid * r[ax] - c->o[ax]) / c->d[ax]);
                if (q < 0) q = 0;
                if (q > c->n[ax] - 1) q = c->n[ax] - 1;
                idx[ax] = q;
            }
            f = (double)vol[(idx[2] * c->n[1] + idx[1]) * c->n[0] + idx[0]];
            p += (t - prev) * f;
        } else {
            f = f_prev;  /* zero-length piece: no value change */
        }
        if (first) {
            /* entry through a face plane: outside value 0 */
            if (ain >= 0) {
                sum_df[ain] += 0.0 - f;
                sum_dft[ain] += (0.0 - f) * amin;
            }
            first = 0;
        }
        f_prev = f;
        if (which < 0) break;
        /* crossing of axis `which` at t: value before f, after = next piece */
        double t_next = amax;
        for (int ax = 0; ax < 3; ++ax) {
            int pp = pos[ax] + (ax == which ? 1 : 0);
            if (pp < len[ax] && seq[ax][pp] < t_next) t_next = seq[ax][pp];
        }
        double f_after = f;
        if (t_next > t) {
            double m2 = 0.5 * (t + t_next);
            long idx[3];
            for (int ax = 0; ax < 3; ++ax) {
                long q = (long)floor((X0[ax] + m2 * r[ax] - c->o[ax]) / c->d[ax]);
                if (q < 0) q = 0;
                if (q > c->n[ax] - 1) q = c->n[ax] - 1;
                idx[ax] = q;
            }
            f_after = (double)vol[(idx[2] * c->n[1] + idx[1]) * c->n[0] + idx[0]];
        }
        sum_df[which] += f - f_after;
        sum_dft[which] += (f - f_after) * t;
        pos[which]++;
        prev = t;
    }
    /* exit through a face plane: outside value 0 */
    if (aout >= 0) {
        sum_df[aout] += f_prev - 0.0;
        sum_dft[aout] += (f_prev - 0.0) * amax;
    }
    p *= norm;
    for (int ax = 0; ax < 3; ++ax) {
        double gx = r[ax] != 0.0 ? -norm * sum_df[ax] / r[ax] : 0.0;
        double gr = (r[ax] != 0.0 ? -norm * sum_dft[ax] / r[ax] : 0.0) +
                    p * r[ax] / (norm * norm);
        if (c->beam == 1) {
            dsrc[ax] = gx - gr;
            dpix[ax] = gr;
        } else {
            dsrc[ax] = gr;
            dpix[ax] = gx;
        }
    }
    return 1;
}

static void ora_cross(const double a[3], const double b[3], double out[3])
{
    out[0] = a[1] * b[2] - a[2] * b[1];
    out[1] = a[2] * b[0] - a[0] * b[2];
    out[2] = a[0] * b[1] - a[1] * b[0];
}

/* The detector frame of view `view` in float64: u, v, the unit normal
 * n = (u x v) / |u x v| and |u x v|. */
static void ora_frame_axes(const ora_ctx *c, long view, double u[3], double v[3], double n[3],
                           double *cn)
{
    const float *U = c->det_u + 3 * view, *V = c->det_v + 3 * view;
    for (int ax = 0; ax < 3; ++ax) {
        u[ax] = (double)U[ax];
        v[ax] = (double)V[ax];
    }
    ora_cross(u, v, n);
    *cn = ora_norm(n);
    for (int ax = 0; ax < 3; ++ax) n[ax] /= *cn;
}

/* Offsets (t, s, e) along u, v and n of the pixel of detector sample `ray`: a
 * curved detector's own table (shared, or the ray's view's), or the pitch grid
 * of a flat one (e = 0). */
static void ora_pixel_offsets(const ora_ctx *c, long ray, double q[3])
{
    long pix = ray % ((long)c->n_u * c->n_v);
    if (c->offsets) {
        long at = c->offsets_per_view ? ray : pix;
        for (int m = 0; m < 3; ++m) q[m] = (double)c->offsets[3 * at + m];
    } else {
        long iv = pix / c->n_u, iu = pix % c->n_u;
        q[0] = ((double)iu - 0.5 * (double)(c->n_u - 1) + c->offset_u) * c->pitch_u;
        q[1] = ((double)iv - 0.5 * (double)(c->n_v - 1) + c->offset_v) * c->pitch_v;
        q[2] = 0.0;
    }
}

/*
 * The chain rule to the frame: pixel = centre + t u + s v + e n, n = (u x v) /
 * |u x v| ((t, s, e) the pitch grid with e = 0 for flat detectors, a curved
 * detector's per-pixel offsets otherwise); divergent: source = X0, pixel = X0 +
 * r; parallel: pixel = X0, src = r.  With g = dp/d pixel, the normal's
 * derivative gives d(e n)/du^T g = e v x h and d(e n)/dv^T g = -e u x h, h =
 * (g - (n.g) n) / |u x v| (dn = (I - n n^T) d(u x v) / |u x v|).
 * Configurations where two crossings coincide (a ray through a cell edge or
 * corner) are kinks of p and have no gradient; whatever the merge order gives
 * there is accepted.  Views run in parallel (each view's sums are owned by one
 * thread).
 */
int ora_geometry_vjp(const ora_ctx *c, const float *vol, const float *w, double *out,
                     int nthreads)
{
    int T = ora_threads(nthreads);
    int B = ora_buf_len(c);
    long per_view = (long)c->n_u * c->n_v;
    int err = 0;
#pragma omp parallel num_threads(T)
    {
        double *buf = (double *)malloc(sizeof(double) * B);
        if (!buf) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int view = 0; view < c->n_views; ++view) {
                double g[12] = {0};
                double u[3], v[3], n[3], cn;
                ora_frame_axes(c, view, u, v, n, &cn);
                for (long pix = 0; pix < per_view; ++pix) {
                    long ray = view * per_view + pix;
                    double wr = (double)w[ray];
                    if (wr == 0.0) continue;
                    double dsrc[3], dpix[3], q[3];
                    if (!ora_ray_gradient(c, vol, ray, buf, dsrc, dpix)) continue;
                    ora_pixel_offsets(c, ray, q);
                    double h[3], vh[3], uh[3];
                    double ng = n[0] * dpix[0] + n[1] * dpix[1] + n[2] * dpix[2];
                    for (int ax = 0; ax < 3; ++ax) h[ax] = (dpix[ax] - ng * n[ax]) / cn;
                    ora_cross(v, h, vh);
                    ora_cross(u, h, uh);
                    for (int ax = 0; ax < 3; ++ax) {
                        g[ax] += wr * dsrc[ax];
                        g[3 + ax] += wr * dpix[ax];
                        g[6 + ax] += wr * (q[0] * dpix[ax] + q[2] * vh[ax]);
                        g[9 + ax] += wr * (q[1] * dpix[ax] - q[2] * uh[ax]);
                    }
                }
                for (int m = 0; m < 12; ++m) out[12 * view + m] = g[m];
            }
        }
        free(buf);
    }
    return err;
}

/*
 * Surface-offset vector-Jacobian product: first-order gradients of the path
 * sums with respect to every pixel's offsets (t, s, e) along the detector axes
 * u, v and the unit normal n, shared by all views (the pages' curved detectors:
 * "Projection and matched backprojection support first-order surface
 * gradients", diffct 2.1.0 -> 2.2.1, README "Curved detectors"; the point
 * centre + t u + s v + e n, diffct 2.4.1 -> 2.4.2, kernels/surface_geometry.py
 * `compose_surface`):
 *
 *     out[pix * 3 + m] = sum over views of w[ray] * (dp/d pixel) . (u, v, n)[m],
 *
 * flat detectors included (their offsets are the pitch grid); with one offset
 * table per view, every view's pixel has its own gradient (out[ray * 3 + m],
 * no sum over views).  Pixels run in parallel (each pixel's sums are owned by
 * one thread).
 */
int ora_surface_vjp(const ora_ctx *c, const float *vol, const float *w, double *out,
                    int nthreads)
{
    int T = ora_threads(nthreads);
    int B = ora_buf_len(c);
    long per_view = (long)c->n_u * c->n_v;
    int per = c->offsets && c->offsets_per_view;  /* one offset table per view */
    int err = 0;
#pragma omp parallel num_threads(T)
    {
        double *buf = (double *)malloc(sizeof(double) * B);
        if (!buf) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long pix = 0; pix < per_view; ++pix) {
                double g[3] = {0, 0, 0};
                for (long view = 0; view < c->n_views; ++view) {
                    long ray = view * per_view + pix;
                    double wr = (double)w[ray];
                    double dsrc[3], dpix[3], u[3], v[3], n[3], cn;
                    if (per) g[0] = g[1] = g[2] = 0.0;
                    if (wr != 0.0 && ora_ray_gradient(c, vol, ray, buf, dsrc, dpix)) {
                        ora_frame_axes(c, view, u, v, n, &cn);
                        g[0] += wr * (dpix[0] * u[0] + dpix[1] * u[1] + dpix[2] * u[2]);
                        g[1] += wr * (dpix[0] * v[0] + dpix[1] * v[1] + dpix[2] * v[2]);
                        g[2] += wr * (dpix[0] * n[0] + dpix[1] * n[1] + dpix[2] * n[2]);
                    }
                    if (per)
                        for (int m = 0; m < 3; ++m) out[3 * ray + m] = g[m];
                }
                if (!per)
                    for (int m = 0; m < 3; ++m) out[3 * pix + m] = g[m];
            }
        }
        free(buf);
    }
    return err;
}

/*
 * Kink flags: rays on which two plane crossings of different axes coincide
 * within `tol` cells (the ray passes through a cell edge or corner, or enters /
 * leaves the grid there), or whose own end point inside the grid lies within
 * `tol` cells of a plane.  The path sum is not differentiable in the geometry
 * there: each side's derivative gives the jump to a different axis, and any
 * finite-precision traversal may pick either.  Used to exclude such rays from
 * gradient comparisons.
 */
int ora_kinks(const ora_ctx *c, double tol, unsigned char *flags, int nthreads)
{
    int T = ora_threads(nthreads);
    int B = c->n[0] + c->n[1] + c->n[2] + 8;
    long nr = ora_n_rays(c);
    double dmin = fmin(c->d[0], fmin(c->d[1], c->d[2]));
    int err = 0;
#pragma omp parallel num_threads(T)
    {
        double *ts = (double *)malloc(sizeof(double) * B);
        int *axs = (int *)malloc(sizeof(int) * B);
        if (!ts || !axs) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (long ray = 0; ray < nr; ++ray) {
                double X0[3], r[3], tlo, thi;
                ora_ray(c, ray, X0, r, &tlo, &thi);
                flags[ray] = 0;
                double amin = tlo, amax = thi;
                int empty = 0;
                for (int ax = 0; ax < 3; ++ax) {
                    double p0 = c->o[ax], p1 = c->o[ax] + (double)c->n[ax] * c->d[ax];
                    if (r[ax] == 0.0) {
                        if (!(X0[ax] >= p0 && X0[ax] < p1)) empty = 1;
                        continue;
                    }
                    double t0 = (p0 - X0[ax]) / r[ax], t1 = (p1 - X0[ax]) / r[ax];
                    amin = fmax(amin, fmin(t0, t1));
                    amax = fmin(amax, fmax(t0, t1));
                }
                if (empty || !(amin < amax)) continue;
                /* every plane crossing within tol of [amin, amax], all axes, unsorted */
                double scale = ora_norm(r) / dmin, eps = tol / scale;
                int m = 0;
                for (int ax = 0; ax < 3; ++ax) {
                    if (r[ax] == 0.0) continue;
                    for (int k = 0; k <= c->n[ax]; ++k) {
                        double t = (c->o[ax] + (double)k * c->d[ax] - X0[ax]) / r[ax];
                        if (t >= amin - eps && t <= amax + eps) {
                            ts[m] = t;
                            axs[m] = ax;
                            ++m;
                        }
                    }
                }
                /* insertion sort by t (m is at most nx + ny + nz + 3) */
                for (int q = 1; q < m; ++q) {
                    double t = ts[q];
                    int a = axs[q], s = q - 1;
                    while (s >= 0 && ts[s] > t) {
                        ts[s + 1] = ts[s];
                        axs[s + 1] = axs[s];
                        --s;
                    }
                    ts[s + 1] = t;
                    axs[s + 1] = a;
                }
                for (int q = 1; q < m; ++q)
                    if (axs[q] != axs[q - 1] && (ts[q] - ts[q - 1]) * scale <= tol) {
                        flags[ray] = 1;
                        break;
                    }
                /* an end point of the ray inside the grid that lies on a plane */
                for (int q = 0; q < m; ++q)
                    if ((amin == tlo && fabs(ts[q] - amin) * scale <= tol) ||
                        (amax == thi && fabs(amax - ts[q]) * scale <= tol)) {
                        flags[ray] = 1;
                        break;
                    }
            }
        }
        free(ts);
        free(axs);
    }
    return err;
}
