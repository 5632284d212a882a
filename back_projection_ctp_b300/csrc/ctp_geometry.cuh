// First-order geometry gradients of the path sums (vector-Jacobian product):
//
//     G[view][m] = sum over rays R of the view of w[R] * d p(R) / d theta_m,
//     theta = (src, det_centre, det_u, det_v) of that view (12 numbers),
//
// the calibration gradient of the pages ("first-order source / centre / axis
// gradients", diffct 2.4.1 -> 2.4.2, docs/video/README.md, shot "Geometry";
// trajectory tensors that require gradients receive geometry gradients, diffct
// 2.1.0 -> 2.2.1, README "Arbitrary trajectories").
//
// For the line X0 + t r (divergent: X0 = source, r = pixel - source, t in
// [0, 1]; parallel: X0 = pixel, r = src) the path sum of the cell-constant
// image is p = |r| sum_j (t_{j+1} - t_j) f_j.  A piece ends where the line
// crosses a grid plane x_a = const (value outside the grid: 0) or at the ray's
// own end point, which does not move with the planes.  A plane crossing at t_k
// moves by dt_k = -(dX0_a + t_k dr_a) / r_a, hence
//     dp/dX0_a = -|r| sum_{k on axis a} (f_before - f_after)_k / r_a
//     dp/dr_a  = -|r| sum_{k on axis a} (f_before - f_after)_k t_k / r_a + p r_a / |r|^2
// and pixel = centre + alpha u + beta v.  Configurations where two crossings
// coincide (a ray through a cell edge) are kinks of p; the walk attributes the
// jump to one of them.
//
// B300 design: the ray path's float64 set-up and exact fixed-point slab walk
// (the same pieces as the forward), one thread per ray, crossings taken from
// the walk's carries in order; the per-ray gradient is reduced over the block
// (all threads of a block belong to one view) and added to the view's twelve
// float64 sums with one atomic each.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ctp_check.h"
#include "ctp_column.cuh"
#include "ctp_internal.h"
#include "ctp_ray.cuh"

// Operand of the bounds-check hooks (dropped in normal builds): cells of the
// padded z-fastest working copy the column walk reads.
#define CTP_GEOM_CELLS ((long long)column_padded_cells(P))

namespace ctp {

struct GeomParams {
    float cu, cv;            // pixel index of the detector centre: (n - 1)/2 - offset
    float pitch_u, pitch_v;
    double pitch_ud, pitch_vd;  // the pitches in float64 (unit axes of a flat detector)
};

// Axes, mirrored start and world direction of the ray through pixel (iu, iv):
// the quantities slab_setup keeps implicit.
struct RayAxes {
    int ax[3];       // world axes of the slab walk's p, b, c (selected, not indexed)
    double Ap, awp;  // mirrored p coordinate of X0 and |w_p| (cell units)
    float r[3];      // world direction r (physical units)
    float rn;        // |r|
};

__device__ __forceinline__ void ray_axes(const RayParams &P, int view, int iu, int iv, RayAxes &A)
{
    const ViewFrame &V = P.views[view];
    double X0[3], w[3];
    double fu = (double)iu, fv = (double)iv, fe = 0.0;
    if (P.offsets) {
        // curved detector: the pixel's (t, s, e) offsets along du, dv, dn (as slab_setup)
        const float *q = pixel_offsets_of(P, view, iu, iv);
        fu = (double)q[0];
        fv = (double)q[1];
        fe = (double)q[2];
    }
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        double pix = __fma_rn(fv, V.dv[a], __fma_rn(fu, V.du[a], V.p00[a]));
        if (P.offsets) pix = __fma_rn(fe, V.dn[a], pix);
        X0[a] = P.beam == 1 ? V.a[a] : pix;
        w[a] = P.beam == 1 ? __dsub_rn(pix, V.a[a]) : V.a[a];
    }
    const double aw0 = fabs(w[0]), aw1 = fabs(w[1]), aw2 = fabs(w[2]);
    const int p = (aw0 >= aw1 && aw0 >= aw2) ? 0 : (aw1 >= aw2 ? 1 : 2);
    A.ax[0] = p;
    A.ax[1] = p == 0 ? 1 : 0;
    A.ax[2] = p == 2 ? 1 : 2;
    A.awp = p == 0 ? aw0 : (p == 1 ? aw1 : aw2);
    A.Ap = w[p] < 0.0 ? __dsub_rn((double)P.n[p], X0[p]) : X0[p];
    double n2 = 0.0;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        const double ra = __dmul_rn(w[a], P.spacing[a]);
        A.r[a] = (float)ra;
        n2 = __fma_rn(ra, ra, n2);
    }
    A.rn = (float)sqrt(n2);
}

// Walk of one ray collecting, per walk axis (0 = p, 1 = b, 2 = c), the sums of
// value jumps (before - after) and of jumps times t over the plane crossings,
// and the path sum.
struct GradSums {
    float df[3], dft[3];
    float path;   // sum of slab fraction * value (times ell: the path sum)
};

// Adds jump j at parameter t to walk axis b (on_b) or c.
__device__ __forceinline__ void grad_add_bc(GradSums &G, bool on_b, float j, float t)
{
    if (on_b) {
        G.df[1] += j;
        G.dft[1] = __fmaf_rn(j, t, G.dft[1]);
    } else {
        G.df[2] += j;
        G.dft[2] = __fmaf_rn(j, t, G.dft[2]);
    }
}

// nvol: cells of vol, read by the bounds-check hooks only.
__device__ __forceinline__ void grad_walk(const SlabRay &R, const RayAxes &A,
                                          const float *__restrict__ vol, long long nvol,
                                          GradSums &G)
{
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        G.df[a] = 0.0f;
        G.dft[a] = 0.0f;
    }
    G.path = 0.0f;
    // t of the mirrored p coordinate xi: t = (xi - Ap) / |w_p|
    const float t0 = (float)__ddiv_rn(__dsub_rn((double)R.k0, A.Ap), A.awp);
    const float tinv = (float)__ddiv_rn(1.0, A.awp);
    uint32_t fb = R.fb, fc = R.fc;
    int jb = R.jb, jc = R.jc, addr = R.addr;
    const unsigned nb = (unsigned)R.nb, nc = (unsigned)R.nc;
    float f_prev = 0.0f;
    for (int k = R.k0; k <= R.k1; ++k) {
        const uint32_t gb = fb + R.bb, gc = fc + R.bc;
        const bool cb = gb < fb, cc = gc < fc;
        const float tb = cb ? fminf(__fmul_rn(__uint2float_rn(0u - fb), R.ib), 1.0f) : 1.0f;
        const float tc = cc ? fminf(__fmul_rn(__uint2float_rn(0u - fc), R.ic), 1.0f) : 1.0f;
        const float lo = k == R.k0 ? R.tlo : 0.0f;
        const float hi = k == R.k1 ? R.thi : 1.0f;
        const bool bfirst = tb < tc;
        const float x1 = fminf(tb, tc), x2 = fmaxf(tb, tc);  // crossing fractions
        const bool c1 = bfirst ? cb : cc, c2 = bfirst ? cc : cb;
        const float e1 = fminf(fmaxf(x1, lo), hi);
        const float e2 = fminf(fmaxf(x2, lo), hi);
        const float d1 = __fsub_rn(e1, lo), d2 = __fsub_rn(e2, e1), d3 = __fsub_rn(hi, e2);
        const int jb2 = jb + (bfirst ? 1 : 0), jc2 = jc + (bfirst ? 0 : 1);
        const int jb3 = jb + (cb ? 1 : 0), jc3 = jc + (cc ? 1 : 0);
        const int a2 = addr + (bfirst ? R.sb : R.sc);
        const int a3 = addr + (cb ? R.sb : 0) + (cc ? R.sc : 0);
        const float v1 = ((unsigned)jb < nb && (unsigned)jc < nc
                              CTP_AND_IN(addr, nvol, kSiteGeomRayLoad)) ? __ldg(vol + addr) : 0.0f;
        const float v2 = ((unsigned)jb2 < nb && (unsigned)jc2 < nc
                              CTP_AND_IN(a2, nvol, kSiteGeomRayLoad)) ? __ldg(vol + a2) : 0.0f;
        const float v3 = ((unsigned)jb3 < nb && (unsigned)jc3 < nc
                              CTP_AND_IN(a3, nvol, kSiteGeomRayLoad)) ? __ldg(vol + a3) : 0.0f;
        G.path = __fmaf_rn(d1, v1, __fmaf_rn(d2, v2, __fmaf_rn(d3, v3, G.path)));
        const float tk = __fmaf_rn((float)(k - R.k0), tinv, t0);  // t at the slab start
        // the p plane at the slab start: crossed unless the ray begins in this slab
        if (k > R.k0 || R.tlo == 0.0f) {
            const float j = f_prev - v1;
            G.df[0] += j;
            G.dft[0] = __fmaf_rn(j, tk, G.dft[0]);
        }
        // transverse crossings strictly inside the ray's extent in this slab
        const bool r1 = c1 && x1 > lo && x1 < hi, r2 = c2 && x2 > lo && x2 < hi;
        if (r1) grad_add_bc(G, bfirst, v1 - v2, __fmaf_rn(x1, tinv, tk));
        if (r2) grad_add_bc(G, !bfirst, v2 - v3, __fmaf_rn(x2, tinv, tk));
        // the cell at the slab's end lies past every crossing before hi, also
        // those before the ray's own start
        const bool h1 = c1 && x1 < hi, h2 = c2 && x2 < hi;
        f_prev = h2 ? v3 : (h1 ? v2 : v1);
        fb = gb;
        fc = gc;
        jb = jb3;
        jc = jc3;
        addr = a3 + R.sp;
    }
    // the p plane at the end of the last slab, when the ray goes on past it
    if (R.thi == 1.0f) {
        const float tk = __fmaf_rn((float)(R.k1 + 1 - R.k0), tinv, t0);
        G.df[0] += f_prev;
        G.dft[0] = __fmaf_rn(f_prev, tk, G.dft[0]);
    }
}

// Gradient of one ray's path sum with respect to the ray's start and end:
// dsrc = dp/d source (parallel: dp/d src, the direction) and dpix = dp/d pixel,
// world axes, from the walk's crossing sums.  False when the ray misses.
__device__ __forceinline__ bool ray_gradient(const RayParams &P, int view, int iu, int iv,
                                             const float *__restrict__ vol, float dsrc[3],
                                             float dpix[3])
{
    SlabRay R;
    if (!slab_setup(P, view, iu, iv, R)) return false;
    RayAxes A;
    ray_axes(P, view, iu, iv, A);
    GradSums S;
    grad_walk(R, A, vol, volume_cells(P), S);
    const float p = __fmul_rn(S.path, R.ell);
    const float rn2 = __fmul_rn(A.rn, A.rn);
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        // the walk axis that is world axis a
        const int q = A.ax[0] == a ? 0 : (A.ax[1] == a ? 1 : 2);
        const float df = q == 0 ? S.df[0] : (q == 1 ? S.df[1] : S.df[2]);
        const float dft = q == 0 ? S.dft[0] : (q == 1 ? S.dft[1] : S.dft[2]);
        const float ra = A.r[a];
        const float gx = ra != 0.0f ? -A.rn * df / ra : 0.0f;
        const float gr = (ra != 0.0f ? -A.rn * dft / ra : 0.0f) + p * ra / rn2;
        dsrc[a] = P.beam == 1 ? gx - gr : gr;
        dpix[a] = P.beam == 1 ? gr : gx;
    }
    return true;
}

// Physical detector axes of a view (float64): u, v, the unit normal n = u x v /
// |u x v| and |u x v|.  Curved frames store the unit axes (and n) over the
// spacing; flat frames the pitch-scaled axes over the spacing.
__device__ __forceinline__ void detector_axes(const RayParams &P, const GeomParams &Q, int view,
                                              double u[3], double v[3], double n[3], double &cn)
{
    const ViewFrame &V = P.views[view];
    const double su = P.offsets ? 1.0 : Q.pitch_ud, sv = P.offsets ? 1.0 : Q.pitch_vd;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        u[a] = __ddiv_rn(__dmul_rn(V.du[a], P.spacing[a]), su);
        v[a] = __ddiv_rn(__dmul_rn(V.dv[a], P.spacing[a]), sv);
    }
    n[0] = __fma_rn(u[1], v[2], -__dmul_rn(u[2], v[1]));
    n[1] = __fma_rn(u[2], v[0], -__dmul_rn(u[0], v[2]));
    n[2] = __fma_rn(u[0], v[1], -__dmul_rn(u[1], v[0]));
    cn = sqrt(__fma_rn(n[0], n[0], __fma_rn(n[1], n[1], __dmul_rn(n[2], n[2]))));
#pragma unroll
    for (int a = 0; a < 3; ++a) n[a] = __ddiv_rn(n[a], cn);
}

// Chain rule of a curved detector's pixel = centre + t u + s v + e n to the
// axes: with g = dp / d pixel and h = (g - (n.g) n) / |u x v| (dn = (I - n n^T)
// d(u x v) / |u x v|), dp/du = t g + e v x h and dp/dv = s g - e u x h.
__device__ __forceinline__ void curved_axis_gradients(const RayParams &P, int view, int iu,
                                                      int iv, const float g[3], float gu[3],
                                                      float gv[3])
{
    const float *q = pixel_offsets_of(P, view, iu, iv);
    const GeomParams unused{};
    double u[3], v[3], n[3], cn;
    detector_axes(P, unused, view, u, v, n, cn);
    const double ng = n[0] * g[0] + n[1] * g[1] + n[2] * g[2];
    double h[3];
#pragma unroll
    for (int a = 0; a < 3; ++a) h[a] = ((double)g[a] - ng * n[a]) / cn;
    const double vh[3] = {v[1] * h[2] - v[2] * h[1], v[2] * h[0] - v[0] * h[2],
                          v[0] * h[1] - v[1] * h[0]};
    const double uh[3] = {u[1] * h[2] - u[2] * h[1], u[2] * h[0] - u[0] * h[2],
                          u[0] * h[1] - u[1] * h[0]};
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        gu[a] = (float)((double)q[0] * g[a] + (double)q[2] * vh[a]);
        gv[a] = (float)((double)q[1] * g[a] - (double)q[2] * uh[a]);
    }
}

template <int TU, int TV>
__global__ void __launch_bounds__(TU *TV) geometry_vjp_kernel(RayParams P, GeomParams Q,
                                                              const float *__restrict__ vol,
                                                              const float *__restrict__ w,
                                                              double *__restrict__ out)
{
    constexpr int kWarps = TU * TV / 32;
    __shared__ float part[kWarps][12];
    const int iu = blockIdx.x * TU + (int)(threadIdx.x % TU);
    const int iv = blockIdx.z * TV + (int)(threadIdx.x / TU);
    const int view = P.view0 + (int)blockIdx.y;
    float g[12];
#pragma unroll
    for (int m = 0; m < 12; ++m) g[m] = 0.0f;
    if (iu < P.n_u && iv < P.n_v) {
        const long long ray = ((long long)view * P.n_v + iv) * P.n_u + iu;
        const float wr = w[ray];
        float dsrc[3], dpix[3];
        if (wr != 0.0f && ray_gradient(P, view, iu, iv, vol, dsrc, dpix)) {
            float gu[3], gv[3];
            if (P.offsets) {
                curved_axis_gradients(P, view, iu, iv, dpix, gu, gv);
            } else {
                const float alpha = ((float)iu - Q.cu) * Q.pitch_u;
                const float beta = ((float)iv - Q.cv) * Q.pitch_v;
#pragma unroll
                for (int a = 0; a < 3; ++a) {
                    gu[a] = alpha * dpix[a];
                    gv[a] = beta * dpix[a];
                }
            }
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                g[a] = wr * dsrc[a];
                g[3 + a] = wr * dpix[a];
                g[6 + a] = wr * gu[a];
                g[9 + a] = wr * gv[a];
            }
        }
    }
    // block reduction (one view per block), then one float64 atomic per component
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 0; m < 12; ++m) {
        float v = g[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
        if (lane == 0) part[warp][m] = v;
    }
    __syncthreads();
    if (threadIdx.x < 12) {
        double s = 0.0;
#pragma unroll
        for (int q = 0; q < kWarps; ++q) s += (double)part[q][threadIdx.x];
        if (true CTP_AND_IN(12 * (long long)view + threadIdx.x, 12LL * P.n_views, kSiteGeomOut))
            atomicAdd(out + 12 * (long long)view + threadIdx.x, s);
    }
}

// Column path (3-D scans whose v axis is +-z): the same crossing sums for the R
// rows a thread owns, over the column's shared xy walk (the b crossing is
// uniform across the warp) and each row's own z crossings, on the padded
// z-fastest working copy of the volume (zero halo in x and y; z validity per
// access).  t of the p coordinate is shared by the column's rows.
template <int R, bool VF>
__global__ void __launch_bounds__(256, 4) column_gvjp_kernel(RayParams P, GeomParams Q,
                                                          const ColumnTrace *__restrict__ T,
                                                          const float *__restrict__ zvol,
                                                          const float *__restrict__ wsino,
                                                          double *__restrict__ out)
{
    __shared__ float part[kColumnsPerBlock][12];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // VF: grid (views, column groups, row bands), as the column forward's
    const int iu = (VF ? (int)blockIdx.y : (int)blockIdx.x) * kColumnsPerBlock + warp;
    const int view = P.view0 + (int)(VF ? blockIdx.x : blockIdx.y);
    float g[12];
#pragma unroll
    for (int m = 0; m < 12; ++m) g[m] = 0.0f;
    const ColumnTrace C = iu < P.n_u ? T[(long long)view * P.n_u + iu] : ColumnTrace{};
    if (iu < P.n_u && C.k0 <= C.k1) {
        // column constants in float64: axes, the t map of the p coordinate, r
        const ViewFrame &V = P.views[view];
        double P0[3];
#pragma unroll
        for (int a = 0; a < 3; ++a) P0[a] = __fma_rn((double)iu, V.du[a], V.p00[a]);
        double X0[2], w[2];
#pragma unroll
        for (int a = 0; a < 2; ++a) {
            X0[a] = P.beam == 1 ? V.a[a] : P0[a];
            w[a] = P.beam == 1 ? __dsub_rn(P0[a], V.a[a]) : V.a[a];
        }
        const int p = fabs(w[0]) >= fabs(w[1]) ? 0 : 1;
        const double awp = fabs(w[p]);
        const double Ap = w[p] < 0.0 ? __dsub_rn((double)P.n[p], X0[p]) : X0[p];
        const float tinv = (float)__ddiv_rn(1.0, awp);
        const float t0 = (float)__ddiv_rn(__dsub_rn((double)C.k0, Ap), awp);
        const float rx = (float)__dmul_rn(w[0], P.spacing[0]);
        const float ry = (float)__dmul_rn(w[1], P.spacing[1]);
        const double z0 = P.beam == 1 ? __dsub_rn(P0[2], V.a[2]) : V.a[2];
        const double zstep = P.beam == 1 ? V.dv[2] : 0.0;
        const float alpha = ((float)iu - Q.cu) * Q.pitch_u;

        const int row0 = blockIdx.z * 32 * R + lane;
        RowZ Z[R];
        float wr[R], acc[R], fprev[R], dfp[R], dfb[R], dfz[R], dtp[R], dtb[R], dtz[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int iv = row0 + 32 * r;
            wr[r] = iv < P.n_v CTP_AND_IN(((long long)view * P.n_v + iv) * P.n_u + iu, sino_cells(P),
                                          kSiteGeomSinoLoad)
                        ? wsino[((long long)view * P.n_v + iv) * P.n_u + iu] : 0.0f;
            Z[r] = wr[r] != 0.0f ? column_row_setup(P, C, iv) : column_row_idle();
            acc[r] = fprev[r] = dfp[r] = dfb[r] = dfz[r] = dtp[r] = dtb[r] = dtz[r] = 0.0f;
        }
        bool any = false;
#pragma unroll
        for (int r = 0; r < R; ++r) any |= wr[r] != 0.0f;
        any = __any_sync(0xffffffffu, any);  // the warp shares the column
        const unsigned nz = (unsigned)P.n[2];
        uint32_t fb = C.fb;
        int xy = C.addr_xy;
        for (int k = C.k0; any && k <= C.k1; ++k) {
            const uint32_t gb = fb + C.bb;
            const bool cb = gb < fb;
            const float tk = __fmaf_rn((float)(k - C.k0), tinv, t0);
            if (!cb && k != C.k0 && k != C.k1) {
                // interior slab without a b crossing (uniform across the warp):
                // the general body below with lo = 0, hi = 1 and tb = 2, where the
                // cells after the first and after both crossings coincide
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t gz = Z[r].fz + Z[r].bz;
                    const bool cz = gz < Z[r].fz;
                    const float tz = fmaxf(__fmaf_rn(-__uint2float_rn(gz), Z[r].ibz, 1.0f), 0.0f);
                    const int za = Z[r].zoff, z1 = za + Z[r].sz;
                    const float vA = (unsigned)za < nz CTP_AND_IN(xy + za, CTP_GEOM_CELLS,
                                                                  kSiteGeomColumnLoad)
                                         ? __ldg(zvol + xy + za) : 0.0f;
                    const float vB = cz ? ((unsigned)z1 < nz CTP_AND_IN(xy + z1, CTP_GEOM_CELLS,
                                                                        kSiteGeomColumnLoad)
                                               ? __ldg(zvol + xy + z1) : 0.0f)
                                        : vA;
                    const float e1 = cz ? tz : 1.0f;
                    acc[r] = __fmaf_rn(e1, vA, __fmaf_rn(__fsub_rn(1.0f, e1), vB, acc[r]));
                    const float j = fprev[r] - vA;
                    dfp[r] += j;
                    dtp[r] = __fmaf_rn(j, tk, dtp[r]);
                    if (cz && tz > 0.0f && tz < 1.0f) {
                        const float jz = vA - vB, t = __fmaf_rn(tz, tinv, tk);
                        dfz[r] += jz;
                        dtz[r] = __fmaf_rn(jz, t, dtz[r]);
                    }
                    fprev[r] = cz && tz < 1.0f ? vB : vA;
                    Z[r].fz = gz;
                    if (cz) Z[r].zoff = z1;
                }
                xy += C.sp;
                fb = gb;
                continue;
            }
            const float lo = k == C.k0 ? C.tlo : 0.0f;
            const float hi = k == C.k1 ? C.thi : 1.0f;
            const float tb = cb ? fmaxf(__fmaf_rn(-__uint2float_rn(gb), C.ib, 1.0f), 0.0f) : 2.0f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t gz = Z[r].fz + Z[r].bz;
                const bool cz = gz < Z[r].fz;
                const float tz =
                    cz ? fmaxf(__fmaf_rn(-__uint2float_rn(gz), Z[r].ibz, 1.0f), 0.0f) : 2.0f;
                const int za = Z[r].zoff, z1 = za + Z[r].sz;
                const bool bfirst = tb < tz;
                const float x1 = fminf(tb, tz), x2 = fmaxf(tb, tz);
                // cells: A before both crossings, B after the first, C after both
                const int zb = bfirst ? za : (cz ? z1 : za), xyb = bfirst ? xy + C.sb : xy;
                const int zc = cz ? z1 : za, xyc = cb ? xy + C.sb : xy;
                const float vA = (unsigned)za < nz CTP_AND_IN(xy + za, CTP_GEOM_CELLS,
                                                              kSiteGeomColumnLoad)
                                     ? __ldg(zvol + xy + za) : 0.0f;
                const float vB = (unsigned)zb < nz CTP_AND_IN(xyb + zb, CTP_GEOM_CELLS,
                                                              kSiteGeomColumnLoad)
                                     ? __ldg(zvol + xyb + zb) : 0.0f;
                const float vC = (unsigned)zc < nz CTP_AND_IN(xyc + zc, CTP_GEOM_CELLS,
                                                              kSiteGeomColumnLoad)
                                     ? __ldg(zvol + xyc + zc) : 0.0f;
                const float e1 = fminf(fmaxf(x1, lo), hi), e2 = fminf(fmaxf(x2, lo), hi);
                acc[r] = __fmaf_rn(__fsub_rn(e1, lo), vA,
                                   __fmaf_rn(__fsub_rn(e2, e1), vB,
                                             __fmaf_rn(__fsub_rn(hi, e2), vC, acc[r])));
                if (k > C.k0 || C.tlo == 0.0f) {
                    const float j = fprev[r] - vA;
                    dfp[r] += j;
                    dtp[r] = __fmaf_rn(j, tk, dtp[r]);
                }
                if (x1 > lo && x1 < hi) {
                    const float j = vA - vB, t = __fmaf_rn(x1, tinv, tk);
                    if (bfirst) {
                        dfb[r] += j;
                        dtb[r] = __fmaf_rn(j, t, dtb[r]);
                    } else {
                        dfz[r] += j;
                        dtz[r] = __fmaf_rn(j, t, dtz[r]);
                    }
                }
                if (x2 > lo && x2 < hi) {
                    const float j = vB - vC, t = __fmaf_rn(x2, tinv, tk);
                    if (bfirst) {
                        dfz[r] += j;
                        dtz[r] = __fmaf_rn(j, t, dtz[r]);
                    } else {
                        dfb[r] += j;
                        dtb[r] = __fmaf_rn(j, t, dtb[r]);
                    }
                }
                fprev[r] = x2 < hi ? vC : (x1 < hi ? vB : vA);
                Z[r].fz = gz;
                if (cz) Z[r].zoff = z1;
            }
            xy += cb ? C.sp + C.sb : C.sp;
            fb = gb;
        }
        const float tend = __fmaf_rn((float)(C.k1 + 1 - C.k0), tinv, t0);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (wr[r] == 0.0f) continue;
            if (C.thi == 1.0f) {
                dfp[r] += fprev[r];
                dtp[r] = __fmaf_rn(fprev[r], tend, dtp[r]);
            }
            const int iv = row0 + 32 * r;
            const float rz = (float)(__fma_rn((double)iv, zstep, z0) * P.spacing[2]);
            const float rv[3] = {rx, ry, rz};
            const float rn2 = rx * rx + ry * ry + rz * rz, rn = sqrtf(rn2);
            const float pval = acc[r] * column_row_ell(P, C, Z[r].bz);
            const float beta = ((float)iv - Q.cv) * Q.pitch_v;
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                const float df = a == 2 ? dfz[r] : (a == p ? dfp[r] : dfb[r]);
                const float dt = a == 2 ? dtz[r] : (a == p ? dtp[r] : dtb[r]);
                const float ra = rv[a];
                const float gx = ra != 0.0f ? -rn * df / ra : 0.0f;
                const float gr = (ra != 0.0f ? -rn * dt / ra : 0.0f) + pval * ra / rn2;
                const float dsrc = P.beam == 1 ? gx - gr : gr;
                const float dpix = P.beam == 1 ? gr : gx;
                g[a] += wr[r] * dsrc;
                g[3 + a] += wr[r] * dpix;
                g[6 + a] += wr[r] * alpha * dpix;
                g[9 + a] += wr[r] * beta * dpix;
            }
        }
    }
#pragma unroll
    for (int m = 0; m < 12; ++m) {
        float v = g[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
        if (lane == 0) part[warp][m] = v;
    }
    __syncthreads();
    if (threadIdx.x < 12) {
        double sum = 0.0;
#pragma unroll
        for (int q = 0; q < kColumnsPerBlock; ++q) sum += (double)part[q][threadIdx.x];
        if (true CTP_AND_IN(12 * (long long)view + threadIdx.x, 12LL * P.n_views, kSiteGeomOut))
            atomicAdd(out + 12 * (long long)view + threadIdx.x, sum);
    }
}

// views_first: the plan's forward block order (circular scans), whose resident
// blocks then read a thin shell of the volume that L2 holds.
inline int column_geometry_vjp(const RayParams &P, const GeomParams &Q, const ColumnTrace *T,
                               const float *zvol, const float *w, double *out, bool views_first,
                               cudaStream_t s)
{
    if (cudaMemsetAsync(out, 0, sizeof(double) * 12 * (size_t)(P.n_views > 0 ? P.n_views : 0), s) !=
        cudaSuccess)
        return 9;
    if (P.view_count <= 0) return 0;
    if (views_first)
        column_gvjp_kernel<2, true><<<column_grid_views_first(P, 2), 256, 0, s>>>(P, Q, T, zvol, w,
                                                                                 out);
    else
        column_gvjp_kernel<2, false><<<column_grid(P, 2), 256, 0, s>>>(P, Q, T, zvol, w, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

// Surface gradient: one thread per pixel walks that pixel's ray in every view
// and sums w * dp/d pixel projected on the view's u, v and unit normal (the
// gradients with respect to the pixel's offsets t, s, e); out (n_v, n_u, 3)
// float64 -- (n_views, n_v, n_u, 3) with one offset table per view --
// overwritten; each pixel's sums are its thread's, no atomics.
template <int TU, int TV>
__global__ void __launch_bounds__(TU *TV) surface_vjp_kernel(RayParams P, GeomParams Q,
                                                             const float *__restrict__ vol,
                                                             const float *__restrict__ w,
                                                             double *__restrict__ out)
{
    const int iu = blockIdx.x * TU + (int)(threadIdx.x % TU);
    const int iv = blockIdx.y * TV + (int)(threadIdx.x / TU);
    if (iu >= P.n_u || iv >= P.n_v) return;
    // one offset table per view: every view's pixel has its own sums (out is
    // (n_views, n_v, n_u, 3)); else the sums run over the views
    const bool per_view = P.offsets && P.offsets_per_view;
    [[maybe_unused]] const long long nout = 3LL * P.n_u * P.n_v * (per_view ? P.n_views : 1);
    double acc[3] = {0.0, 0.0, 0.0};
    for (int view = 0; view < P.n_views; ++view) {
        const long long ray = ((long long)view * P.n_v + iv) * P.n_u + iu;
        if (per_view) acc[0] = acc[1] = acc[2] = 0.0;
        const float wr = (true CTP_AND_IN(ray, sino_cells(P), kSiteGeomSinoLoad)) ? w[ray] : 0.0f;
        float dsrc[3], dpix[3];
        if (wr != 0.0f && ray_gradient(P, view, iu, iv, vol, dsrc, dpix)) {
            double u[3], v[3], n[3], cn;
            detector_axes(P, Q, view, u, v, n, cn);
            double gu = 0.0, gv = 0.0, gn = 0.0;
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                gu = __fma_rn((double)dpix[a], u[a], gu);
                gv = __fma_rn((double)dpix[a], v[a], gv);
                gn = __fma_rn((double)dpix[a], n[a], gn);
            }
            acc[0] = __fma_rn((double)wr, gu, acc[0]);
            acc[1] = __fma_rn((double)wr, gv, acc[1]);
            acc[2] = __fma_rn((double)wr, gn, acc[2]);
        }
        if (per_view) {
#pragma unroll
            for (int m = 0; m < 3; ++m)
                if (true CTP_AND_IN(3 * ray + m, nout, kSiteGeomOut)) out[3 * ray + m] = acc[m];
        }
    }
    if (per_view) return;
    const long long o = 3 * ((long long)iv * P.n_u + iu);
#pragma unroll
    for (int m = 0; m < 3; ++m)
        if (true CTP_AND_IN(o + m, nout, kSiteGeomOut)) out[o + m] = acc[m];
}

inline int surface_vjp(const RayParams &P, const GeomParams &Q, const float *vol, const float *w,
                       double *out, cudaStream_t s)
{
    dim3 grid((P.n_u + 31) / 32, (P.n_v + 3) / 4, 1);
    surface_vjp_kernel<32, 4><<<grid, 128, 0, s>>>(P, Q, vol, w, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int geometry_vjp(const RayParams &P, const GeomParams &Q, const float *vol, const float *w,
                        double *out, cudaStream_t s)
{
    if (cudaMemsetAsync(out, 0, sizeof(double) * 12 * (size_t)(P.n_views > 0 ? P.n_views : 0), s) !=
        cudaSuccess)
        return 9;
    if (P.view_count <= 0) return 0;
    if (P.n_v == 1) {
        dim3 grid((P.n_u + 127) / 128, P.view_count, 1);
        geometry_vjp_kernel<128, 1><<<grid, 128, 0, s>>>(P, Q, vol, w, out);
    } else {
        dim3 grid((P.n_u + 31) / 32, P.view_count, (P.n_v + 3) / 4);
        geometry_vjp_kernel<32, 4><<<grid, 128, 0, s>>>(P, Q, vol, w, out);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

}  // namespace ctp
