// Ray path: one thread per detector ray, slab DDA with exact fixed-point
// transverse positions.
//
// Parametrisation.  In cell coordinates (X - o) / d the ray is X0 + t w.  Its
// dominant axis p (largest |w_a|) is the slab axis; the two other axes b, c are
// transverse.  Every axis whose w is negative is mirrored (x -> n - x) so all
// coordinates grow along the ray.  With xi the (mirrored) p coordinate, the
// transverse coordinates are alpha_q + beta_q * xi with 0 <= beta_q <= 1, so a
// unit slab [k, k+1) of p holds at most one crossing of each transverse axis and
// the ray's pieces in it are:
//     [lo, t1) in cell (k, jb, jc), [t1, t2) after the first crossing,
//     [t2, hi) after both,   t_q = (1 - frac_q) / beta_q  if a crossing occurs.
// This is the same set of cells and lengths as the parametric Siddon traversal
// (exact path sum of the cell-constant model), reached slab by slab.
//
// Precision.  The ray set-up is float64 (the pages' portable path likewise clips
// rays and locates tile entries in FP64, diffct CHANGELOG 2.3.0 "Added").  The
// per-slab state is the transverse fraction in 32-bit fixed point (2^-32 of a
// cell) advanced by an integer add whose carry IS the plane crossing: no
// rounding drift however long the ray, so crossing positions stay within
// ~1e-7 cell of the float64 line ("distant endpoints keep voxel widths",
// same changelog entry).  Forward, backward and the segment counter call the
// same set-up and walk, so they visit bit-identical (cell, length) pieces and
// form a matched pair by construction.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ctp_internal.h"

namespace ctp {

struct SlabRay {
    int k0, k1;        // inclusive slab range along p (mirrored index)
    float tlo, thi;    // start fraction in slab k0, end fraction in slab k1
    uint32_t fb, fc;   // transverse fractions at slab k0 (units of 2^-32 cell)
    uint32_t bb, bc;   // transverse slopes per slab (units of 2^-32 cell)
    float ib, ic;      // 1 / bb, 1 / bc (0 when the slope is 0)
    int jb, jc;        // transverse (mirrored) cell indices at slab k0
    int nb, nc;        // transverse extents
    int addr;          // element offset of cell (k0, jb, jc)
    int sp, sb, sc;    // signed element strides along p, b, c
    float ell;         // physical length of the ray per unit slab
};

__device__ __forceinline__ uint32_t to_fixed_slope(double beta)
{
    double s = rint(beta * 4294967296.0);
    return s >= 4294967295.0 ? 0xffffffffu : (uint32_t)s;
}

// Float64 set-up of the ray through pixel (iu, iv) of view `view`.  Returns
// false when the ray misses the volume.
__device__ __forceinline__ bool slab_setup(const RayParams &P, int view, int iu, int iv,
                                           SlabRay &R)
{
    const ViewFrame &V = P.views[view];
    double X0[3], w[3];
    double fu = (double)iu, fv = (double)iv, fe = 0.0;
    if (P.offsets) {
        // curved detector: the pixel's (t, s, e) offsets along du, dv, dn
        const float *q = pixel_offsets_of(P, view, iu, iv);
        fu = (double)q[0];
        fv = (double)q[1];
        fe = (double)q[2];
    }
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        double pix = __fma_rn(fv, V.dv[a], __fma_rn(fu, V.du[a], V.p00[a]));
        if (P.offsets) pix = __fma_rn(fe, V.dn[a], pix);
        if (P.beam == 1) {
            X0[a] = V.a[a];
            w[a] = __dsub_rn(pix, V.a[a]);
        } else {
            X0[a] = pix;
            w[a] = V.a[a];
        }
    }
    const double aw0 = fabs(w[0]), aw1 = fabs(w[1]), aw2 = fabs(w[2]);
    const int p = (aw0 >= aw1 && aw0 >= aw2) ? 0 : (aw1 >= aw2 ? 1 : 2);
    const int b = p == 0 ? 1 : 0;
    const int c = p == 2 ? 1 : 2;
    const double awp = p == 0 ? aw0 : (p == 1 ? aw1 : aw2);
    if (!(awp > 0.0)) return false;

    double A[3], aw[3] = {aw0, aw1, aw2};
#pragma unroll
    for (int a = 0; a < 3; ++a) A[a] = w[a] < 0.0 ? __dsub_rn((double)P.n[a], X0[a]) : X0[a];

    const double inv = __ddiv_rn(1.0, awp);
    const double beta_b = __dmul_rn(aw[b], inv), beta_c = __dmul_rn(aw[c], inv);
    const double alpha_b = __fma_rn(-A[p], beta_b, A[b]);
    const double alpha_c = __fma_rn(-A[p], beta_c, A[c]);

    // Clip xi to the volume, to the ray's own extent and to the transverse range.
    double lo = 0.0, hi = (double)P.n[p];
    double lo_t = -1.0e300, hi_t = 1.0e300;
    if (P.beam == 1) {
        lo_t = A[p];
        hi_t = __dadd_rn(A[p], awp);
        lo = fmax(lo, lo_t);
        hi = fmin(hi, hi_t);
    }
    const double nb = (double)P.n[b], nc = (double)P.n[c];
    if (beta_b > 0.0) {
        const double r = __ddiv_rn(awp, aw[b]);
        lo = fmax(lo, __dmul_rn(-alpha_b, r));
        hi = fmin(hi, __dmul_rn(__dsub_rn(nb, alpha_b), r));
    } else if (!(alpha_b >= 0.0 && alpha_b < nb)) {
        return false;
    }
    if (beta_c > 0.0) {
        const double r = __ddiv_rn(awp, aw[c]);
        lo = fmax(lo, __dmul_rn(-alpha_c, r));
        hi = fmin(hi, __dmul_rn(__dsub_rn(nc, alpha_c), r));
    } else if (!(alpha_c >= 0.0 && alpha_c < nc)) {
        return false;
    }
    if (!(lo < hi)) return false;

    // Slabs that hold part of [lo, hi).  Where the fixed-point walk and this
    // float64 clip disagree by rounding (~1e-9 slab), the walk's bounds test
    // drops the sliver outside the grid.
    double k0 = fmax(floor(lo), 0.0);
    double k1 = fmin(ceil(hi) - 1.0, (double)(P.n[p] - 1));
    if (k0 > k1) return false;
    R.k0 = (int)k0;
    R.k1 = (int)k1;
    R.tlo = (float)fmin(fmax(__dsub_rn(lo_t, k0), 0.0), 1.0);
    R.thi = (float)fmin(fmax(__dsub_rn(hi_t, k1), 0.0), 1.0);

    const double xb = __fma_rn(k0, beta_b, alpha_b), xc = __fma_rn(k0, beta_c, alpha_c);
    const double fjb = floor(xb), fjc = floor(xc);
    R.jb = (int)fjb;
    R.jc = (int)fjc;
    R.fb = (uint32_t)__dmul_rn(__dsub_rn(xb, fjb), 4294967296.0);
    R.fc = (uint32_t)__dmul_rn(__dsub_rn(xc, fjc), 4294967296.0);
    R.bb = to_fixed_slope(beta_b);
    R.bc = to_fixed_slope(beta_c);
    R.ib = R.bb ? __frcp_rn((float)R.bb) : 0.0f;
    R.ic = R.bc ? __frcp_rn((float)R.bc) : 0.0f;
    R.nb = P.n[b];
    R.nc = P.n[c];

    // Length per slab: |(w_a d_a)| / |w_p| = sqrt(sum over axes of (beta_a d_a)^2),
    // beta_p = 1; float32 is ample for this per-ray scale factor.
    const float sp = (float)P.spacing[p];
    const float db = (float)(P.spacing[b] * beta_b), dc = (float)(P.spacing[c] * beta_c);
    R.ell = __fsqrt_rn(__fadd_rn(__fadd_rn(__fmul_rn(sp, sp), __fmul_rn(db, db)),
                                 __fmul_rn(dc, dc)));

    int sgn[3], base = 0;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        const bool m = w[a] < 0.0;
        sgn[a] = m ? -P.stride[a] : P.stride[a];
        if (m) base += P.stride[a] * (P.n[a] - 1);
    }
    R.sp = sgn[p];
    R.sb = sgn[b];
    R.sc = sgn[c];
    R.addr = base + sgn[p] * R.k0 + sgn[b] * R.jb + sgn[c] * R.jc;
    return true;
}

// Walk the slabs of a set-up ray; op(addr, length_in_slab_units, active) is
// called three times per slab.  All lengths are exact float differences of
// fractions in [0, 1]; the physical length is length * R.ell.
template <class Op>
__device__ __forceinline__ void slab_walk(const SlabRay &R, Op &op)
{
    uint32_t fb = R.fb, fc = R.fc;
    int jb = R.jb, jc = R.jc, addr = R.addr;
    const unsigned nb = (unsigned)R.nb, nc = (unsigned)R.nc;
    for (int k = R.k0; k <= R.k1; ++k) {
        const uint32_t gb = fb + R.bb, gc = fc + R.bc;
        const bool cb = gb < fb, cc = gc < fc;
        const float tb = cb ? fminf(__fmul_rn(__uint2float_rn(0u - fb), R.ib), 1.0f) : 1.0f;
        const float tc = cc ? fminf(__fmul_rn(__uint2float_rn(0u - fc), R.ic), 1.0f) : 1.0f;
        const float lo = k == R.k0 ? R.tlo : 0.0f;
        const float hi = k == R.k1 ? R.thi : 1.0f;
        const bool bfirst = tb < tc;
        const float e1 = fminf(fmaxf(fminf(tb, tc), lo), hi);
        const float e2 = fminf(fmaxf(fmaxf(tb, tc), lo), hi);
        const float d1 = __fsub_rn(e1, lo), d2 = __fsub_rn(e2, e1), d3 = __fsub_rn(hi, e2);
        const int jb2 = jb + (bfirst ? 1 : 0), jc2 = jc + (bfirst ? 0 : 1);
        const int jb3 = jb + (cb ? 1 : 0), jc3 = jc + (cc ? 1 : 0);
        const int a2 = addr + (bfirst ? R.sb : R.sc);
        const int a3 = addr + (cb ? R.sb : 0) + (cc ? R.sc : 0);
        op(addr, d1, d1 > 0.0f && (unsigned)jb < nb && (unsigned)jc < nc);
        op(a2, d2, d2 > 0.0f && (unsigned)jb2 < nb && (unsigned)jc2 < nc);
        op(a3, d3, d3 > 0.0f && (unsigned)jb3 < nb && (unsigned)jc3 < nc);
        fb = gb;
        fc = gc;
        jb = jb3;
        jc = jc3;
        addr = a3 + R.sp;
    }
}

struct GatherOp {
    const float *__restrict__ vol;
    float acc;
    long long lim;  // cells of vol (bounds-checked builds)
    __device__ __forceinline__ void operator()(int a, float d, bool on)
    {
        if (on && ctp_in(a, lim, kSiteRayGather)) acc = __fmaf_rn(d, __ldg(vol + a), acc);
    }
};

struct ScatterOp {
    float *__restrict__ vol;
    float w;  // ell * y
    long long lim;
    __device__ __forceinline__ void operator()(int a, float d, bool on)
    {
        if (on && ctp_in(a, lim, kSiteRayScatter)) atomicAdd(vol + a, __fmul_rn(d, w));
    }
};

// Cells of the (nz, ny, nx) volume the ray path addresses.
__host__ __device__ __forceinline__ long long volume_cells(const RayParams &P)
{
    return (long long)P.n[0] * P.n[1] * P.n[2];
}

// Counts the pieces longer than thr slab units (the counting threshold over
// the ray's length per slab).
struct CountOp {
    unsigned n;
    float thr;
    __device__ __forceinline__ void operator()(int, float d, bool on)
    {
        n += (on && d > thr) ? 1u : 0u;
    }
};

template <int TU, int TV>
__global__ void __launch_bounds__(TU *TV) ray_forward_kernel(RayParams P,
                                                             const float *__restrict__ vol,
                                                             float *__restrict__ sino)
{
    const int iu = blockIdx.x * TU + (int)(threadIdx.x % TU);
    const int iv = blockIdx.z * TV + (int)(threadIdx.x / TU);
    const int view = P.view0 + (int)blockIdx.y;
    if (iu >= P.n_u || iv >= P.n_v) return;
    float out = 0.0f;
    SlabRay R;
    if (slab_setup(P, view, iu, iv, R)) {
        GatherOp op{vol, 0.0f, volume_cells(P)};
        slab_walk(R, op);
        out = __fmul_rn(op.acc, R.ell);
    }
    const long long ray = ((long long)view * P.n_v + iv) * P.n_u + iu;
    if (ctp_in(ray, sino_cells(P), kSiteRaySinoStore)) sino[ray] = out;
}

template <int TU, int TV>
__global__ void __launch_bounds__(TU *TV) ray_backward_kernel(RayParams P,
                                                              const float *__restrict__ sino,
                                                              float *__restrict__ vol)
{
    const int iu = blockIdx.x * TU + (int)(threadIdx.x % TU);
    const int iv = blockIdx.z * TV + (int)(threadIdx.x / TU);
    const int view = P.view0 + (int)blockIdx.y;
    if (iu >= P.n_u || iv >= P.n_v) return;
    const long long ray = ((long long)view * P.n_v + iv) * P.n_u + iu;
    if (!ctp_in(ray, sino_cells(P), kSiteRaySinoLoad)) return;
    const float y = sino[ray];
    if (y == 0.0f) return;
    SlabRay R;
    if (slab_setup(P, view, iu, iv, R)) {
        ScatterOp op{vol, __fmul_rn(R.ell, y), volume_cells(P)};
        slab_walk(R, op);
    }
}

template <int TU, int TV>
__global__ void __launch_bounds__(TU *TV) ray_count_kernel(RayParams P,
                                                           unsigned long long *__restrict__ total)
{
    const int iu = blockIdx.x * TU + (int)(threadIdx.x % TU);
    const int iv = blockIdx.z * TV + (int)(threadIdx.x / TU);
    const int view = P.view0 + (int)blockIdx.y;
    unsigned n = 0;
    if (iu < P.n_u && iv < P.n_v) {
        SlabRay R;
        if (slab_setup(P, view, iu, iv, R)) {
            CountOp op{0u, __fdiv_rn(P.min_len, R.ell)};
            slab_walk(R, op);
            n = op.n;
        }
    }
    n = __reduce_add_sync(0xffffffffu, n);
    if ((threadIdx.x & 31) == 0 && n) atomicAdd(total, (unsigned long long)n);
}

}  // namespace ctp
