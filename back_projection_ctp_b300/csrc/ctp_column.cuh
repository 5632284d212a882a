// Column path: for scans whose detector v axis is exactly +-z in every view.
//
// Then every ray of one detector column (fixed view and iu) has the same xy
// trace: the column's rays differ only in z.  (The pages' cone backprojection
// exploits the same structure: it walks the z crossings of each xy cell and
// groups adjacent detector rows in a warp so that a warp's atomics hit
// neighbouring voxels of one column -- diffct CHANGELOG 2.4.0 "Changed".)
//
// Here one warp owns 32 adjacent rows of one column.  The xy part of the slab
// walk (dominant xy axis p, other xy axis b) is set up ONCE per column in
// float64 at plan time and is identical in every lane; each lane adds its own z
// line (z = zc + iv zd at the first slab, slope bc + iv bd per slab, both
// affine in the row index) as the walk's second transverse axis.  The volume is
// walked in a z-fastest working copy, so the 32 lanes of a warp touch ~20
// consecutive floats per step: one or two cache lines per load or atomic.
//
// The walk itself is the ray path's slab_walk (same exact fixed-point
// arithmetic), so forward, backward and the counter visit bit-identical pieces.
#pragma once

#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>

#include "ctp_internal.h"
#include "ctp_ray.cuh"

namespace ctp {

struct ColumnTrace {
    int k0, k1;          // slab range along p (mirrored); k1 < k0: the column misses
    float tlo, thi;      // partial first / last slab fractions (ray ends)
    uint32_t fb, bb;     // b fraction at slab k0 and slope (2^-32 cell units)
    float ib;            // 1 / bb
    int jb;              // mirrored b index at slab k0
    int sp, sb;          // signed strides along p and b in the padded z-fastest copy
    int addr_xy;         // padded offset of xy cell (k0, jb) with z = 0
    int nb;              // extent along b
    float lxy2;          // squared physical xy length per slab
    int pad_;
    // Row iv's z line in fixed point (2^-40 cell): z at slab k0 = Z0 + iv * ZD,
    // signed z change per slab = B0 + iv * BD.  Exact integer arithmetic per row.
    long long Z0, ZD, B0, BD;
};

constexpr int kRowFrac = 40;  // fractional bits of the rows' fixed-point z lines

struct ColumnPlan {
    int n_columns;       // n_views * n_u
    int rows_fwd;        // detector rows per thread of the forward (1 to 4)
    int rows_bwd;        // ... of the backward and the counter
    bool bwd_interleave; // backward with 2 rows: rows interleaved across lanes
    bool fwd_ahead;      // forward gathers one slab ahead (column_slab_ahead)
    bool fwd_views_first; // forward grid: views before detector columns
};

// Zero halo (cells) around x and y of the padded working copies: the walk's
// widened slab range reaches at most this far outside the grid, so the forward
// reads zeros there and the backward's stray pieces land in cells that are
// never copied out -- no xy bounds tests in the walk.
constexpr int kHalo = 2;

// Cells of a padded z-fastest working copy.
__host__ __device__ __forceinline__ size_t column_padded_cells(const RayParams &P)
{
    return ((size_t)P.n[0] + 2 * kHalo) * ((size_t)P.n[1] + 2 * kHalo) * (size_t)P.n[2];
}

// Float64 set-up of the shared xy trace of every detector column.
__global__ void column_setup_kernel(RayParams P, ColumnTrace *__restrict__ T,
                                    int *__restrict__ flag)
{
    const long long col = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= (long long)P.n_views * P.n_u) return;
    const int view = (int)(col / P.n_u), iu = (int)(col % P.n_u);
    const ViewFrame &V = P.views[view];
    ColumnTrace C;
    C.k0 = 0;
    C.k1 = -1;
    C.tlo = 0.0f;
    C.thi = 1.0f;
    C.fb = C.bb = 0;
    C.ib = 0.0f;
    C.jb = 0;
    C.sp = C.sb = 0;
    C.addr_xy = 0;
    C.nb = 1;
    C.lxy2 = 0.0f;
    C.pad_ = 0;
    C.Z0 = C.ZD = C.B0 = C.BD = 0;

    // pixel of row 0 and the z step per row: the pitch grid, or a curved
    // detector's column (t, e fixed, s = s0 + iv ds; frames hold unit axes)
    double P0[3], dvz = V.dv[2];
    if (P.columns) {
        const ColumnOffsets q = P.columns[(P.offsets_per_view ? view * P.n_u : 0) + iu];
#pragma unroll
        for (int a = 0; a < 3; ++a)
            P0[a] = __fma_rn(q.e, V.dn[a], __fma_rn(q.s0, V.dv[a], __fma_rn(q.t, V.du[a], V.p00[a])));
        dvz = __dmul_rn(q.ds, V.dv[2]);
    } else {
#pragma unroll
        for (int a = 0; a < 3; ++a) P0[a] = __fma_rn((double)iu, V.du[a], V.p00[a]);
    }
    double X0[2], w[2];
    if (P.beam == 1) {
        for (int a = 0; a < 2; ++a) {
            X0[a] = V.a[a];
            w[a] = __dsub_rn(P0[a], V.a[a]);
        }
    } else {
        for (int a = 0; a < 2; ++a) {
            X0[a] = P0[a];
            w[a] = V.a[a];
        }
    }
    const double awx = fabs(w[0]), awy = fabs(w[1]);
    const int p = awx >= awy ? 0 : 1, b = 1 - p;
    const double awp = p == 0 ? awx : awy, awb = p == 0 ? awy : awx;
    if (!(awp > 0.0)) {  // vertical rays: not a column-path scan
        atomicOr(flag, 1);
        T[col] = C;
        return;
    }
    double A[2];
    for (int a = 0; a < 2; ++a) A[a] = w[a] < 0.0 ? __dsub_rn((double)P.n[a], X0[a]) : X0[a];
    const double inv = __ddiv_rn(1.0, awp);
    const double beta_b = __dmul_rn(awb, inv);
    const double alpha_b = __fma_rn(-A[p], beta_b, A[b]);

    double lo = 0.0, hi = (double)P.n[p];
    double lo_t = -1.0e300, hi_t = 1.0e300;
    if (P.beam == 1) {
        lo_t = A[p];
        hi_t = __dadd_rn(A[p], awp);
        lo = fmax(lo, lo_t);
        hi = fmin(hi, hi_t);
    }
    const double nb = (double)P.n[b];
    bool hit = true;
    if (beta_b > 0.0) {
        const double r = __ddiv_rn(awp, awb);
        lo = fmax(lo, __dmul_rn(-alpha_b, r));
        hi = fmin(hi, __dmul_rn(__dsub_rn(nb, alpha_b), r));
    } else if (!(alpha_b >= 0.0 && alpha_b < nb)) {
        hit = false;
    }
    if (!(lo < hi)) hit = false;
    // Slabs that hold part of [lo, hi).  The fixed-point walk and this float64
    // clip may disagree on the b entry / exit by rounding (~1e-9 slab); such a
    // sliver outside [k0, k1] is left out by forward and backward alike.  The
    // walk's b index then stays within [-2, n_b + 1], inside the zero halo.
    double k0 = fmax(floor(lo), 0.0);
    double k1 = fmin(ceil(hi) - 1.0, (double)(P.n[p] - 1));
    if (!hit || k0 > k1) {
        T[col] = C;
        return;
    }
    C.k0 = (int)k0;
    C.k1 = (int)k1;
    C.tlo = (float)fmin(fmax(__dsub_rn(lo_t, k0), 0.0), 1.0);
    C.thi = (float)fmin(fmax(__dsub_rn(hi_t, k1), 0.0), 1.0);
    const double xb = __fma_rn(k0, beta_b, alpha_b);
    const double fjb = floor(xb);
    C.jb = (int)fjb;
    C.fb = (uint32_t)__dmul_rn(__dsub_rn(xb, fjb), 4294967296.0);
    C.bb = to_fixed_slope(beta_b);
    C.ib = C.bb ? __frcp_rn((float)C.bb) : 0.0f;
    C.nb = P.n[b];
    const float sp = (float)P.spacing[p], db = (float)(P.spacing[b] * beta_b);
    C.lxy2 = __fadd_rn(__fmul_rn(sp, sp), __fmul_rn(db, db));

    // Padded z-fastest strides: x -> (ny + 2H) nz, y -> nz, z -> 1; cell (x, y)
    // sits at ((x + H) (ny + 2H) + y + H) nz.  Mirrored index j maps to n - 1 - j.
    const int stride[2] = {(P.n[1] + 2 * kHalo) * P.n[2], P.n[2]};
    int sgn[2], base = 0;
    for (int a = 0; a < 2; ++a) {
        const bool m = w[a] < 0.0;
        sgn[a] = m ? -stride[a] : stride[a];
        base += stride[a] * (m ? (P.n[a] - 1 + kHalo) : kHalo);
    }
    C.sp = sgn[p];
    C.sb = sgn[b];
    C.addr_xy = base + sgn[p] * C.k0 + sgn[b] * C.jb;

    // z of row iv at slab k0 and its slope per slab.  t(xi) = (xi - A_p) / |w_p|.
    const double lam = __dmul_rn(__dsub_rn(k0, A[p]), inv);
    double zc, zd, bc, bd;
    if (P.beam == 1) {
        const double wz0 = __dsub_rn(P0[2], V.a[2]);
        zc = __fma_rn(lam, wz0, V.a[2]);
        zd = __dmul_rn(lam, dvz);
        bc = __dmul_rn(wz0, inv);
        bd = __dmul_rn(dvz, inv);
    } else {
        zc = __fma_rn(lam, V.a[2], P0[2]);
        zd = dvz;
        bc = __dmul_rn(V.a[2], inv);
        bd = 0.0;
    }
    // every row must cross at most one z plane per slab, and the rows' z lines
    // must fit the fixed-point range (|z| < 2^21 cells at the first slab)
    const double zl = (double)(P.n_v - 1);
    const double s0 = fabs(bc), s1 = fabs(__fma_rn(zl, bd, bc));
    if (!(fmax(s0, s1) < 1.0)) atomicOr(flag, 2);
    if (!(fabs(zc) < 2097152.0 && fabs(__fma_rn(zl, zd, zc)) < 2097152.0 &&
          fabs(zd) < 32768.0)) {
        atomicOr(flag, 4);
        T[col] = C;
        return;
    }
    const double one = 1099511627776.0;  // 2^40
    C.Z0 = llrint(zc * one);
    C.ZD = llrint(zd * one);
    C.B0 = llrint(bc * one);
    C.BD = llrint(bd * one);
    T[col] = C;
}

// Per-row z state: each row's own transverse axis of the slab walk.
struct RowZ {
    uint32_t fz, bz;     // mirrored z fraction at slab k0 and slope (2^-32 cell units)
    float ibz;           // 1 / bz (0 when the row never crosses a z plane)
    int zoff;            // z index of the current cell (inside the grid iff 0 <= zoff < nz)
    int sz;              // +-1: step of zoff at a z crossing
    int kin, kout;       // slabs k in [kin, kout]: the row and its next z cell are inside
};

// Physical length per slab of a row with fixed-point z slope bz (2^-32 cell per
// slab); forward, backward and the counter all take it from here.
__device__ __forceinline__ float column_row_ell(const RayParams &P, const ColumnTrace &C,
                                                uint32_t bz)
{
    const float slope = __fmul_rn(__uint2float_rn(bz), 2.3283064365386963e-10f);  // 2^-32
    const float dz = __fmul_rn(slope, (float)P.spacing[2]);
    return __fsqrt_rn(__fadd_rn(C.lxy2, __fmul_rn(dz, dz)));
}

// A row that contributes nothing (beyond the detector, or zero weight): it stays
// in z cell 0 (a valid address) and its weight / result is zero or discarded.
__device__ __forceinline__ RowZ column_row_idle()
{
    RowZ Z;
    Z.fz = 0;
    Z.bz = 0;
    Z.ibz = 0.0f;
    Z.zoff = 0;
    Z.sz = 1;
    Z.kin = -(1 << 30);
    Z.kout = 1 << 30;
    return Z;
}

// Row set-up: this row's z line at the column's first slab, from the column's
// fixed-point affine forms -- integer arithmetic, then the walk's 2^-32 state.
__device__ __forceinline__ RowZ column_row_setup(const RayParams &P, const ColumnTrace &C, int iv)
{
    RowZ Z;
    const long long z = C.Z0 + (long long)iv * C.ZD;
    const long long b = C.B0 + (long long)iv * C.BD;
    const bool m = b < 0;
    const long long nzf = (long long)P.n[2] << kRowFrac;
    const long long absb = m ? -b : b;
    // rows far outside the grid in z touch no cell; bound them so the walk's
    // integer arithmetic stays small
    const long long lim = (long long)(65536 + P.n[2]) << kRowFrac;
    const long long zm = min(max(m ? nzf - z : z, -lim), lim);
    const int jz = (int)(zm >> kRowFrac);
    Z.fz = (uint32_t)(zm >> (kRowFrac - 32));
    const long long bq = (absb + (1LL << (kRowFrac - 33))) >> (kRowFrac - 32);
    Z.bz = bq >= 0xffffffffLL ? 0xffffffffu : (uint32_t)bq;
    Z.ibz = Z.bz ? __frcp_rn((float)Z.bz) : 0.0f;
    Z.sz = m ? -1 : 1;
    Z.zoff = m ? P.n[2] - 1 - jz : jz;
    // Slabs k where the walk's mirrored z index j(k) and j(k+1) are both in
    // [0, nz).  The walk follows zm + (k - k0) |b| to within (k1 - k0 + 2) 2^-33
    // cell (start truncated to 2^-32, slope rounded to 2^-33 per slab), so the line
    // is required to stay a margin of 1e-6 cell plus that bound inside; the
    // float32 quotients below err by far less than the one slab added to each side.
    if (absb > 0) {
        const long long margin = 1099511LL + ((long long)(C.k1 - C.k0 + 2) << (kRowFrac - 33));
        const long long lo = margin - zm;
        const long long hi = nzf - margin - zm;
        const float q_lo = fminf(__fdiv_rn((float)lo, (float)absb), 1e9f);
        const float q_hi = fmaxf(fminf(__fdiv_rn((float)hi, (float)absb), 1e9f), -1e9f);
        Z.kin = lo <= 0 ? C.k0 : C.k0 + (int)ceilf(q_lo) + 1;
        Z.kout = hi < 0 ? C.k0 - 2 : C.k0 - 1 + (int)floorf(q_hi) - 1;
    } else {
        const bool inside = jz >= 0 && jz < P.n[2];
        Z.kin = inside ? -(1 << 30) : (1 << 30);
        Z.kout = inside ? (1 << 30) : -(1 << 30);
    }
    return Z;
}

// One slab of the column walk for the R rows a thread owns.  The b (xy)
// crossing is the same for every row of the column, so the branch on it is
// taken by the whole warp and its cost is shared by the R rows; the common slab
// holds one or two pieces per row, split only by the row's own z crossing.  A
// crossing's slab fraction comes from the wrapped sum g of the fixed-point add:
// t = (beta - g) / beta = 1 - g / beta.  CLAMP restricts the slab to [lo, hi]
// (first / last slab of rays that start or end inside).  op(r, addr, length,
// on, jb) sees every piece of row r; `on` = inside the grid in z (x and y are
// covered by the zero halo), jb lets the counter test x / y.  SZ = +-1: the
// z step of every row that crosses z planes (then a row's next z cell is a
// fixed address offset from its current one); 0: each row's own.
template <int R, bool CLAMP, bool CHECK, int SZ, class Op>
__device__ __forceinline__ void column_slab(uint32_t &fb, uint32_t bb, float ib, int &jb, int sb,
                                            int &xy, int sp, RowZ (&Z)[R], unsigned nz, float lo,
                                            float hi, Op &op)
{
    const uint32_t gb = fb + bb;
    const bool cb = gb < fb;
    if (!cb) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t gz = Z[r].fz + Z[r].bz;
            const bool cz = gz < Z[r].fz;
            float e = cz ? fmaxf(__fmaf_rn(-__uint2float_rn(gz), Z[r].ibz, 1.0f), 0.0f) : 1.0f;
            if (CLAMP) e = fminf(fmaxf(e, lo), hi);
            const float d0 = CLAMP ? __fsub_rn(e, lo) : e;
            const float d1 = __fsub_rn(CLAMP ? hi : 1.0f, e);
            const int sz = SZ ? SZ : Z[r].sz;
            const int z1 = Z[r].zoff + sz;
            const int a0 = xy + Z[r].zoff;
            op(r, a0, d0, !CHECK || (unsigned)Z[r].zoff < nz, jb);
            op(r, a0 + sz, d1, cz && (!CHECK || (unsigned)z1 < nz), jb);
            Z[r].fz = gz;
            if (cz) Z[r].zoff = z1;
        }
        xy += sp;
    } else {
        const float tb = fmaxf(__fmaf_rn(-__uint2float_rn(gb), ib, 1.0f), 0.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t gz = Z[r].fz + Z[r].bz;
            const bool cz = gz < Z[r].fz;
            const float tz =
                cz ? fmaxf(__fmaf_rn(-__uint2float_rn(gz), Z[r].ibz, 1.0f), 0.0f) : 1.0f;
            const bool bfirst = tb < tz;
            float e1 = fminf(tb, tz), e2 = fmaxf(tb, tz);
            if (CLAMP) {
                e1 = fminf(fmaxf(e1, lo), hi);
                e2 = fminf(fmaxf(e2, lo), hi);
            }
            const float d1 = CLAMP ? __fsub_rn(e1, lo) : e1;
            const float d2 = __fsub_rn(e2, e1);
            const float d3 = __fsub_rn(CLAMP ? hi : 1.0f, e2);
            const int sz = SZ ? SZ : Z[r].sz;
            const int z0 = Z[r].zoff, z1 = z0 + sz;
            const bool v0 = !CHECK || (unsigned)z0 < nz, v1 = !CHECK || (unsigned)z1 < nz;
            const int a0 = xy + z0;
            op(r, a0, d1, v0, jb);
            op(r, a0 + (bfirst ? sb : sz), d2, bfirst ? v0 : v1, bfirst ? jb + 1 : jb);
            op(r, a0 + sb + sz, d3, cz && v1, jb + 1);
            Z[r].fz = gz;
            if (cz) Z[r].zoff = z1;
        }
        xy += sp + sb;
        jb += 1;
    }
    fb = gb;
}

// A check-free slab of the forward gather with its first piece's value loaded
// one slab ahead: v[r] holds the value of row r's cell at the slab's start,
// and the slab ends by loading the cell where the row's next slab starts (in
// the check-free range that cell is inside the grid: the row's z index at the
// slab's end is).  The gather's latency is then hidden behind a whole slab;
// the pieces and the order of the sums are those of column_slab.
template <int R, int SZ>
__device__ __forceinline__ void column_slab_ahead(uint32_t &fb, uint32_t bb, float ib, int &jb,
                                                  int sb, int &xy, int sp, RowZ (&Z)[R],
                                                  const float *__restrict__ vol, float (&acc)[R],
                                                  float (&v)[R], long long lim)
{
    const uint32_t gb = fb + bb;
    const bool cb = gb < fb;
    if (!cb) {
        const int nx = xy + sp;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t gz = Z[r].fz + Z[r].bz;
            const bool cz = gz < Z[r].fz;
            const float e = cz ? fmaxf(__fmaf_rn(-__uint2float_rn(gz), Z[r].ibz, 1.0f), 0.0f) : 1.0f;
            const float d1 = __fsub_rn(1.0f, e);
            const int sz = SZ ? SZ : Z[r].sz;
            const int a1 = xy + Z[r].zoff + sz;
            acc[r] = __fmaf_rn(e, v[r], acc[r]);
            if (cz && ctp_in(a1, lim, kSiteColumnGather))
                acc[r] = __fmaf_rn(d1, __ldg(vol + a1), acc[r]);
            Z[r].fz = gz;
            if (cz) Z[r].zoff += sz;
            const int an = nx + Z[r].zoff;
            v[r] = ctp_in(an, lim, kSiteColumnGather) ? __ldg(vol + an) : 0.0f;
        }
        xy = nx;
    } else {
        const float tb = fmaxf(__fmaf_rn(-__uint2float_rn(gb), ib, 1.0f), 0.0f);
        const int nx = xy + sp + sb;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t gz = Z[r].fz + Z[r].bz;
            const bool cz = gz < Z[r].fz;
            const float tz =
                cz ? fmaxf(__fmaf_rn(-__uint2float_rn(gz), Z[r].ibz, 1.0f), 0.0f) : 1.0f;
            const bool bfirst = tb < tz;
            const float e1 = fminf(tb, tz), e2 = fmaxf(tb, tz);
            const float d2 = __fsub_rn(e2, e1);
            const float d3 = __fsub_rn(1.0f, e2);
            const int sz = SZ ? SZ : Z[r].sz;
            const int a0 = xy + Z[r].zoff;
            const int a2 = a0 + (bfirst ? sb : sz), a3 = a0 + sb + sz;
            acc[r] = __fmaf_rn(e1, v[r], acc[r]);
            if (ctp_in(a2, lim, kSiteColumnGather)) acc[r] = __fmaf_rn(d2, __ldg(vol + a2), acc[r]);
            if (cz && ctp_in(a3, lim, kSiteColumnGather))
                acc[r] = __fmaf_rn(d3, __ldg(vol + a3), acc[r]);
            Z[r].fz = gz;
            if (cz) Z[r].zoff += sz;
            const int an = nx + Z[r].zoff;
            v[r] = ctp_in(an, lim, kSiteColumnGather) ? __ldg(vol + an) : 0.0f;
        }
        xy = nx;
        jb += 1;
    }
    fb = gb;
}

// Walk all slabs of a column for R rows: partial first / last slab peeled off;
// between them the slabs where every row of the warp is inside the grid in z
// (ka..kb) run without validity tests, the others with them.
template <int R, int SZ, class Op>
__device__ __forceinline__ void column_walk_sz(const ColumnTrace &C, RowZ (&Z)[R], unsigned nz,
                                               Op &op)
{
    uint32_t fb = C.fb;
    int jb = C.jb, xy = C.addr_xy;
    const uint32_t bb = C.bb;
    const float ib = C.ib;
    const int sb = C.sb, sp = C.sp;
    int kin = -(1 << 30), kout = 1 << 30;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        kin = max(kin, Z[r].kin);
        kout = min(kout, Z[r].kout);
    }
    const int ka = max(__reduce_max_sync(0xffffffffu, kin), C.k0 + 1);
    const int kb = min(__reduce_min_sync(0xffffffffu, kout), C.k1 - 1);
    column_slab<R, true, true, SZ>(fb, bb, ib, jb, sb, xy, sp, Z, nz, C.tlo,
                               C.k0 == C.k1 ? C.thi : 1.0f, op);
    int k = C.k0 + 1;
    if (ka <= kb) {
        for (; k < ka; ++k)
            column_slab<R, false, true, SZ>(fb, bb, ib, jb, sb, xy, sp, Z, nz, 0.0f, 1.0f, op);
        if constexpr (Op::kAhead) {
            // the gather: each row's first piece loaded one slab ahead
            float v[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int a = xy + Z[r].zoff;
                v[r] = ctp_in(a, op.lim, kSiteColumnGather) ? __ldg(op.vol + a) : 0.0f;
            }
            for (; k <= kb; ++k)
                column_slab_ahead<R, SZ>(fb, bb, ib, jb, sb, xy, sp, Z, op.vol, op.acc, v, op.lim);
        } else if constexpr (Op::kUnrollPairs) {
            // two slabs per iteration: the next slab's reductions issue while
            // this one's are in flight (the forward's gathers would spill)
#pragma unroll 2
            for (; k <= kb; ++k)
                column_slab<R, false, false, SZ>(fb, bb, ib, jb, sb, xy, sp, Z, nz, 0.0f, 1.0f,
                                                 op);
        } else {
            for (; k <= kb; ++k)
                column_slab<R, false, false, SZ>(fb, bb, ib, jb, sb, xy, sp, Z, nz, 0.0f, 1.0f,
                                                 op);
        }
    }
    for (; k < C.k1; ++k)
        column_slab<R, false, true, SZ>(fb, bb, ib, jb, sb, xy, sp, Z, nz, 0.0f, 1.0f, op);
    if (C.k1 > C.k0)
        column_slab<R, true, true, SZ>(fb, bb, ib, jb, sb, xy, sp, Z, nz, 0.0f, C.thi, op);
}

// The walk with the z step fixed at compile time when every row of the warp
// that crosses z planes steps the same way (all warps but those whose rows
// straddle the source's z), else per row.
template <int R, class Op>
__device__ __forceinline__ void column_walk(const ColumnTrace &C, RowZ (&Z)[R], unsigned nz,
                                            Op &op)
{
    unsigned dir = 0;
#pragma unroll
    for (int r = 0; r < R; ++r)
        if (Z[r].bz) dir |= Z[r].sz > 0 ? 1u : 2u;
    dir = __reduce_or_sync(0xffffffffu, dir);
    if (dir == 2u) column_walk_sz<R, -1>(C, Z, nz, op);
    else if (dir == 3u) column_walk_sz<R, 0>(C, Z, nz, op);
    else column_walk_sz<R, 1>(C, Z, nz, op);
}

// kUnrollPairs: the walk's check-free slab loop runs two slabs per iteration
// (measured: backward 0.7-1.4 % faster; the gather at 64 registers spills and
// slows by up to 16 %).  kAhead: the gather's check-free slabs load each row's
// first piece one slab ahead (column_slab_ahead).
template <int R, bool AHEAD = false>
struct ColumnGather {
    static constexpr bool kUnrollPairs = false;
    static constexpr bool kAhead = AHEAD;
    const float *__restrict__ vol;
    float acc[R];
    long long lim;  // cells of the padded working copy (bounds-checked builds)
    __device__ __forceinline__ void operator()(int r, int a, float d, bool on, int)
    {
        if (on && ctp_in(a, lim, kSiteColumnGather)) acc[r] = __fmaf_rn(d, __ldg(vol + a), acc[r]);
    }
};

template <int R>
struct ColumnScatter {
    static constexpr bool kUnrollPairs = true;
    static constexpr bool kAhead = false;
    float *__restrict__ vol;
    float w[R];  // ell * y of each row
    long long lim;
    __device__ __forceinline__ void operator()(int r, int a, float d, bool on, int)
    {
        if (on && d > 0.0f && w[r] != 0.0f && ctp_in(a, lim, kSiteColumnScatter))
            atomicAdd(vol + a, __fmul_rn(d, w[r]));
    }
};

template <int R>
struct ColumnCount {
    static constexpr bool kUnrollPairs = false;
    static constexpr bool kAhead = false;
    unsigned n;
    float thr[R];
    unsigned nb;
    __device__ __forceinline__ void operator()(int r, int, float d, bool on, int jb)
    {
        n += (on && (unsigned)jb < nb && d > thr[r]) ? 1u : 0u;
    }
};

constexpr int kColumnsPerBlock = 8;  // 8 warps: 8 columns, each 32 * R rows

// Rows a forward thread owns: iv = band * 32R + 32 r + lane, r < R (each load
// instruction then covers 32 adjacent rows; the backward interleaves its rows,
// see column_row_slot).
template <int R, bool AHEAD, bool VF>
__global__ void __launch_bounds__(256, R >= 4 ? 4 : 5) column_forward_kernel(RayParams P,
                                                             const ColumnTrace *__restrict__ T,
                                                             const float *__restrict__ zvol,
                                                             float *__restrict__ sino)
{
    __shared__ float tile[32 * R][kColumnsPerBlock + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // VF: grid (views, column groups, row bands), else (column groups, views, bands)
    const int ublock = VF ? (int)blockIdx.y : (int)blockIdx.x;
    const int iu = ublock * kColumnsPerBlock + warp;
    const int view = P.view0 + (int)(VF ? blockIdx.x : blockIdx.y);
    const int row0 = blockIdx.z * 32 * R + lane;
    float out[R];
#pragma unroll
    for (int r = 0; r < R; ++r) out[r] = 0.0f;
    if (iu < P.n_u) {
        const ColumnTrace C = T[(long long)view * P.n_u + iu];
        if (C.k0 <= C.k1) {
            RowZ Z[R];
            ColumnGather<R, AHEAD> op;
            op.vol = zvol;
            op.lim = (long long)column_padded_cells(P);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int iv = row0 + 32 * r;
                Z[r] = iv < P.n_v ? column_row_setup(P, C, iv) : column_row_idle();
                op.acc[r] = 0.0f;
            }
            column_walk<R>(C, Z, (unsigned)P.n[2], op);
#pragma unroll
            for (int r = 0; r < R; ++r)
                out[r] = __fmul_rn(op.acc[r], column_row_ell(P, C, Z[r].bz));
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) tile[lane + 32 * r][warp] = out[r];
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * R * kColumnsPerBlock; e += 256) {
        const int rr = e / kColumnsPerBlock, c = e % kColumnsPerBlock;
        const int ivw = blockIdx.z * 32 * R + rr, iuw = ublock * kColumnsPerBlock + c;
        const long long ray = ((long long)view * P.n_v + ivw) * P.n_u + iuw;
        if (ivw < P.n_v && iuw < P.n_u && ctp_in(ray, sino_cells(P), kSiteColumnSinoStore))
            sino[ray] = tile[rr][c];
    }
}

// Row of slot r of a lane.  STRIDED: row lane + 32 r (an instruction covers 32
// adjacent rows); INTERLEAVED: row R lane + r (an instruction covers every R-th
// row of the warp's 32 R rows, so with rows under ~1 z cell apart its lanes hit
// distinct cells: a reduction instruction with repeated addresses costs a
// sector request per repeat).
template <int R, bool INTERLEAVED>
__device__ __forceinline__ int column_row_slot(int lane, int r)
{
    return INTERLEAVED ? R * lane + r : lane + 32 * r;
}

template <int R, bool INTERLEAVED = false>
__global__ void __launch_bounds__(256, 4) column_backward_kernel(RayParams P,
                                                              const ColumnTrace *__restrict__ T,
                                                              const float *__restrict__ sino,
                                                              float *__restrict__ zvol)
{
    __shared__ float tile[32 * R][kColumnsPerBlock + 1];
    const int view = P.view0 + (int)blockIdx.y;
    for (int e = threadIdx.x; e < 32 * R * kColumnsPerBlock; e += 256) {
        const int rr = e / kColumnsPerBlock, c = e % kColumnsPerBlock;
        const int ivr = blockIdx.z * 32 * R + rr, iur = blockIdx.x * kColumnsPerBlock + c;
        const long long ray = ((long long)view * P.n_v + ivr) * P.n_u + iur;
        tile[rr][c] = (ivr < P.n_v && iur < P.n_u && ctp_in(ray, sino_cells(P), kSiteColumnSinoLoad))
                          ? sino[ray]
                          : 0.0f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int iu = blockIdx.x * kColumnsPerBlock + warp;
    if (iu >= P.n_u) return;
    const ColumnTrace C = T[(long long)view * P.n_u + iu];
    if (C.k0 > C.k1) return;
    RowZ Z[R];
    ColumnScatter<R> op;
    op.vol = zvol;
    op.lim = (long long)column_padded_cells(P);
    bool any = false;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int slot = column_row_slot<R, INTERLEAVED>(lane, r);
        const int iv = blockIdx.z * 32 * R + slot;
        const float y = tile[slot][warp];
        const bool live = iv < P.n_v && y != 0.0f;
        Z[r] = live ? column_row_setup(P, C, iv) : column_row_idle();
        op.w[r] = live ? __fmul_rn(column_row_ell(P, C, Z[r].bz), y) : 0.0f;
        any |= op.w[r] != 0.0f;
    }
    if (!__any_sync(0xffffffffu, any)) return;
    column_walk<R>(C, Z, (unsigned)P.n[2], op);
}

template <int R>
__global__ void __launch_bounds__(256) column_count_kernel(RayParams P,
                                                           const ColumnTrace *__restrict__ T,
                                                           unsigned long long *__restrict__ total)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int iu = blockIdx.x * kColumnsPerBlock + warp;
    const int view = P.view0 + (int)blockIdx.y;
    const int row0 = blockIdx.z * 32 * R + lane;
    unsigned n = 0;
    if (iu < P.n_u) {
        const ColumnTrace C = T[(long long)view * P.n_u + iu];
        if (C.k0 <= C.k1) {
            RowZ Z[R];
            ColumnCount<R> op;
            op.n = 0u;
            op.nb = (unsigned)C.nb;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int iv = row0 + 32 * r;
                const bool live = iv < P.n_v;
                Z[r] = live ? column_row_setup(P, C, iv) : column_row_idle();
                op.thr[r] = live ? __fdiv_rn(P.min_len, column_row_ell(P, C, Z[r].bz)) : 3.0e38f;
            }
            column_walk<R>(C, Z, (unsigned)P.n[2], op);
            n = op.n;
        }
    }
    n = __reduce_add_sync(0xffffffffu, n);
    if (lane == 0 && n) atomicAdd(total, (unsigned long long)n);
}

// (nz, ny, nx) x-fastest  ->  padded (nx + 2H, ny + 2H, nz) z-fastest interior,
// one y plane per grid row; the halo is left untouched.
__global__ void __launch_bounds__(256) xfast_to_zfast_kernel(const float *__restrict__ in,
                                                             float *__restrict__ out, int nx,
                                                             int ny, int nz)
{
    __shared__ float tile[32][33];
    const int x0 = blockIdx.x * 32, z0 = blockIdx.y * 32, y = blockIdx.z;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const size_t pny = (size_t)ny + 2 * kHalo;
    for (int j = ty; j < 32; j += 8) {
        const int z = z0 + j, x = x0 + tx;
        if (z < nz && x < nx) tile[j][tx] = in[((size_t)z * ny + y) * nx + x];
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int x = x0 + j, z = z0 + tx;
        const long long o = ((long long)(x + kHalo) * pny + (y + kHalo)) * nz + z;
        if (x < nx && z < nz &&
            ctp_in(o, ((long long)nx + 2 * kHalo) * (long long)pny * nz, kSiteColumnLayoutIn))
            out[o] = tile[tx][j];
    }
}

// Padded z-fastest interior  ->  (nz, ny, nx) x-fastest.
__global__ void __launch_bounds__(256) zfast_to_xfast_kernel(const float *__restrict__ in,
                                                             float *__restrict__ out, int nx,
                                                             int ny, int nz)
{
    __shared__ float tile[32][33];
    const int x0 = blockIdx.x * 32, z0 = blockIdx.y * 32, y = blockIdx.z;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const size_t pny = (size_t)ny + 2 * kHalo;
    for (int j = ty; j < 32; j += 8) {
        const int x = x0 + j, z = z0 + tx;
        const long long o = ((long long)(x + kHalo) * pny + (y + kHalo)) * nz + z;
        if (x < nx && z < nz &&
            ctp_in(o, ((long long)nx + 2 * kHalo) * (long long)pny * nz, kSiteColumnLayoutOut))
            tile[j][tx] = in[o];
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int z = z0 + j, x = x0 + tx;
        if (z < nz && x < nx) out[((size_t)z * ny + y) * nx + x] = tile[tx][j];
    }
}


// Rows per thread.  The shared xy walk is paid once per R rows, at the cost of
// registers.  The forward gather runs 4 rows (4 blocks of 256 threads per SM,
// 64 registers; 2 rows at 5 blocks on short detectors); the backward, bound by
// its atomics' L1/L2 throughput, runs 2 rows at 4 blocks per SM.  A plan
// option (1 to 4; 0 = this choice) overrides it.
inline int column_rows(const RayParams &P, int requested, int preferred)
{
    if (requested >= 1 && requested <= 4) return requested;
    int r = preferred;
    while (r > 1 && P.n_v < 24 * r) r /= 2;
    return r;
}

// Builds the column table and the two padded working copies (forward: halo
// zeroed once here and never written again; backward: zeroed per call).
// Returns 0, 9 (CUDA error) or 11 (scan not eligible for the column path).
// rows_fwd / rows_bwd: requested rows per thread (0 = the measured default);
// bwd_adjacent: the 2-row backward covers 32 adjacent rows per instruction
// instead of interleaving a thread's rows across lanes.
inline int column_plan_build(const RayParams &P, int rows_fwd, int rows_bwd, bool bwd_adjacent,
                             int fwd_ahead, bool fwd_views_first, ColumnPlan *plan,
                             void **d_columns, float **d_zfwd, float **d_zbwd,
                             unsigned long long *bytes)
{
    if ((long long)P.n_views * P.n_u >= (1LL << 31)) return 11;
    if (column_padded_cells(P) >= (1ULL << 31)) return 11;
    plan->n_columns = P.n_views * P.n_u;
    plan->rows_fwd = column_rows(P, rows_fwd, 4);
    plan->rows_bwd = column_rows(P, rows_bwd, 2);
    plan->bwd_interleave = !bwd_adjacent;
    // The forward's resident blocks read the volume along their rays: in the
    // default order (columns, then views) they cover a few views of every
    // column, the whole band of the volume, re-read from DRAM view after view;
    // views first they cover many angles of a few columns, a thin shell that L2
    // holds (C4 forward 104.3 -> 99.5 ms, C3 10.43 -> 10.36 ms).  Not for
    // helical scans, whose consecutive views move in z (C5 26.0 -> 27.5 ms),
    // nor for the backward, whose reductions then pile onto the same lines
    // (C4 159.3 -> 169.5 ms).
    plan->fwd_views_first = fwd_views_first;
    // Loading a slab ahead hides the latency of gathers that miss L2: measured
    // faster where the blocks run columns first over a working copy larger
    // than L2 (C5 26.2 -> 26.0 ms; C4 106.4 -> 104.3 ms in that order) and
    // slower where the reads stay in L2: a copy that fits (C3 10.4 -> 10.9 ms)
    // or the views-first order (C4 93.3 -> 99.4 ms).  fwd_ahead: 0 = by that
    // rule, 1 = never, 2 = always.
    int dev = 0, l2 = 0;
    if (fwd_ahead == 0 && (cudaGetDevice(&dev) != cudaSuccess ||
                           cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess))
        return 9;
    plan->fwd_ahead = fwd_ahead == 2 ||
                      (fwd_ahead == 0 && !fwd_views_first &&
                       sizeof(float) * column_padded_cells(P) > (size_t)l2);
    const size_t cbytes = sizeof(ColumnTrace) * (size_t)(plan->n_columns > 0 ? plan->n_columns : 1);
    const size_t vbytes = sizeof(float) * column_padded_cells(P);
    int *d_flag = nullptr;
    if (cudaMalloc(d_columns, cbytes) != cudaSuccess || cudaMalloc(d_zfwd, vbytes) != cudaSuccess ||
        cudaMalloc(d_zbwd, vbytes) != cudaSuccess || cudaMemset(*d_zfwd, 0, vbytes) != cudaSuccess ||
        cudaMalloc(&d_flag, sizeof(int)) != cudaSuccess ||
        cudaMemset(d_flag, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(d_flag);
        return 9;
    }
    *bytes += cbytes + 2 * vbytes;
    if (plan->n_columns > 0) {
        const int threads = 128;
        const int blocks = (plan->n_columns + threads - 1) / threads;
        column_setup_kernel<<<blocks, threads>>>(P, (ColumnTrace *)*d_columns, d_flag);
    }
    int flag = 0;
    const bool ok = cudaGetLastError() == cudaSuccess &&
                    cudaMemcpy(&flag, d_flag, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaFree(d_flag);
    if (!ok) return 9;
    if (flag) return 11;
    return 0;
}

inline dim3 column_grid_views_first(const RayParams &P, int R)
{
    return dim3(P.view_count, (P.n_u + kColumnsPerBlock - 1) / kColumnsPerBlock,
                (P.n_v + 32 * R - 1) / (32 * R));
}

inline dim3 column_grid(const RayParams &P, int R)
{
    return dim3((P.n_u + kColumnsPerBlock - 1) / kColumnsPerBlock, P.view_count,
                (P.n_v + 32 * R - 1) / (32 * R));
}

inline dim3 transpose_grid(const RayParams &P)
{
    return dim3((P.n[0] + 31) / 32, (P.n[2] + 31) / 32, P.n[1]);
}

// Stages of a call: layout in (forward), walk over P's view range, layout out
// (backward).  ctp_forward / ctp_backward run them over all views; the host-
// buffer entry points run the walk in view chunks overlapped with copies.
inline int column_layout_in(const RayParams &P, float *d_zfwd, const float *vol, cudaStream_t s)
{
    xfast_to_zfast_kernel<<<transpose_grid(P), 256, 0, s>>>(vol, d_zfwd, P.n[0], P.n[1], P.n[2]);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

template <bool AHEAD, bool VF>
inline void column_forward_launch(const RayParams &P, int R, const ColumnTrace *T,
                                  const float *d_zfwd, float *sino, cudaStream_t s)
{
    const dim3 g = VF ? column_grid_views_first(P, R) : column_grid(P, R);
    if (R == 4) column_forward_kernel<4, AHEAD, VF><<<g, 256, 0, s>>>(P, T, d_zfwd, sino);
    else if (R == 3) column_forward_kernel<3, AHEAD, VF><<<g, 256, 0, s>>>(P, T, d_zfwd, sino);
    else if (R == 2) column_forward_kernel<2, AHEAD, VF><<<g, 256, 0, s>>>(P, T, d_zfwd, sino);
    else column_forward_kernel<1, AHEAD, VF><<<g, 256, 0, s>>>(P, T, d_zfwd, sino);
}

inline int column_walk_forward(const RayParams &P, const ColumnPlan &plan, const void *d_columns,
                               const float *d_zfwd, float *sino, cudaStream_t s)
{
    if (P.view_count <= 0) return 0;
    const ColumnTrace *T = (const ColumnTrace *)d_columns;
    const int R = plan.rows_fwd;
    if (plan.fwd_ahead && plan.fwd_views_first)
        column_forward_launch<true, true>(P, R, T, d_zfwd, sino, s);
    else if (plan.fwd_ahead)
        column_forward_launch<true, false>(P, R, T, d_zfwd, sino, s);
    else if (plan.fwd_views_first)
        column_forward_launch<false, true>(P, R, T, d_zfwd, sino, s);
    else
        column_forward_launch<false, false>(P, R, T, d_zfwd, sino, s);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int column_backward_prepare(const RayParams &P, float *d_zbwd, cudaStream_t s)
{
    return cudaMemsetAsync(d_zbwd, 0, sizeof(float) * column_padded_cells(P), s) == cudaSuccess ? 0 : 9;
}

inline int column_walk_backward(const RayParams &P, const ColumnPlan &plan, const void *d_columns,
                                const float *sino, float *d_zbwd, cudaStream_t s)
{
    if (P.view_count <= 0 || P.n_u <= 0 || P.n_v <= 0) return 0;
    const ColumnTrace *T = (const ColumnTrace *)d_columns;
    const int R = plan.rows_bwd;
    // rows interleaved across lanes (measured 1-4 % faster on the cone scans)
    const bool il = plan.bwd_interleave;
    if (R == 4) column_backward_kernel<4><<<column_grid(P, 4), 256, 0, s>>>(P, T, sino, d_zbwd);
    else if (R == 3) column_backward_kernel<3><<<column_grid(P, 3), 256, 0, s>>>(P, T, sino, d_zbwd);
    else if (R == 2 && il)
        column_backward_kernel<2, true><<<column_grid(P, 2), 256, 0, s>>>(P, T, sino, d_zbwd);
    else if (R == 2) column_backward_kernel<2><<<column_grid(P, 2), 256, 0, s>>>(P, T, sino, d_zbwd);
    else column_backward_kernel<1><<<column_grid(P, 1), 256, 0, s>>>(P, T, sino, d_zbwd);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int column_layout_out(const RayParams &P, const float *d_zbwd, float *vol, cudaStream_t s)
{
    zfast_to_xfast_kernel<<<transpose_grid(P), 256, 0, s>>>(d_zbwd, vol, P.n[0], P.n[1], P.n[2]);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int column_count(const RayParams &P, const ColumnPlan &plan, const void *d_columns,
                        unsigned long long *d_total, cudaStream_t s)
{
    const ColumnTrace *T = (const ColumnTrace *)d_columns;
    const int R = plan.rows_bwd;
    if (R == 4) column_count_kernel<4><<<column_grid(P, 4), 256, 0, s>>>(P, T, d_total);
    else if (R == 3) column_count_kernel<3><<<column_grid(P, 3), 256, 0, s>>>(P, T, d_total);
    else if (R == 2) column_count_kernel<2><<<column_grid(P, 2), 256, 0, s>>>(P, T, d_total);
    else column_count_kernel<1><<<column_grid(P, 1), 256, 0, s>>>(P, T, d_total);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

}  // namespace ctp
