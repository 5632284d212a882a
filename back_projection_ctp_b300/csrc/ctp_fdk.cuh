// Analytical FBP / FDK operators on a plan's geometry: the ramp filter (with
// its cosine and view weights), the voxel-driven weighted gather with bilinear
// interpolation, and the gather's exact transpose.
//
// What they compute (diffct release pages, my.diffend.io): the analytical
// helpers -- ramp filters (Ram-Lak and Shepp-Logan among them), fan / cone
// weights and FBP / FDK backprojection (diffct 2.1.0 -> 2.2.1, README
// "Analytical helpers"); a voxel-driven gather, one thread per output voxel,
// with the analytical constant 1/(2 pi) (parallel) or SDD/(2 pi SID) per view
// (fan, cone), and a dedicated transpose of the same interpolation stencil
// (diffct 2.1.0 -> 2.2.1 and 2.4.3 -> 2.4.4, diffct/analytical.py,
// `_analytical_transpose_raw`; README "Differentiable FBP and FDK").
//
//   filter:    q[k,iv,i] = post * tau * sum_j h[i-j] * pre * p[k,iv,j]
//              (forward: pre = cosine weight SDD/|P_pix - a|, post = view
//              weight w_k; transpose: pre = w_k, post = cosine weight)
//   gather:    g(x) = sum_k s_k (SID_k / U_k(x))^2 I(q_k; u_k(x), v_k(x))
//   transpose: scatter of s_k W_k g(x) onto the same bilinear stencil.
//
// B300 design.  Per view the detector coordinates of a voxel centre are ratios
// of affine functions of the voxel index, u = Nu / E and v = Nv / E with E =
// depth / SID.  For scans whose detector v axis is +-z and whose u axis is
// horizontal (the circular and helical cone scans, and every 2-D scan), E and
// Nu do not depend on z: a thread owns K voxels of one (x, y) column, and per
// view it evaluates the affine forms exactly in 64-bit fixed point (2^-40) and
// divides exactly (float estimate of the floor, integer remainder), so the
// interpolation fractions are good to ~1e-7 pixel without float64 arithmetic,
// which runs at a small fraction of the float32 rate on this part.  Along the
// column v advances by the fixed step Nv_z / E, split into integer and
// fractional parts.  Lanes of a warp are consecutive x, so the four stencil
// loads of a warp touch neighbouring pixels of two detector rows.
#pragma once

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <vector>

#include <cuda_runtime.h>

#include "ctp_check.h"

// Operands of the bounds-check hooks (they appear only inside CTP_AND_IN and
// CTP_CHECKED_LDG, which drop them in normal builds): the element of row iv,
// column C.iu of a view's detector plane, and the plane's size.
#define CTP_FDK_ELEM ((long long)iv * F.n_u + C.iu)
#define CTP_FDK_PLANE ((long long)F.n_u * F.n_v)

namespace ctp {

constexpr double kFixOne = 1099511627776.0;  // 2^40
constexpr float kFixInv = 9.094947017729282e-13f;  // 2^-40

// Per-view constants, fixed point 2^-40 for the affine forms in voxel indices
// (i, j, k) = (x, y, z).
struct FdkView {
    long long e[3];    // depth / SID = e0 + e1 i + e2 j (parallel: 1)
    long long nu[3];   // u * depth / SID
    long long nv[4];   // v * depth / SID, including the z term nv[3] k
    float scale;       // SDD / (2 pi SID); parallel 1 / (2 pi)
    float sdd;         // cosine weight SDD / |P_pix - a| (parallel: unused)
    float g[6];        // |c-a|^2, (c-a).u, (c-a).v, u.v, |u|^2, |v|^2
};

struct FdkParams {
    const FdkView *views;
    int n_views, n_u, n_v;
    int n[3];
    int ndim, beam;
    float pitch_u, pitch_v;
    float cu, cv;      // pixel index of the detector centre: (n - 1)/2 - offset
    int tx;            // warp tile width in x (32, 16, 8 or 4)
};

// Warp tile width in x: 8 x 4 columns per warp (measured against 32 x 1,
// 16 x 2 and 4 x 8 on the cone scans: the warp's stencils of one view then fall
// on the fewest detector rows).
constexpr int kFdkTileX = 8;

// A 64-bit integer as float from its two 32-bit halves (relative error below
// 2^-23): 32-bit conversions, where a 64-bit conversion would run on the slow
// float64 pipe.
__device__ __forceinline__ float i64_to_float(long long x)
{
    return __fmaf_rn(__int2float_rn((int)(x >> 32)), 4294967296.0f,
                     __uint2float_rn((unsigned)(x & 0xffffffffLL)));
}

// floor(num / den) and its fraction, exactly up to the final float rounding of
// the fraction; den > 0, rden ~ 1 / den.  False when |num / den| >= 2^20 (far
// off the detector).
__device__ __forceinline__ bool fix_floor_div(long long num, long long den, float rden, int &q,
                                              float &f)
{
    const float qf = floorf(i64_to_float(num) * rden);
    if (!(fabsf(qf) < 1048576.0f)) return false;
    q = (int)qf;
    long long r = num - (long long)q * den;
    // the float estimate is off by at most one
    if (r < 0) {
        r += den;
        q -= 1;
    } else if (r >= den) {
        r -= den;
        q += 1;
    }
    f = fminf(i64_to_float(r) * rden, 0.99999994f);
    return true;
}

// Per (column, view) set-up shared by the gather and the scatter.  Returns false
// when the view contributes nothing to this column.
struct ColumnView {
    int iu, iv, dvi;
    float fu, fv, dvf, w;
    bool c0, c1;
};

__device__ __forceinline__ bool fdk_column_view(const FdkParams &F, const FdkView &V, int i, int j,
                                                int k0, ColumnView &C)
{
    const long long den = V.e[0] + V.e[1] * i + V.e[2] * j;
    if (den < (1LL << 20)) return false;  // depth below 1e-6 SID: behind or at the source
    const float denf = i64_to_float(den);
    const float rden = __frcp_rn(denf);
    if (!fix_floor_div(V.nu[0] + V.nu[1] * i + V.nu[2] * j, den, rden, C.iu, C.fu)) return false;
    if (C.iu < -1 || C.iu >= F.n_u) return false;
    const float ef = denf * kFixInv;
    C.w = __fdividef(V.scale, ef * ef);
    C.c0 = C.iu >= 0;
    C.c1 = C.iu + 1 < F.n_u;
    if (F.ndim == 2) {
        C.iv = 0;
        C.fv = 0.0f;
        C.dvi = 0;
        C.dvf = 0.0f;
        return true;
    }
    if (!fix_floor_div(V.nv[0] + V.nv[1] * i + V.nv[2] * j + V.nv[3] * k0, den, rden, C.iv, C.fv))
        return false;
    // the step per z voxel needs no exact division: its float rounding (2^-24
    // relative) accumulates over at most K steps from the exact start
    const float dv = i64_to_float(V.nv[3]) * rden;
    if (!(fabsf(dv) < 1048576.0f)) return false;
    const float dfl = floorf(dv);
    C.dvi = (int)dfl;
    C.dvf = fminf(dv - dfl, 0.99999994f);
    return true;
}

// Column (i, j) of a thread.  A block covers 32 x 8 columns; a warp covers tx x
// (32 / tx) of them (tx = 32, 16, 8 or 4), so that in every view the warp's
// stencils stay close on the detector: along a ray parallel to x the 32 columns
// of a 32 x 1 warp lie at 32 different depths and, away from the mid-plane,
// on as many different detector rows.
__device__ __forceinline__ void fdk_column_of(int tx, int &i, int &j)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wx = 32 / tx;                  // warps across x
    i = blockIdx.x * 32 + (warp % wx) * tx + lane % tx;
    j = blockIdx.y * 8 + (warp / wx) * (32 / tx) + lane / tx;
}

// True when no stencil row of the K steps is on the detector: the rows of step
// t lie in [iv + t dvi, iv + t (dvi + 1) + 1].
template <int K>
__device__ __forceinline__ bool fdk_rows_miss(const FdkParams &F, const ColumnView &C)
{
    return C.iv + (K - 1) * max(C.dvi + 1, 0) + 1 < 0 || C.iv + (K - 1) * min(C.dvi, 0) >= F.n_v;
}

// The K updates of one column in one view, stencil values read straight from
// the filtered sinogram.  Rows of step t lie in [iv + t dvi, iv + t (dvi + 1)];
// when the stencils of all K steps are on the detector the loop runs without
// tests.
template <int K>
__device__ __forceinline__ void gather_column(const FdkParams &F, const ColumnView &C,
                                              const float *__restrict__ base, float (&acc)[K])
{
    int iv = C.iv;
    float fv = C.fv;
    const bool inside = C.c0 && C.c1 && iv + (K - 1) * min(C.dvi, 0) >= 0 &&
                        iv + (K - 1) * max(C.dvi + 1, 0) + 1 < F.n_v;
    if (inside) {
        const float *col = base + C.iu;
#pragma unroll
        for (int t = 0; t < K; ++t) {
            const float *row = col + (long long)iv * F.n_u;
            const float a0 = CTP_CHECKED_LDG(row, CTP_FDK_ELEM, CTP_FDK_PLANE, kSiteFdkGather),
                        a1 = CTP_CHECKED_LDG(row + 1, CTP_FDK_ELEM + 1, CTP_FDK_PLANE, kSiteFdkGather);
            const float b0 = CTP_CHECKED_LDG(row + F.n_u, CTP_FDK_ELEM + F.n_u, CTP_FDK_PLANE, kSiteFdkGather),
                        b1 = CTP_CHECKED_LDG(row + F.n_u + 1, CTP_FDK_ELEM + F.n_u + 1, CTP_FDK_PLANE,
                                             kSiteFdkGather);
            const float a = __fmaf_rn(C.fu, a1 - a0, a0);
            const float b = __fmaf_rn(C.fu, b1 - b0, b0);
            acc[t] = __fmaf_rn(C.w, __fmaf_rn(fv, b - a, a), acc[t]);
            fv += C.dvf;
            iv += C.dvi;
            if (fv >= 1.0f) {
                fv -= 1.0f;
                iv += 1;
            }
        }
        return;
    }
#pragma unroll
    for (int t = 0; t < K; ++t) {
        const bool r0 = (unsigned)iv < (unsigned)F.n_v;
        const bool r1 = (unsigned)(iv + 1) < (unsigned)F.n_v;
        if (r0 || r1) {
            const float *row = base + (long long)iv * F.n_u + C.iu;
            const float a0 = (r0 && C.c0 CTP_AND_IN(CTP_FDK_ELEM, CTP_FDK_PLANE, kSiteFdkGather)) ? __ldg(row)
                                                                                     : 0.0f;
            const float a1 = (r0 && C.c1 CTP_AND_IN(CTP_FDK_ELEM + 1, CTP_FDK_PLANE, kSiteFdkGather))
                                 ? __ldg(row + 1) : 0.0f;
            const float b0 = (r1 && C.c0 CTP_AND_IN(CTP_FDK_ELEM + F.n_u, CTP_FDK_PLANE, kSiteFdkGather))
                                 ? __ldg(row + F.n_u) : 0.0f;
            const float b1 = (r1 && C.c1 CTP_AND_IN(CTP_FDK_ELEM + F.n_u + 1, CTP_FDK_PLANE, kSiteFdkGather))
                                 ? __ldg(row + F.n_u + 1) : 0.0f;
            const float a = __fmaf_rn(C.fu, a1 - a0, a0);
            const float b = __fmaf_rn(C.fu, b1 - b0, b0);
            acc[t] = __fmaf_rn(C.w, __fmaf_rn(fv, b - a, a), acc[t]);
        }
        fv += C.dvf;
        iv += C.dvi;
        if (fv >= 1.0f) {
            fv -= 1.0f;
            iv += 1;
        }
    }
}

template <int K>
__device__ __forceinline__ void store_column(const FdkParams &F, int i, int j, int k0,
                                             const float (&acc)[K], float *__restrict__ vol)
{
    const int kn = F.ndim == 2 ? 1 : K;
#pragma unroll
    for (int t = 0; t < K; ++t)
        if (t < kn && k0 + t < F.n[2] CTP_AND_IN(((long long)(k0 + t) * F.n[1] + j) * F.n[0] + i,
                                                 (long long)F.n[0] * F.n[1] * F.n[2],
                                                 kSiteFdkStore))
            vol[((long long)(k0 + t) * F.n[1] + j) * F.n[0] + i] = acc[t];
}

// One thread per (x, y) column and K consecutive z; blocks of 32 x 8 columns;
// stencil values straight from global memory (2-D scans, and a tuning override).
// 3-D: 4 blocks per SM (64 registers) with the view loop unrolled by two; 5
// blocks (48 registers, spilling) measured C3 8.61 / C4 101.2 / C5 55.2 ms
// against 8.14 / 97.2 / 57.3.
template <int K>
__global__ void __launch_bounds__(256, K > 1 ? 4 : 8) wbp_gather_kernel(FdkParams F, const float *__restrict__ q,
                                                         float *__restrict__ vol)
{
    int i, j;
    fdk_column_of(F.tx, i, j);
    const int k0 = blockIdx.z * K;
    if (i >= F.n[0] || j >= F.n[1]) return;
    float acc[K];
#pragma unroll
    for (int t = 0; t < K; ++t) acc[t] = 0.0f;
    const long long plane = (long long)F.n_u * F.n_v;
    // two views per iteration: the second view's set-up chain overlaps the
    // first's (C3 / C4 / C5 gather 6-7 % faster; the same for the transpose
    // measured no faster)
#pragma unroll 2
    for (int s = 0; s < F.n_views; ++s) {
        ColumnView C;
        if (!fdk_column_view(F, F.views[s], i, j, k0, C)) continue;
        const float *base = q + s * plane;
        if (F.ndim == 2) {
            const float a0 = C.c0 CTP_AND_IN(C.iu, CTP_FDK_PLANE, kSiteFdkGather) ? __ldg(base + C.iu)
                                                                          : 0.0f;
            const float a1 = C.c1 CTP_AND_IN(C.iu + 1, CTP_FDK_PLANE, kSiteFdkGather)
                                 ? __ldg(base + C.iu + 1) : 0.0f;
            acc[0] = __fmaf_rn(C.w, __fmaf_rn(C.fu, a1 - a0, a0), acc[0]);
            continue;
        }
        if (fdk_rows_miss<K>(F, C)) continue;
        gather_column<K>(F, C, base, acc);
    }
    store_column<K>(F, i, j, k0, acc, vol);
}

// Transpose: the same stencil, each voxel's s_k W_k g reduced with float
// atomics into a zeroed sinogram.  In 3-D the taps of consecutive z steps on a
// shared detector row are first summed in registers: the stencil rows of step
// t are (iv, iv + 1) and iv moves monotonically by floor(dv) or floor(dv) + 1
// per step, so a row pair overlaps the previous one in at most one row (or
// both, for steps under a pixel).  The pending pair (pa at row P, pb at row
// P + 1) takes the new step's taps where rows coincide and is reduced into the
// sinogram only when a row is left (C4 transpose 370 -> 288 ms on B300).
template <int K>
__global__ void __launch_bounds__(256, K > 1 ? 4 : 8) wbp_scatter_kernel(FdkParams F,
                                                          const float *__restrict__ vol,
                                                          float *__restrict__ q)
{
    int i, j;
    fdk_column_of(F.tx, i, j);
    const int k0 = blockIdx.z * K;
    if (i >= F.n[0] || j >= F.n[1]) return;
    const int kn = F.ndim == 2 ? 1 : K;
    float g[K];
#pragma unroll
    for (int t = 0; t < K; ++t)
        g[t] = (t < kn && k0 + t < F.n[2] CTP_AND_IN(((long long)(k0 + t) * F.n[1] + j) * F.n[0] + i,
                                                     (long long)F.n[0] * F.n[1] * F.n[2],
                                                     kSiteFdkScatterLoad))
                   ? vol[((long long)(k0 + t) * F.n[1] + j) * F.n[0] + i] : 0.0f;
    const long long plane = (long long)F.n_u * F.n_v;
    for (int s = 0; s < F.n_views; ++s) {
        ColumnView C;
        if (!fdk_column_view(F, F.views[s], i, j, k0, C)) continue;
        if (F.ndim == 2) {
            float *base = q + s * plane;
            const float val = C.w * g[0];
            if (val != 0.0f) {
                if (C.c0 CTP_AND_IN(C.iu, CTP_FDK_PLANE, kSiteFdkScatter))
                    atomicAdd(base + C.iu, val * (1.0f - C.fu));
                if (C.c1 CTP_AND_IN(C.iu + 1, CTP_FDK_PLANE, kSiteFdkScatter))
                    atomicAdd(base + C.iu + 1, val * C.fu);
            }
            continue;
        }
        if (fdk_rows_miss<K>(F, C)) continue;
        float *col = q + s * plane + C.iu;
        const float wu0 = C.c0 ? 1.0f - C.fu : 0.0f, wu1 = C.c1 ? C.fu : 0.0f;
        // reduce row r's value x into the sinogram (both columns)
        auto flush = [&](int r, float x) {
            if ((unsigned)r < (unsigned)F.n_v && x != 0.0f) {
                float *px = col + (long long)r * F.n_u;
                if (C.c0 CTP_AND_IN((long long)r * F.n_u + C.iu, CTP_FDK_PLANE, kSiteFdkScatter))
                    atomicAdd(px, x * wu0);
                if (C.c1 CTP_AND_IN((long long)r * F.n_u + C.iu + 1, CTP_FDK_PLANE, kSiteFdkScatter))
                    atomicAdd(px + 1, x * wu1);
            }
        };
        int P = C.iv;
        float fv = C.fv;
        float pa = C.w * g[0] * (1.0f - fv), pb = C.w * g[0] * fv;
#pragma unroll
        for (int t = 1; t < K; ++t) {
            // the step from the previous row P, as in the gather
            fv += C.dvf;
            int iv = P + C.dvi;
            if (fv >= 1.0f) {
                fv -= 1.0f;
                iv += 1;
            }
            const float val = C.w * g[t];
            const float va = val * (1.0f - fv), vb = val * fv;
            const int d = iv - P;
            if (d != 0 && d != -1) flush(P, pa);
            if (d != 0 && d != 1) flush(P + 1, pb);
            const float na = d == 0 ? pa + va : (d == 1 ? pb + va : va);
            const float nb = d == 0 ? pb + vb : (d == -1 ? pa + vb : vb);
            pa = na;
            pb = nb;
            P = iv;
        }
        flush(P, pa);
        flush(P + 1, pb);
    }
}

// Cosine of pixel (iu, iv)'s ray to the detector normal: SDD / |P_pix - a|.
__device__ __forceinline__ float fdk_cosine(const FdkParams &F, const FdkView &V, int iu, int iv)
{
    if (F.beam != 1) return 1.0f;
    const float al = ((float)iu - F.cu) * F.pitch_u;
    const float be = F.ndim == 2 ? 0.0f : ((float)iv - F.cv) * F.pitch_v;
    const float d2 = V.g[0] + 2.0f * al * V.g[1] + 2.0f * be * V.g[2] + 2.0f * al * be * V.g[3] +
                     al * al * V.g[4] + be * be * V.g[5];
    return __fdiv_rn(V.sdd, __fsqrt_rn(d2));
}

// Ramp filter along u: RB detector rows per block staged in shared memory with
// the kernel h; each thread forms 4 outputs (stride blockDim) of every row, so
// per input sample it issues RB + 4 shared loads (the row values are warp
// broadcasts, the kernel values consecutive) for 4 RB fused multiply-adds.
template <int RB, bool ODD>
__global__ void ramp_filter_kernel(FdkParams F, const float *__restrict__ h,
                                   const float *__restrict__ x, float *__restrict__ out,
                                   const float *__restrict__ view_weight,
                                   const float *__restrict__ pixel_weight, int transpose,
                                   long long n_rows)
{
    extern __shared__ float sm[];
    const int nu = F.n_u;
    float *xs = sm;
    float *hs = sm + RB * nu;
    const long long row0 = (long long)blockIdx.x * RB;
    for (int t = threadIdx.x; t < 2 * nu - 1; t += blockDim.x) hs[t] = h[t];
    for (int t = threadIdx.x; t < RB * nu; t += blockDim.x) {
        const int r = t / nu, jj = t - r * nu;
        const long long row = row0 + r;
        float val = 0.0f;
        if (row < n_rows) {
            const int view = (int)(row / F.n_v), iv = (int)(row - (long long)view * F.n_v);
            float pre;
            if (transpose) {
                pre = view_weight ? view_weight[view] : 1.0f;
            } else {
                pre = fdk_cosine(F, F.views[view], jj, iv);
                if (pixel_weight) pre *= pixel_weight[(long long)view * nu + jj];
            }
            val = x[row * nu + jj] * pre;
        }
        xs[t] = val;
    }
    __syncthreads();
    const int T = blockDim.x;
    for (int i0 = threadIdx.x; i0 < nu; i0 += 4 * T) {
        float acc[RB][4];
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int m = 0; m < 4; ++m) acc[r][m] = 0.0f;
        int hoff[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) hoff[m] = min(i0 + m * T, nu - 1) + nu - 1;
        // ODD: every even nonzero tap is zero (Ram-Lak).  A thread's outputs
        // i0 + m T share i0's parity (T is a multiple of 32), so only inputs of
        // the other parity meet nonzero taps; the centre tap is added last.
        for (int jj = ODD ? ((i0 & 1) ^ 1) : 0; jj < nu; jj += ODD ? 2 : 1) {
            float hv[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) hv[m] = hs[hoff[m] - jj];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float xv = xs[r * nu + jj];
#pragma unroll
                for (int m = 0; m < 4; ++m) acc[r][m] = __fmaf_rn(hv[m], xv, acc[r][m]);
            }
        }
        if (ODD) {
            const float h0 = hs[nu - 1];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int i = i0 + m * T;
                if (i >= nu) continue;
#pragma unroll
                for (int r = 0; r < RB; ++r) acc[r][m] = __fmaf_rn(h0, xs[r * nu + i], acc[r][m]);
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const long long row = row0 + r;
            if (row >= n_rows) continue;
            const int view = (int)(row / F.n_v), iv = (int)(row - (long long)view * F.n_v);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int i = i0 + m * T;
                if (i >= nu) continue;
                float post;
                if (transpose) {
                    post = fdk_cosine(F, F.views[view], i, iv);
                    if (pixel_weight) post *= pixel_weight[(long long)view * nu + i];
                } else {
                    post = view_weight ? view_weight[view] : 1.0f;
                }
                out[row * nu + i] = __fmul_rn(__fmul_rn(acc[r][m], F.pitch_u), post);
            }
        }
    }
}

// ----------------------------------------------------------------- host side
// Plan-time tables.  Returns 0, or 13 when the geometry is outside the class
// these kernels handle (3-D: a view's depth or u coordinate depends on z, i.e.
// the detector v axis is not +-z or its u axis not horizontal; a source not in
// front of the isocentre; affine forms beyond the fixed-point range).
inline int fdk_build(int ndim, int beam, int n_views, int n_u, int n_v, const float *src,
                     const float *det_centre, const float *det_u, const float *det_v,
                     double pitch_u, double pitch_v, double offset_u, double offset_v,
                     const int n[3], const double d[3], const double o[3],
                     std::vector<FdkView> &out, FdkParams &P)
{
    const double kPi = 3.14159265358979323846;
    out.assign(n_views > 0 ? n_views : 1, FdkView{});
    P.n_views = n_views;
    P.n_u = n_u;
    P.n_v = n_v;
    for (int a = 0; a < 3; ++a) P.n[a] = n[a];
    P.ndim = ndim;
    P.beam = beam;
    P.pitch_u = (float)pitch_u;
    P.pitch_v = (float)pitch_v;
    const double cu = 0.5 * (n_u - 1) - offset_u, cv = 0.5 * (n_v - 1) - offset_v;
    P.cu = (float)cu;
    P.cv = (float)cv;
    P.tx = kFdkTileX;
    const double iso[3] = {o[0] + 0.5 * n[0] * d[0], o[1] + 0.5 * n[1] * d[1],
                           o[2] + 0.5 * n[2] * d[2]};
    const double x0[3] = {o[0] + 0.5 * d[0], o[1] + 0.5 * d[1], o[2] + 0.5 * d[2]};
    auto dot = [](const double *p, const double *q) { return p[0] * q[0] + p[1] * q[1] + p[2] * q[2]; };
    auto cross = [](const double *p, const double *q, double *r) {
        r[0] = p[1] * q[2] - p[2] * q[1];
        r[1] = p[2] * q[0] - p[0] * q[2];
        r[2] = p[0] * q[1] - p[1] * q[0];
    };
    // fixed point with a range check: |value| * (largest index + 1) < 2^61
    bool ok = true;
    auto fix = [&](double value, int extent) -> long long {
        const double f = value * kFixOne;
        if (!std::isfinite(f) || std::fabs(f) * (double)(extent + 1) >= 2305843009213693952.0) {
            ok = false;
            return 0;
        }
        return (long long)std::llrint(f);
    };
    for (int s = 0; s < n_views; ++s) {
        double A[3], C[3], U[3], V[3], N[3], US[3], VS[3], cr[3];
        for (int q = 0; q < 3; ++q) {
            A[q] = src[3 * s + q];
            C[q] = det_centre[3 * s + q];
            U[q] = det_u[3 * s + q];
            V[q] = det_v[3 * s + q];
        }
        cross(U, V, N);
        const double nn = std::sqrt(dot(N, N));
        for (double &t : N) t /= nn;
        double side;
        if (beam == 1) {
            const double ca[3] = {C[0] - A[0], C[1] - A[1], C[2] - A[2]};
            side = dot(ca, N);
        } else {
            side = dot(A, N);
        }
        if (!(side != 0.0)) return 13;
        if (side < 0)
            for (double &t : N) t = -t;
        cross(U, V, cr);
        const double triple = dot(cr, N);
        cross(V, N, US);
        cross(N, U, VS);
        for (int q = 0; q < 3; ++q) {
            US[q] /= triple;
            VS[q] /= triple;
        }
        FdkView &F = out[s];
        // depth / SID, u and v numerators as affine forms of the voxel centre
        double e0, ex[3], u0, ux[3], v0, vx[3], scale;
        if (beam == 1) {
            const double ca[3] = {C[0] - A[0], C[1] - A[1], C[2] - A[2]};
            const double ia[3] = {iso[0] - A[0], iso[1] - A[1], iso[2] - A[2]};
            const double xa[3] = {x0[0] - A[0], x0[1] - A[1], x0[2] - A[2]};
            const double sdd = dot(ca, N), sid = dot(ia, N);
            if (!(sdd > 0.0) || !(sid > 0.0)) return 13;
            e0 = dot(xa, N) / sid;
            for (int q = 0; q < 3; ++q) ex[q] = d[q] * N[q] / sid;
            const double au = cu - dot(ca, US) / pitch_u, bu = sdd / (pitch_u * sid);
            const double av = cv - dot(ca, VS) / pitch_v, bv = sdd / (pitch_v * sid);
            u0 = au * e0 + bu * dot(xa, US);
            v0 = av * e0 + bv * dot(xa, VS);
            for (int q = 0; q < 3; ++q) {
                ux[q] = au * ex[q] + bu * d[q] * US[q];
                vx[q] = av * ex[q] + bv * d[q] * VS[q];
            }
            scale = sdd / (2.0 * kPi * sid);
            F.sdd = (float)sdd;
            F.g[0] = (float)dot(ca, ca);
            F.g[1] = (float)dot(ca, U);
            F.g[2] = (float)dot(ca, V);
        } else {
            const double an = std::sqrt(dot(A, A));
            const double R[3] = {A[0] / an, A[1] / an, A[2] / an};
            const double rn = dot(R, N);
            double WU[3], WV[3];
            for (int q = 0; q < 3; ++q) {
                WU[q] = US[q] - N[q] * dot(R, US) / rn;
                WV[q] = VS[q] - N[q] * dot(R, VS) / rn;
            }
            const double xc[3] = {x0[0] - C[0], x0[1] - C[1], x0[2] - C[2]};
            e0 = 1.0;
            ex[0] = ex[1] = ex[2] = 0.0;
            u0 = cu + dot(xc, WU) / pitch_u;
            v0 = cv + dot(xc, WV) / pitch_v;
            for (int q = 0; q < 3; ++q) {
                ux[q] = d[q] * WU[q] / pitch_u;
                vx[q] = d[q] * WV[q] / pitch_v;
            }
            scale = 1.0 / (2.0 * kPi);
            F.sdd = 1.0f;
            F.g[0] = F.g[1] = F.g[2] = 0.0f;
        }
        F.g[3] = (float)dot(U, V);
        F.g[4] = (float)dot(U, U);
        F.g[5] = (float)dot(V, V);
        F.scale = (float)scale;
        if (ndim == 3) {
            // the column walk needs depth and u independent of z
            const double tol = 1e-12 * (std::fabs(e0) + std::fabs(u0) + 1.0);
            if (std::fabs(ex[2]) > tol || std::fabs(ux[2]) > tol) return 13;
        } else {
            // 2-D: one slice at k = 0; v is not used
            v0 = 0.0;
            vx[0] = vx[1] = vx[2] = 0.0;
        }
        F.e[0] = fix(e0, 0);
        F.e[1] = fix(ex[0], n[0]);
        F.e[2] = fix(ex[1], n[1]);
        F.nu[0] = fix(u0, 0);
        F.nu[1] = fix(ux[0], n[0]);
        F.nu[2] = fix(ux[1], n[1]);
        F.nv[0] = fix(v0, 0);
        F.nv[1] = fix(vx[0], n[0]);
        F.nv[2] = fix(vx[1], n[1]);
        F.nv[3] = fix(vx[2], n[2]);
        // the sum of the terms must stay in range as well
        const double umax = std::fabs(u0) + std::fabs(ux[0]) * n[0] + std::fabs(ux[1]) * n[1];
        const double vmax = std::fabs(v0) + std::fabs(vx[0]) * n[0] + std::fabs(vx[1]) * n[1] +
                            std::fabs(vx[2]) * n[2];
        const double emax = std::fabs(e0) + std::fabs(ex[0]) * n[0] + std::fabs(ex[1]) * n[1];
        fix(umax, 1);
        fix(vmax, 1);
        fix(emax, 1);
        if (!ok) return 13;
    }
    return 0;
}

// Ramp kernels h[m], m = -(n-1) .. n-1: the inverse transforms of H(omega) =
// |omega| (radians per unit length) times a window, for |omega| <= pi / tau:
// none (Ram-Lak), (2/(tau |omega|)) |sin(omega tau / 2)| (Shepp-Logan),
// cos(omega tau / 2) (cosine), 0.54 + 0.46 cos(omega tau) (Hamming) and
// (1 + cos(omega tau)) / 2 (Hann).  The cosine windows shift the band-limited
// ramp r(x) = (pi sin(pi x) / x + (cos(pi x) - 1) / x^2) / (pi tau^2) by half or
// whole samples.
constexpr int kRampKinds = 5;

inline double fdk_band_ramp(double x, double tau)
{
    const double kPi = 3.14159265358979323846;
    if (x == 0.0) return kPi / (2.0 * tau * tau);
    const long long m = (long long)x;
    if ((double)m == x)  // whole samples: 0 (even) or -2 / (pi m^2 tau^2) (odd)
        return (m % 2 == 0) ? 0.0 : -2.0 / (kPi * x * x * tau * tau);
    return (kPi * std::sin(kPi * x) / x + (std::cos(kPi * x) - 1.0) / (x * x)) / (kPi * tau * tau);
}

inline void fdk_ramp_kernel(int n, double tau, int kind, std::vector<float> &h)
{
    const double kPi = 3.14159265358979323846;
    h.assign(2 * n - 1, 0.0f);
    for (int t = 0; t < 2 * n - 1; ++t) {
        const double m = (double)(t - (n - 1));
        double v;
        switch (kind) {
        // the band-limited ramp is exactly zero at even nonzero offsets (sin and
        // cos - 1 of an even multiple of pi); its float64 evaluation leaves
        // ~1e-17 there, so those samples are set to zero directly
        case 0: v = (t - (n - 1)) % 2 == 0 && t != n - 1 ? 0.0 : fdk_band_ramp(m, tau); break;
        case 1: v = -4.0 / (kPi * tau * tau * (4.0 * m * m - 1.0)); break;
        case 2: v = 0.5 * (fdk_band_ramp(m - 0.5, tau) + fdk_band_ramp(m + 0.5, tau)); break;
        case 3:
            v = 0.54 * fdk_band_ramp(m, tau) +
                0.23 * (fdk_band_ramp(m - 1.0, tau) + fdk_band_ramp(m + 1.0, tau));
            break;
        default:
            v = 0.5 * fdk_band_ramp(m, tau) +
                0.25 * (fdk_band_ramp(m - 1.0, tau) + fdk_band_ramp(m + 1.0, tau));
            break;
        }
        h[t] = (float)v;
    }
}

inline dim3 fdk_grid(const FdkParams &F, int K)
{
    const int kz = F.ndim == 2 ? 1 : (F.n[2] + K - 1) / K;
    return dim3((F.n[0] + 31) / 32, (F.n[1] + 7) / 8, kz);
}

// z voxels per thread of the scatter: more steps merge more taps per detector
// row in registers before the reductions (K = 16 / 24 / 32: C3 11.5 / 11.6 /
// 14.4, C4 288 / 281 / 281, C5 58.6 / 54.8 / 65.2 ms on a phantom volume)
constexpr int kFdkK = 24;

// z voxels per thread of the gather: the per-(column, view) set-up is shared by
// K voxels, at the cost of registers.  With the view loop unrolled by two at 4
// blocks per SM, K = 12 / 16 / 20 / 24 measured C3 9.01 / 8.18 / 8.60 / 9.16,
// C4 106.5 / 97.2 / 95.3 / 101.6, C5 67.8 / 57.3 / 53.0 / 51.4 ms (16 had been
// faster than 8, 32 and 64 without the unroll).
constexpr int kFdkGatherK = 20;

inline int fdk_gather(const FdkParams &F, const float *q, float *vol, cudaStream_t s)
{
    if (F.ndim == 2) {
        wbp_gather_kernel<1><<<fdk_grid(F, 1), 256, 0, s>>>(F, q, vol);
    } else {
        wbp_gather_kernel<kFdkGatherK><<<fdk_grid(F, kFdkGatherK), 256, 0, s>>>(F, q, vol);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int fdk_scatter(const FdkParams &F, const float *vol, float *q, cudaStream_t s)
{
    const size_t bytes = sizeof(float) * (size_t)F.n_views * F.n_u * F.n_v;
    if (cudaMemsetAsync(q, 0, bytes, s) != cudaSuccess) return 9;
    if (F.n_views == 0) return 0;
    if (F.ndim == 2) wbp_scatter_kernel<1><<<fdk_grid(F, 1), 256, 0, s>>>(F, vol, q);
    else wbp_scatter_kernel<kFdkK><<<fdk_grid(F, kFdkK), 256, 0, s>>>(F, vol, q);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

// Largest detector row this filter takes (shared memory: one row and the kernel).
constexpr int kFilterMaxU = 16384;

template <int RB, bool ODD>
inline int ramp_launch(const FdkParams &F, const float *h, const float *x, float *out,
                       const float *view_weight, const float *pixel_weight, int transpose,
                       cudaStream_t s)
{
    const long long rows = (long long)F.n_views * F.n_v;
    const size_t smem = sizeof(float) * ((size_t)RB * F.n_u + 2 * (size_t)F.n_u);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(ramp_filter_kernel<RB, ODD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 9;
    int threads = (F.n_u + 3) / 4;
    threads = ((threads + 31) / 32) * 32;
    threads = threads < 32 ? 32 : (threads > 256 ? 256 : threads);
    const long long blocks = (rows + RB - 1) / RB;
    ramp_filter_kernel<RB, ODD><<<(unsigned)blocks, threads, smem, s>>>(
        F, h, x, out, view_weight, pixel_weight, transpose, rows);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

template <bool ODD>
inline int fdk_filter_rows(const FdkParams &F, const float *h, const float *x, float *out,
                           const float *vw, const float *pw, int transpose, cudaStream_t s)
{
    // rows per block: as many as fit 48 KB of shared memory, at most 8
    const size_t per_row = sizeof(float) * (size_t)F.n_u;
    const size_t hbytes = 2 * per_row;
    if (hbytes + 8 * per_row <= 48 * 1024) return ramp_launch<8, ODD>(F, h, x, out, vw, pw, transpose, s);
    if (hbytes + 4 * per_row <= 48 * 1024) return ramp_launch<4, ODD>(F, h, x, out, vw, pw, transpose, s);
    if (hbytes + 2 * per_row <= 48 * 1024) return ramp_launch<2, ODD>(F, h, x, out, vw, pw, transpose, s);
    return ramp_launch<1, ODD>(F, h, x, out, vw, pw, transpose, s);
}

// odd: every even nonzero tap of h is zero (ramp_taps_odd), so the filter skips
// them (C4 Ram-Lak filter about half the time).
inline int fdk_filter(const FdkParams &F, const float *h, bool odd, const float *x, float *out,
                      const float *view_weight, const float *pixel_weight, int transpose,
                      cudaStream_t s)
{
    if ((long long)F.n_views * F.n_v == 0) return 0;
    return odd ? fdk_filter_rows<true>(F, h, x, out, view_weight, pixel_weight, transpose, s)
               : fdk_filter_rows<false>(F, h, x, out, view_weight, pixel_weight, transpose, s);
}

// True when every tap of h (2 n - 1 taps, centre n - 1) at an even nonzero
// offset is exactly zero.
inline bool ramp_taps_odd(const std::vector<float> &h, int n)
{
    for (int t = 0; t < 2 * n - 1; ++t)
        if ((t - (n - 1)) % 2 == 0 && t != n - 1 && h[t] != 0.0f) return false;
    return true;
}

// Parker's short-scan weights (Parker 1982) of a circular divergent scan about
// the vertical axis through the volume centre: per view the scan angle beta
// (source azimuth from view 0, in the turning sense), per view and column the
// signed fan angle gamma in the xy plane (central ray to the column's ray, in
// the turning sense), Gamma the largest |gamma| of view 0;
//   w = sin^2(pi/4 beta / (Gamma - gamma))              for beta < 2 (Gamma - gamma)
//     = sin^2(pi/4 (pi + 2 Gamma - beta) / (Gamma + gamma))  for beta > pi - 2 gamma
//     = 1 between, 0 outside [0, pi + 2 Gamma],
// so that the weights of a ray and its conjugate (beta + pi + 2 gamma, -gamma)
// sum to one.  Host float64 (n_views x n_u values, set-up work).
inline void fdk_parker(int n_views, int n_u, const float *src, const float *centre,
                       const float *det_u, double pitch_u, double offset_u, const double iso[2],
                       std::vector<float> &out)
{
    const double kPi = 3.14159265358979323846;
    out.assign((size_t)n_views * n_u, 0.0f);
    if (n_views == 0) return;
    std::vector<double> az(n_views), gam((size_t)n_views * n_u);
    for (int k = 0; k < n_views; ++k) {
        az[k] = std::atan2((double)src[3 * k + 1] - iso[1], (double)src[3 * k] - iso[0]);
        if (k > 0) {  // unwrap
            while (az[k] - az[k - 1] > kPi) az[k] -= 2 * kPi;
            while (az[k] - az[k - 1] < -kPi) az[k] += 2 * kPi;
        }
    }
    const double sense = (n_views < 2 || az[1] >= az[0]) ? 1.0 : -1.0;
    double big = 0.0;
    for (int k = 0; k < n_views; ++k) {
        const double ax = src[3 * k], ay = src[3 * k + 1];
        const double rx = ax - iso[0], ry = ay - iso[1], rn = std::sqrt(rx * rx + ry * ry);
        const double cx = -rx / rn, cy = -ry / rn;  // central ray direction
        for (int i = 0; i < n_u; ++i) {
            const double off = ((double)i - 0.5 * (n_u - 1) + offset_u) * pitch_u;
            const double dx = centre[3 * k] + off * det_u[3 * k] - ax;
            const double dy = centre[3 * k + 1] + off * det_u[3 * k + 1] - ay;
            const double g = sense * std::atan2(cx * dy - cy * dx, cx * dx + cy * dy);
            gam[(size_t)k * n_u + i] = g;
            if (k == 0) big = std::fmax(big, std::fabs(g));
        }
    }
    for (int k = 0; k < n_views; ++k) {
        const double beta = sense * (az[k] - az[0]);
        for (int i = 0; i < n_u; ++i) {
            const double g = gam[(size_t)k * n_u + i];
            double w = 1.0;
            if (beta < 0.0 || beta > kPi + 2 * big) {
                w = 0.0;
            } else if (beta < 2 * (big - g)) {
                const double t = std::sin(0.25 * kPi * beta / (big - g));
                w = t * t;
            } else if (beta > kPi - 2 * g) {
                const double t = std::sin(0.25 * kPi * (kPi + 2 * big - beta) / (big + g));
                w = t * t;
            }
            out[(size_t)k * n_u + i] = (float)w;
        }
    }
}

}  // namespace ctp
