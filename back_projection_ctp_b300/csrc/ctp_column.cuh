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
    double zc, zd;       // z (cells) at slab k0 of row iv: zc + iv * zd
    double bc, bd;       // z slope per slab of row iv: bc + iv * bd (signed)
};

struct ColumnPlan {
    int n_columns;       // n_views * n_u
};

// Zero halo (cells) around x and y of the padded working copies: the walk's
// widened slab range reaches at most this far outside the grid, so the forward
// reads zeros there and the backward's stray pieces land in cells that are
// never copied out -- no xy bounds tests in the walk.
constexpr int kHalo = 2;

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
    C.zc = C.zd = C.bc = C.bd = 0.0;

    double P0[3];
#pragma unroll
    for (int a = 0; a < 3; ++a) P0[a] = __fma_rn((double)iu, V.du[a], V.p00[a]);
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
    if (P.beam == 1) {
        const double wz0 = __dsub_rn(P0[2], V.a[2]);
        C.zc = __fma_rn(lam, wz0, V.a[2]);
        C.zd = __dmul_rn(lam, V.dv[2]);
        C.bc = __dmul_rn(wz0, inv);
        C.bd = __dmul_rn(V.dv[2], inv);
    } else {
        C.zc = __fma_rn(lam, V.a[2], P0[2]);
        C.zd = V.dv[2];
        C.bc = __dmul_rn(V.a[2], inv);
        C.bd = 0.0;
    }
    // every row must cross at most one z plane per slab
    const double s0 = fabs(C.bc), s1 = fabs(__fma_rn((double)(P.n_v - 1), C.bd, C.bc));
    if (!(fmax(s0, s1) < 1.0)) atomicOr(flag, 2);
    T[col] = C;
}

// Per-lane z state: the row's own transverse axis of the slab walk.
struct LaneZ {
    uint32_t fz, bz;     // z fraction at slab k0 and slope (2^-32 cell units), mirrored
    float ibz;           // 1 / bz
    int jz;              // mirrored z index at slab k0
    int sz;              // +-1: z stride in the padded z-fastest copy
    int addr;            // padded offset of cell (k0, jb, jz)
    float ell;           // physical length per slab
};

// Lane set-up: the column's xy state plus this row's z line (float64: about
// ten operations per lane; the shared xy part was built at plan time).
__device__ __forceinline__ LaneZ column_lane_setup(const RayParams &P, const ColumnTrace &C,
                                                   int iv)
{
    LaneZ L;
    const double z = __fma_rn((double)iv, C.zd, C.zc);
    const double bz = __fma_rn((double)iv, C.bd, C.bc);
    const bool m = bz < 0.0;
    const double zm = m ? __dsub_rn((double)P.n[2], z) : z;
    const double abz = fabs(bz);
    // rows far outside the grid in z touch no cell; bound their index so the
    // walk's integer address arithmetic stays small
    const double zcl = fmin(fmax(zm, -65536.0), (double)P.n[2] + 65536.0);
    const double fjz = floor(zcl);
    L.jz = (int)fjz;
    L.fz = (uint32_t)__dmul_rn(__dsub_rn(zcl, fjz), 4294967296.0);
    L.bz = to_fixed_slope(abz);
    L.ibz = L.bz ? __frcp_rn((float)L.bz) : 0.0f;
    L.sz = m ? -1 : 1;
    L.addr = C.addr_xy + (m ? (P.n[2] - 1) : 0) + L.sz * L.jz;
    const float dz = (float)(abz * P.spacing[2]);
    L.ell = __fsqrt_rn(__fadd_rn(C.lxy2, __fmul_rn(dz, dz)));
    return L;
}

// One slab of the column walk.  The b (xy) crossing is the same for every lane
// of a warp (one column per warp), so the branch on it does not diverge; the
// common slab without it holds one or two pieces, split only by the lane's own
// z crossing.  A crossing's slab fraction comes from the wrapped sum g of the
// fixed-point add: t = (beta - g) / beta = 1 - g / beta.  CLAMP restricts the
// slab to [lo, hi] (first / last slab of a ray that starts or ends inside).
// op(addr, length, on, jb) sees every piece; `on` = the piece lies inside the
// grid in z (x and y are covered by the halo); jb lets the counter test x / y.
template <bool CLAMP, class Op>
__device__ __forceinline__ void column_slab(uint32_t &fb, uint32_t bb, float ib, int &jb, int sb,
                                            uint32_t &fz, uint32_t bz, float ibz, int &jz,
                                            int sz, unsigned nz, int &addr, int sp, float lo,
                                            float hi, Op &op)
{
    const uint32_t gz = fz + bz;
    const bool cz = gz < fz;
    const float tz = cz ? fmaxf(__fmaf_rn(-__uint2float_rn(gz), ibz, 1.0f), 0.0f) : 1.0f;
    const bool v0 = (unsigned)jz < nz;
    const bool v1 = (unsigned)(jz + 1) < nz;
    const uint32_t gb = fb + bb;
    const bool cb = gb < fb;
    if (!cb) {
        float e = tz;
        if (CLAMP) e = fminf(fmaxf(e, lo), hi);
        const float d0 = CLAMP ? __fsub_rn(e, lo) : e;
        const float d1 = __fsub_rn(CLAMP ? hi : 1.0f, e);
        op(addr, d0, v0, jb);
        op(addr + sz, d1, cz && v1, jb);
        addr += sp + (cz ? sz : 0);
    } else {
        const float tb = fmaxf(__fmaf_rn(-__uint2float_rn(gb), ib, 1.0f), 0.0f);
        const bool bfirst = tb < tz;
        float e1 = fminf(tb, tz), e2 = fmaxf(tb, tz);
        if (CLAMP) {
            e1 = fminf(fmaxf(e1, lo), hi);
            e2 = fminf(fmaxf(e2, lo), hi);
        }
        const float d1 = CLAMP ? __fsub_rn(e1, lo) : e1;
        const float d2 = __fsub_rn(e2, e1);
        const float d3 = __fsub_rn(CLAMP ? hi : 1.0f, e2);
        const int a3 = addr + sb + (cz ? sz : 0);
        op(addr, d1, v0, jb);
        op(addr + (bfirst ? sb : sz), d2, bfirst ? v0 : v1, bfirst ? jb + 1 : jb);
        op(a3, d3, cz && v1, jb + 1);
        addr = a3 + sp;
        jb += 1;
    }
    fz = gz;
    jz += cz ? 1 : 0;
    fb = gb;
}

// Walk all slabs of one lane: partial first / last slab peeled off, the main
// loop without clamps.
template <class Op>
__device__ __forceinline__ void column_walk(const ColumnTrace &C, const LaneZ &L, unsigned nz,
                                            Op &op)
{
    uint32_t fb = C.fb, fz = L.fz;
    int jb = C.jb, jz = L.jz, addr = L.addr;
    const uint32_t bb = C.bb, bz = L.bz;
    const float ib = C.ib, ibz = L.ibz;
    const int sb = C.sb, sp = C.sp, sz = L.sz;
    column_slab<true>(fb, bb, ib, jb, sb, fz, bz, ibz, jz, sz, nz, addr, sp, C.tlo,
                      C.k0 == C.k1 ? C.thi : 1.0f, op);
    for (int k = C.k0 + 1; k < C.k1; ++k)
        column_slab<false>(fb, bb, ib, jb, sb, fz, bz, ibz, jz, sz, nz, addr, sp, 0.0f, 1.0f, op);
    if (C.k1 > C.k0)
        column_slab<true>(fb, bb, ib, jb, sb, fz, bz, ibz, jz, sz, nz, addr, sp, 0.0f, C.thi, op);
}

struct ColumnGather {
    const float *__restrict__ vol;
    float acc;
    __device__ __forceinline__ void operator()(int a, float d, bool on, int)
    {
        if (on) acc = __fmaf_rn(d, __ldg(vol + a), acc);
    }
};

struct ColumnScatter {
    float *__restrict__ vol;
    float w;  // ell * y
    __device__ __forceinline__ void operator()(int a, float d, bool on, int)
    {
        if (on && d > 0.0f) atomicAdd(vol + a, __fmul_rn(d, w));
    }
};

struct ColumnCount {
    unsigned n;
    float thr;
    unsigned nb;
    __device__ __forceinline__ void operator()(int, float d, bool on, int jb)
    {
        n += (on && (unsigned)jb < nb && d > thr) ? 1u : 0u;
    }
};

constexpr int kColumnsPerBlock = 8;  // 8 warps: 8 columns x 32 rows

__global__ void __launch_bounds__(256) column_forward_kernel(RayParams P,
                                                             const ColumnTrace *__restrict__ T,
                                                             const float *__restrict__ zvol,
                                                             float *__restrict__ sino)
{
    __shared__ float tile[32][kColumnsPerBlock + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int iu = blockIdx.x * kColumnsPerBlock + warp;
    const int view = blockIdx.y;
    const int iv = blockIdx.z * 32 + lane;
    float out = 0.0f;
    if (iu < P.n_u && iv < P.n_v) {
        const ColumnTrace C = T[(long long)view * P.n_u + iu];
        if (C.k0 <= C.k1) {
            const LaneZ L = column_lane_setup(P, C, iv);
            ColumnGather op{zvol, 0.0f};
            column_walk(C, L, (unsigned)P.n[2], op);
            out = __fmul_rn(op.acc, L.ell);
        }
    }
    tile[lane][warp] = out;
    __syncthreads();
    const int r = threadIdx.x / kColumnsPerBlock, c = threadIdx.x % kColumnsPerBlock;
    const int ivw = blockIdx.z * 32 + r, iuw = blockIdx.x * kColumnsPerBlock + c;
    if (ivw < P.n_v && iuw < P.n_u)
        sino[((long long)view * P.n_v + ivw) * P.n_u + iuw] = tile[r][c];
}

__global__ void __launch_bounds__(256) column_backward_kernel(RayParams P,
                                                              const ColumnTrace *__restrict__ T,
                                                              const float *__restrict__ sino,
                                                              float *__restrict__ zvol)
{
    __shared__ float tile[32][kColumnsPerBlock + 1];
    const int view = blockIdx.y;
    {
        const int r = threadIdx.x / kColumnsPerBlock, c = threadIdx.x % kColumnsPerBlock;
        const int ivr = blockIdx.z * 32 + r, iur = blockIdx.x * kColumnsPerBlock + c;
        tile[r][c] = (ivr < P.n_v && iur < P.n_u)
                         ? sino[((long long)view * P.n_v + ivr) * P.n_u + iur]
                         : 0.0f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int iu = blockIdx.x * kColumnsPerBlock + warp;
    const int iv = blockIdx.z * 32 + lane;
    const float y = tile[lane][warp];
    if (iu >= P.n_u || iv >= P.n_v || y == 0.0f) return;
    const ColumnTrace C = T[(long long)view * P.n_u + iu];
    if (C.k0 > C.k1) return;
    const LaneZ L = column_lane_setup(P, C, iv);
    ColumnScatter op{zvol, __fmul_rn(L.ell, y)};
    column_walk(C, L, (unsigned)P.n[2], op);
}

__global__ void __launch_bounds__(256) column_count_kernel(RayParams P,
                                                           const ColumnTrace *__restrict__ T,
                                                           unsigned long long *__restrict__ total)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int iu = blockIdx.x * kColumnsPerBlock + warp;
    const int view = blockIdx.y;
    const int iv = blockIdx.z * 32 + lane;
    unsigned n = 0;
    if (iu < P.n_u && iv < P.n_v) {
        const ColumnTrace C = T[(long long)view * P.n_u + iu];
        if (C.k0 <= C.k1) {
            const LaneZ L = column_lane_setup(P, C, iv);
            ColumnCount op{0u, __fdiv_rn(P.min_len, L.ell), (unsigned)C.nb};
            column_walk(C, L, (unsigned)P.n[2], op);
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
        if (x < nx && z < nz) out[((x + kHalo) * pny + (y + kHalo)) * nz + z] = tile[tx][j];
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
        if (x < nx && z < nz) tile[j][tx] = in[((x + kHalo) * pny + (y + kHalo)) * nz + z];
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int z = z0 + j, x = x0 + tx;
        if (z < nz && x < nx) out[((size_t)z * ny + y) * nx + x] = tile[tx][j];
    }
}

inline size_t column_padded_cells(const RayParams &P)
{
    return ((size_t)P.n[0] + 2 * kHalo) * ((size_t)P.n[1] + 2 * kHalo) * (size_t)P.n[2];
}

// Builds the column table and the two padded working copies (forward: halo
// zeroed once here and never written again; backward: zeroed per call).
// Returns 0, 9 (CUDA error) or 11 (scan not eligible for the column path).
inline int column_plan_build(const RayParams &P, ColumnPlan *plan, void **d_columns,
                             float **d_zfwd, float **d_zbwd, unsigned long long *bytes)
{
    if ((long long)P.n_views * P.n_u >= (1LL << 31)) return 11;
    if (column_padded_cells(P) >= (1ULL << 31)) return 11;
    plan->n_columns = P.n_views * P.n_u;
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

inline dim3 column_grid(const RayParams &P)
{
    return dim3((P.n_u + kColumnsPerBlock - 1) / kColumnsPerBlock, P.n_views, (P.n_v + 31) / 32);
}

inline dim3 transpose_grid(const RayParams &P)
{
    return dim3((P.n[0] + 31) / 32, (P.n[2] + 31) / 32, P.n[1]);
}

inline int column_forward(const RayParams &P, const ColumnPlan &, const void *d_columns,
                          float *d_zfwd, const float *vol, float *sino, cudaStream_t s)
{
    xfast_to_zfast_kernel<<<transpose_grid(P), 256, 0, s>>>(vol, d_zfwd, P.n[0], P.n[1], P.n[2]);
    column_forward_kernel<<<column_grid(P), 256, 0, s>>>(P, (const ColumnTrace *)d_columns, d_zfwd,
                                                        sino);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int column_backward(const RayParams &P, const ColumnPlan &, const void *d_columns,
                           float *d_zbwd, const float *sino, float *vol, cudaStream_t s)
{
    if (cudaMemsetAsync(d_zbwd, 0, sizeof(float) * column_padded_cells(P), s) != cudaSuccess)
        return 9;
    if ((long long)P.n_views * P.n_u * P.n_v > 0)
        column_backward_kernel<<<column_grid(P), 256, 0, s>>>(P, (const ColumnTrace *)d_columns,
                                                             sino, d_zbwd);
    zfast_to_xfast_kernel<<<transpose_grid(P), 256, 0, s>>>(d_zbwd, vol, P.n[0], P.n[1], P.n[2]);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int column_count(const RayParams &P, const ColumnPlan &, const void *d_columns,
                        unsigned long long *d_total, cudaStream_t s)
{
    column_count_kernel<<<column_grid(P), 256, 0, s>>>(P, (const ColumnTrace *)d_columns, d_total);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

}  // namespace ctp
