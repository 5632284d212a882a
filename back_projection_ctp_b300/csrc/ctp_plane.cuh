// Plane path: 2-D scans (one slice, rays in the slice plane).
//
// A 2-D ray has one transverse axis: within a unit slab of its dominant axis it
// holds one or two pieces.  Each ray's walk state (the same fixed-point slab
// parametrisation as the 3-D paths) is built once per plan in float64 and stored;
// a call only walks.  The image is walked in two zero-halo padded copies, one
// x-fastest and one y-fastest: a ray whose transverse axis is x reads the first,
// one whose transverse axis is y the second, so the 32 adjacent rays of a warp,
// stepping the same slab, touch consecutive floats.  The halo (2 cells) covers
// the walk's reach outside the grid, so the walk has no bounds tests; the
// backward accumulates into both padded copies and adds them in one pass.
#pragma once

#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>

#include "ctp_internal.h"
#include "ctp_ray.cuh"

namespace ctp {

constexpr int kPlaneHalo = 2;

// 64 bytes; the walks read only the first 48 (plane_ray_walk_state).
struct __align__(16) PlaneRay {
    int k0, k1;          // slab range (k1 < k0: the ray misses)
    float tlo, thi;      // partial first / last slab fractions (ray ends)
    uint32_t fb, bb;     // transverse fraction at slab k0 and slope (2^-32 cell)
    float ib;            // 1 / bb
    int addr;            // offset of cell (k0, jb) in the combined padded buffer
    int sp, sb;          // signed strides along the slab axis and the transverse axis
    int jb;              // transverse (mirrored) index at slab k0
    float ell;           // physical length per slab
    int nb;              // transverse extent
    int pad_[3];         // pad_[0]: the slab axis (0 = x, 1 = y)
};

static_assert(sizeof(PlaneRay) == 64 && offsetof(PlaneRay, ell) == 44,
              "the walk state is the first three 16-byte words");

// The walk state of a ray (every field but nb and pad_) in three 16-byte
// loads: a warp reading 32 adjacent records field by field would touch 32
// sectors per field, for 11 fields.
__device__ __forceinline__ PlaneRay plane_ray_walk_state(const PlaneRay *__restrict__ T,
                                                         long long ray)
{
    const int4 *q = reinterpret_cast<const int4 *>(T + ray);
    const int4 a = __ldg(q), b = __ldg(q + 1), c = __ldg(q + 2);
    PlaneRay R;
    R.k0 = a.x;
    R.k1 = a.y;
    R.tlo = __int_as_float(a.z);
    R.thi = __int_as_float(a.w);
    R.fb = (uint32_t)b.x;
    R.bb = (uint32_t)b.y;
    R.ib = __int_as_float(b.z);
    R.addr = b.w;
    R.sp = c.x;
    R.sb = c.y;
    R.jb = c.z;
    R.ell = __int_as_float(c.w);
    R.nb = 0;
    R.pad_[0] = R.pad_[1] = R.pad_[2] = 0;
    return R;
}

// The whole record (four 16-byte loads).
__device__ __forceinline__ PlaneRay plane_ray_record(const PlaneRay *__restrict__ T, long long ray)
{
    PlaneRay R = plane_ray_walk_state(T, ray);
    const int4 d = __ldg(reinterpret_cast<const int4 *>(T + ray) + 3);
    R.nb = d.x;
    R.pad_[0] = d.y;
    R.pad_[1] = d.z;
    R.pad_[2] = d.w;
    return R;
}

struct PlaneLayout {
    int nx, ny;
    int px, py;          // padded extents
    int off1;            // offset of the y-fastest copy in the combined buffer
};

inline PlaneLayout plane_layout(const RayParams &P)
{
    PlaneLayout L;
    L.nx = P.n[0];
    L.ny = P.n[1];
    L.px = P.n[0] + 2 * kPlaneHalo;
    L.py = P.n[1] + 2 * kPlaneHalo;
    L.off1 = L.px * L.py;
    return L;
}

// Float64 set-up of every ray (plan time).  flag |= 1 when a ray leaves the
// slice plane (then the scan is not a plane-path scan).
__global__ void plane_setup_kernel(RayParams P, PlaneLayout G, PlaneRay *__restrict__ T,
                                   int *__restrict__ flag)
{
    const long long ray = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (ray >= (long long)P.n_views * P.n_u) return;
    const int view = (int)(ray / P.n_u), iu = (int)(ray % P.n_u);
    const ViewFrame &V = P.views[view];
    PlaneRay R;
    R.k0 = 0;
    R.k1 = -1;
    R.tlo = 0.0f;
    R.thi = 1.0f;
    R.fb = R.bb = 0;
    R.ib = 0.0f;
    R.addr = 0;
    R.sp = R.sb = 0;
    R.jb = 0;
    R.nb = 1;
    R.ell = 0.0f;
    R.pad_[0] = R.pad_[1] = R.pad_[2] = 0;

    double pix[3], X0[3], w[3];
    for (int a = 0; a < 3; ++a) pix[a] = __fma_rn((double)iu, V.du[a], V.p00[a]);
    for (int a = 0; a < 3; ++a) {
        if (P.beam == 1) {
            X0[a] = V.a[a];
            w[a] = __dsub_rn(pix[a], V.a[a]);
        } else {
            X0[a] = pix[a];
            w[a] = V.a[a];
        }
    }
    if (w[2] != 0.0) {  // the ray leaves the slice plane
        atomicOr(flag, 1);
        T[ray] = R;
        return;
    }
    // inside the single z cell?  (half-open, as everywhere)
    if (!(X0[2] >= 0.0 && X0[2] < 1.0)) {
        T[ray] = R;
        return;
    }
    const double awx = fabs(w[0]), awy = fabs(w[1]);
    const int p = awx >= awy ? 0 : 1, b = 1 - p;
    const double awp = p == 0 ? awx : awy, awb = p == 0 ? awy : awx;
    if (!(awp > 0.0)) {
        T[ray] = R;
        return;
    }
    double A[2];
    for (int a = 0; a < 2; ++a) A[a] = w[a] < 0.0 ? __dsub_rn((double)P.n[a], X0[a]) : X0[a];
    const double inv = __ddiv_rn(1.0, awp);
    const double beta = __dmul_rn(awb, inv);
    const double alpha = __fma_rn(-A[p], beta, A[b]);
    double lo = 0.0, hi = (double)P.n[p];
    double lo_t = -1.0e300, hi_t = 1.0e300;
    if (P.beam == 1) {
        lo_t = A[p];
        hi_t = __dadd_rn(A[p], awp);
        lo = fmax(lo, lo_t);
        hi = fmin(hi, hi_t);
    }
    const double nb = (double)P.n[b];
    if (beta > 0.0) {
        const double r = __ddiv_rn(awp, awb);
        lo = fmax(lo, __dmul_rn(-alpha, r));
        hi = fmin(hi, __dmul_rn(__dsub_rn(nb, alpha), r));
    } else if (!(alpha >= 0.0 && alpha < nb)) {
        T[ray] = R;
        return;
    }
    if (!(lo < hi)) {
        T[ray] = R;
        return;
    }
    // Slabs holding part of [lo, hi); the transverse index then stays within
    // [-2, n_b + 1], inside the zero halo.
    const double k0 = fmax(floor(lo), 0.0);
    const double k1 = fmin(ceil(hi) - 1.0, (double)(P.n[p] - 1));
    if (k0 > k1) {
        T[ray] = R;
        return;
    }
    R.k0 = (int)k0;
    R.k1 = (int)k1;
    R.tlo = (float)fmin(fmax(__dsub_rn(lo_t, k0), 0.0), 1.0);
    R.thi = (float)fmin(fmax(__dsub_rn(hi_t, k1), 0.0), 1.0);
    const double xb = __fma_rn(k0, beta, alpha);
    const double fjb = floor(xb);
    R.jb = (int)fjb;
    R.fb = (uint32_t)__dmul_rn(__dsub_rn(xb, fjb), 4294967296.0);
    R.bb = to_fixed_slope(beta);
    R.ib = R.bb ? __frcp_rn((float)R.bb) : 0.0f;
    R.nb = P.n[b];
    const float sp = (float)P.spacing[p], db = (float)(P.spacing[b] * beta);
    R.ell = __fsqrt_rn(__fadd_rn(__fmul_rn(sp, sp), __fmul_rn(db, db)));
    // layout: transverse axis fastest.  p = y (b = x): x-fastest copy at 0;
    // p = x (b = y): y-fastest copy at G.off1.
    const int base_off = p == 1 ? 0 : G.off1;
    const int stride_b = 1;
    const int stride_p = p == 1 ? G.px : G.py;
    const int np = P.n[p], nbi = P.n[b];
    const bool mp = w[p] < 0.0, mb = w[b] < 0.0;
    R.sp = mp ? -stride_p : stride_p;
    R.sb = mb ? -stride_b : stride_b;
    R.pad_[0] = p;  // slab axis: 0 = x, 1 = y
    const int base = base_off + stride_p * (mp ? np - 1 + kPlaneHalo : kPlaneHalo) +
                     stride_b * (mb ? nbi - 1 + kPlaneHalo : kPlaneHalo);
    R.addr = base + R.sp * R.k0 + R.sb * R.jb;
    T[ray] = R;
}

// One slab of a plane ray: at most one transverse crossing, two pieces.
template <bool CLAMP, class Op>
__device__ __forceinline__ void plane_slab(uint32_t &fb, uint32_t bb, float ib, int &jb,
                                           int &addr, int sp, int sb, float lo, float hi, Op &op)
{
    const uint32_t gb = fb + bb;
    const bool cb = gb < fb;
    float e = cb ? fmaxf(__fmaf_rn(-__uint2float_rn(gb), ib, 1.0f), 0.0f) : 1.0f;
    if (CLAMP) e = fminf(fmaxf(e, lo), hi);
    const float d0 = CLAMP ? __fsub_rn(e, lo) : e;
    const float d1 = __fsub_rn(CLAMP ? hi : 1.0f, e);
    op(addr, d0, true, jb);
    op(addr + sb, d1, cb, jb + 1);
    addr += sp + (cb ? sb : 0);
    jb += cb ? 1 : 0;
    fb = gb;
}

template <class Op>
__device__ __forceinline__ void plane_walk(const PlaneRay &R, Op &op)
{
    uint32_t fb = R.fb;
    int jb = R.jb, addr = R.addr;
    plane_slab<true>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, R.tlo, R.k0 == R.k1 ? R.thi : 1.0f,
                     op);
    for (int k = R.k0 + 1; k < R.k1; ++k)
        plane_slab<false>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, 0.0f, 1.0f, op);
    if (R.k1 > R.k0) plane_slab<true>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, 0.0f, R.thi, op);
}

// Walk the slabs [ka, kb] of a ray (a chunk of [k0, k1]).  The fixed-point
// state at slab ka follows exactly from the state at k0: the transverse position
// in 2^-32 cell units is a 64-bit integer that grows by bb per slab, so its
// carries up to ka are ((fb + (ka - k0) bb) >> 32).  The chunks of a ray thus
// visit exactly the pieces of the whole walk.
template <class Op>
__device__ __forceinline__ void plane_walk_range(const PlaneRay &R, int ka, int kb, Op &op)
{
    const unsigned long long n = (unsigned long long)(ka - R.k0);
    const unsigned long long F = (unsigned long long)R.fb + n * (unsigned long long)R.bb;
    const int carries = (int)(F >> 32);
    uint32_t fb = (uint32_t)F;
    int jb = R.jb + carries;
    int addr = R.addr + (int)n * R.sp + carries * R.sb;
    int k = ka;
    if (ka == R.k0 || ka == R.k1) {
        plane_slab<true>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, ka == R.k0 ? R.tlo : 0.0f,
                         ka == R.k1 ? R.thi : 1.0f, op);
        ++k;
    }
    const int kend = kb == R.k1 ? kb - 1 : kb;
    for (; k <= kend; ++k) plane_slab<false>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, 0.0f, 1.0f, op);
    if (kb == R.k1 && kb > ka) plane_slab<true>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, 0.0f, R.thi, op);
}

// Lockstep walk of the slabs [la, lb] of a ray inside a warp-uniform slab loop
// [ka, kb] ([la, lb] within both [ka, kb] and the ray's [k0, k1]; la > lb: the
// lane walks nothing and its op is switched off).  Every lane of the warp steps
// the same slab k at the same time, so the 32 adjacent rays of a view touch one
// row of the padded copy per instruction (consecutive transverse cells) instead
// of rows as far apart as their entry slabs.  The fixed-point state jumps
// exactly to slab la, as in plane_walk_range, so the pieces are those of the
// whole walk.  The slabs where every active lane is inside its range and off
// its ray's end slabs run unclamped and untested; only the warp's boundary
// slabs clamp to [lo, hi] (the ray's own ends, else [0, 1]) and test the range.
template <class Op>
__device__ __forceinline__ void plane_walk_lockstep(const PlaneRay &R, int ka, int kb, int la,
                                                    int lb, Op &op)
{
    const bool active = la <= lb;
    const int start = active ? la : R.k0;
    const unsigned long long n = (unsigned long long)(start - R.k0);
    const unsigned long long F = (unsigned long long)R.fb + n * (unsigned long long)R.bb;
    const int carries = (int)(F >> 32);
    uint32_t fb = (uint32_t)F;
    int jb = R.jb + carries;
    int addr = R.addr + (int)n * R.sp + carries * R.sb;
    op.live = active;
    // a chunk of the warp's union of ranges can fall in a gap between the
    // lanes' ranges: then no lane walks anything
    if (!__any_sync(0xffffffffu, active)) return;
    // interior [ia, ib] within [ka, kb] (idle lanes pass the chunk's own ends)
    const int ia = __reduce_max_sync(0xffffffffu, active ? max(la, R.k0 + 1) : ka);
    const int ib = __reduce_min_sync(0xffffffffu, active ? min(lb, R.k1 - 1) : kb);
    const int ea = ia <= ib ? ia : kb + 1;
    for (int k = ka; k < ea; ++k) {
        if (k < la || k > lb) continue;
        plane_slab<true>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, k == R.k0 ? R.tlo : 0.0f,
                         k == R.k1 ? R.thi : 1.0f, op);
    }
    if (ia > ib) return;
    for (int k = ia; k <= ib; ++k)
        plane_slab<false>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, 0.0f, 1.0f, op);
    for (int k = ib + 1; k <= kb; ++k) {
        if (k < la || k > lb) continue;
        plane_slab<true>(fb, R.bb, R.ib, jb, addr, R.sp, R.sb, k == R.k0 ? R.tlo : 0.0f,
                         k == R.k1 ? R.thi : 1.0f, op);
    }
}

// Warp-uniform chunk [ka, kb] of the union of the live lanes' slab ranges, cut
// in CH equal parts (chunk c of CH), and this lane's part [la, lb] of it.
// Returns false when the warp has no live lane or the chunk is empty.
template <int CH>
__device__ __forceinline__ bool plane_lockstep_range(const PlaneRay &R, bool live, int chunk,
                                                     int &ka, int &kb, int &la, int &lb)
{
    const int K0 = __reduce_min_sync(0xffffffffu, live ? R.k0 : 0x7fffffff);
    const int K1 = __reduce_max_sync(0xffffffffu, live ? R.k1 : -0x7fffffff);
    if (K0 > K1) return false;
    const int len = (K1 - K0 + CH) / CH;
    ka = K0 + chunk * len;
    kb = min(ka + len - 1, K1);
    if (ka > kb) return false;
    la = live ? max(ka, R.k0) : 1;
    lb = live ? min(kb, R.k1) : 0;
    return true;
}

struct PlaneGather {
    const float *__restrict__ img;
    float acc;
    long long lim;  // cells of the padded copies (bounds-checked builds)
    __device__ __forceinline__ void operator()(int a, float d, bool on, int)
    {
        if (on && ctp_in(a, lim, kSitePlaneGather)) acc = __fmaf_rn(d, __ldg(img + a), acc);
    }
};

// A piece of zero length adds 0 (no test: the first piece of a slab is all
// but never empty, the second goes out only after a crossing).  live: the
// lane walks a ray in this chunk (the lockstep walk switches idle lanes off).
struct PlaneScatter {
    float *__restrict__ img;
    float w;
    long long lim;
    bool live = true;
    __device__ __forceinline__ void operator()(int a, float d, bool on, int)
    {
        if (on && live && ctp_in(a, lim, kSitePlaneScatter)) atomicAdd(img + a, __fmul_rn(d, w));
    }
};

// Cells of the two padded copies (x-fastest, then y-fastest) of one accumulator.
__host__ __device__ __forceinline__ long long plane_cells(const RayParams &P)
{
    return 2LL * (P.n[0] + 2 * kPlaneHalo) * (P.n[1] + 2 * kPlaneHalo);
}

struct PlaneCount {
    unsigned n;
    float thr;
    unsigned nb;
    __device__ __forceinline__ void operator()(int, float d, bool on, int jb)
    {
        n += (on && (unsigned)jb < nb && d > thr) ? 1u : 0u;
    }
};

constexpr int kPlaneBlock = 128;

// Chunked kernels: a block holds 32 adjacent rays of one view (the lanes) and
// CH chunks of their slab ranges (the warps), CH * 32 threads.
template <int CH>
__global__ void __launch_bounds__(32 * CH) plane_forward_kernel(RayParams P,
                                                                const PlaneRay *__restrict__ T,
                                                                const float *__restrict__ img,
                                                                float *__restrict__ sino)
{
    __shared__ float part[CH][32];
    const int lane = threadIdx.x & 31, chunk = threadIdx.x >> 5;
    const int iu = blockIdx.x * 32 + lane;
    const long long ray = (long long)(P.view0 + (int)blockIdx.y) * P.n_u + iu;
    float acc = 0.0f;
    PlaneRay R;
    R.k0 = 0;
    R.k1 = -1;
    R.ell = 0.0f;
    // The warp's union of slab ranges is cut in CH chunks (the same boundaries
    // for every lane), and each lane walks its own ray's part of its chunk on
    // its own: in the chunks where no ray of the warp starts or ends, the lanes
    // step the same slabs together and their gathers fall on one row of the
    // padded copy, without the idle iterations of a lockstep walk.  C2 forward:
    // each ray cut in CH parts of its own 0.138 ms, lockstep over the union
    // 0.152 ms (0.193 ms clamping every slab), this 0.111 ms.  (The backward,
    // bound by its reduction sectors, keeps the lockstep walk: 0.216 against
    // 0.256 ms this way.)
    if (iu < P.n_u) R = plane_ray_walk_state(T, ray);
    int ka, kb, la, lb;
    if (plane_lockstep_range<CH>(R, R.k0 <= R.k1, chunk, ka, kb, la, lb) && la <= lb) {
        PlaneGather op{img, 0.0f, plane_cells(P)};
        plane_walk_range(R, la, lb, op);
        acc = op.acc;
    }
    part[chunk][lane] = acc;
    __syncthreads();
    if (chunk == 0 && iu < P.n_u) {
        float sum = 0.0f;
#pragma unroll
        for (int c = 0; c < CH; ++c) sum = __fadd_rn(sum, part[c][lane]);
        if (ctp_in(ray, sino_cells(P), kSitePlaneSinoStore)) sino[ray] = __fmul_rn(sum, R.ell);
    }
}

// View s accumulates into copy s % copies of the padded buffers (copy_cells
// floats apart): concurrent views of a small image then rarely update the same
// L2 lines; the unpack adds the copies.
template <int CH>
__global__ void __launch_bounds__(32 * CH) plane_backward_kernel(RayParams P,
                                                                 const PlaneRay *__restrict__ T,
                                                                 const float *__restrict__ sino,
                                                                 float *__restrict__ img,
                                                                 int copies, long long copy_cells)
{
    const int lane = threadIdx.x & 31, chunk = threadIdx.x >> 5;
    const int iu = blockIdx.x * 32 + lane;
    const int view = P.view0 + (int)blockIdx.y;
    const long long ray = (long long)view * P.n_u + iu;
    float y = 0.0f;
    PlaneRay R;
    R.k0 = 0;
    R.k1 = -1;
    R.ell = 0.0f;
    if (iu < P.n_u && ctp_in(ray, sino_cells(P), kSitePlaneSinoLoad)) {
        y = sino[ray];
        if (y != 0.0f) R = plane_ray_walk_state(T, ray);
    }
    int ka, kb, la, lb;
    if (!plane_lockstep_range<CH>(R, y != 0.0f && R.k0 <= R.k1, chunk, ka, kb, la, lb)) return;
    PlaneScatter op{img + (long long)(view % copies) * copy_cells, __fmul_rn(R.ell, y),
                    plane_cells(P)};
    plane_walk_lockstep(R, ka, kb, la, lb, op);
}

__global__ void __launch_bounds__(kPlaneBlock) plane_count_kernel(RayParams P,
                                                                  const PlaneRay *__restrict__ T,
                                                                  unsigned long long *__restrict__ total)
{
    const long long ray =
        (long long)(P.view0 + (int)blockIdx.y) * P.n_u + blockIdx.x * kPlaneBlock + threadIdx.x;
    unsigned n = 0;
    if (blockIdx.x * kPlaneBlock + threadIdx.x < P.n_u) {
        const PlaneRay R = plane_ray_record(T, ray);
        if (R.k0 <= R.k1) {
            PlaneCount op{0u, __fdiv_rn(P.min_len, R.ell), (unsigned)R.nb};
            plane_walk(R, op);
            n = op.n;
        }
    }
    n = __reduce_add_sync(0xffffffffu, n);
    if ((threadIdx.x & 31) == 0 && n) atomicAdd(total, (unsigned long long)n);
}

// image (ny, nx) x-fastest  ->  interiors of both padded copies.
__global__ void __launch_bounds__(256) plane_pack_kernel(PlaneLayout G, const float *__restrict__ in,
                                                         float *__restrict__ buf)
{
    __shared__ float tile[32][33];
    const int x0 = blockIdx.x * 32, y0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int j = ty; j < 32; j += 8) {
        const int y = y0 + j, x = x0 + tx;
        if (y < G.ny && x < G.nx) {
            const float v = in[(size_t)y * G.nx + x];
            tile[j][tx] = v;
            buf[(size_t)(y + kPlaneHalo) * G.px + (x + kPlaneHalo)] = v;
        }
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int x = x0 + j, y = y0 + tx;
        if (x < G.nx && y < G.ny)
            buf[G.off1 + (size_t)(x + kPlaneHalo) * G.py + (y + kPlaneHalo)] = tile[tx][j];
    }
}

// Sum over the copies of one cell (stride apart), added in copy order to v.
// The loads go out four at a time: a thread sums several cells over every
// copy, and one load in flight per thread left the unpack latency-bound
// (C2: 31 us of 34 MB in the launch list).
__device__ __forceinline__ float plane_sum_copies(const float *__restrict__ p, int copies,
                                                  long long stride, float v)
{
    int c = 0;
    for (; c + 4 <= copies; c += 4) {
        const float *q = p + c * stride;
        const float a0 = q[0], a1 = q[stride], a2 = q[2 * stride], a3 = q[3 * stride];
        v = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(v, a0), a1), a2), a3);
    }
    for (; c < copies; ++c) v = __fadd_rn(v, p[c * stride]);
    return v;
}

// out (ny, nx) = sum over copies of (interior of the x-fastest buffer +
// transposed interior of the y-fastest buffer).
__global__ void __launch_bounds__(256) plane_unpack_kernel(PlaneLayout G,
                                                           const float *__restrict__ buf,
                                                           float *__restrict__ out, int copies,
                                                           long long copy_cells)
{
    __shared__ float tile[32][33];
    const int x0 = blockIdx.x * 32, y0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int j = ty; j < 32; j += 8) {
        const int x = x0 + j, y = y0 + tx;
        if (x < G.nx && y < G.ny)
            tile[j][tx] = plane_sum_copies(
                buf + G.off1 + (size_t)(x + kPlaneHalo) * G.py + (y + kPlaneHalo), copies,
                copy_cells, 0.0f);
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int y = y0 + j, x = x0 + tx;
        if (y < G.ny && x < G.nx)
            out[(size_t)y * G.nx + x] = plane_sum_copies(
                buf + (size_t)(y + kPlaneHalo) * G.px + (x + kPlaneHalo), copies, copy_cells,
                tile[tx][j]);
    }
}

// ---------------------------------------------------------------------------
// Tiled backward (small scans): a block owns a kTile x kTile tile of the image and a range of
// views.  For each view it walks the rays that cross the tile (found by
// projecting the tile's corners onto the detector line), only over the slabs
// and transverse cells inside the tile, with the walk state jumped exactly to
// the tile's first slab.  Pieces accumulate in shared memory; the finished tile
// is added to the zeroed output once.  Every (slab, cell) piece of a ray lies in
// exactly one tile, so the tiles together visit exactly the pieces of the walk.
// ---------------------------------------------------------------------------
constexpr int kTile = 32;

struct TileScatter {
    float *tile;      // shared memory, (kTile) x (kTile + 1), x fastest
    float w;
    int jlo;          // mirrored transverse index of the tile's first in-tile cell
    unsigned tb;      // tile extent along the transverse axis
    __device__ __forceinline__ void operator()(int a, float d, bool on, int jb)
    {
        if (on && d > 0.0f && (unsigned)(jb - jlo) < tb &&
            ctp_in(a, kTile * (kTile + 1), kSitePlaneTile))
            atomicAdd(tile + a, __fmul_rn(d, w));
    }
};

// Detector-line coordinate iu of the ray through cell-coordinate point (x, y)
// of view V (float32 is ample: the result only bounds a candidate range).
// Divergent beams: NaN when the point is not on the detector's side of the
// source (its rays then do not form an interval bounded by the corners).
__device__ __forceinline__ float plane_project_u(const ViewFrame &V, int beam, float x, float y)
{
    const float ax = (float)V.a[0], ay = (float)V.a[1];
    const float px = (float)V.p00[0], py = (float)V.p00[1];
    const float dx = (float)V.du[0], dy = (float)V.du[1];
    if (beam == 1) {  // (p00 + iu du - S) x (X - S) = 0
        const float qx = x - ax, qy = y - ay;
        const float num = (px - ax) * qy - (py - ay) * qx;
        const float den = dx * qy - dy * qx;
        // the ray S + lam (X - S) meets the detector line at lam = ((p00 - S) x du) / ((X - S) x du)
        const float lam_num = (px - ax) * dy - (py - ay) * dx;
        const float lam_den = qx * dy - qy * dx;
        if (!(lam_num * lam_den > 0.0f)) return __int_as_float(0x7fffffff);
        return -num / den;
    }
    // parallel: (p00 + iu du - X) x a = 0
    const float num = (x - px) * ay - (y - py) * ax;
    const float den = dx * ay - dy * ax;
    return num / den;
}

__global__ void __launch_bounds__(256) plane_backward_tiled_kernel(RayParams P,
                                                                   const PlaneRay *__restrict__ T,
                                                                   const float *__restrict__ sino,
                                                                   float *__restrict__ out,
                                                                   int views_per_block)
{
    __shared__ float tile[kTile * (kTile + 1)];
    const int ntx = (P.n[0] + kTile - 1) / kTile;
    const int tx0 = (blockIdx.x % ntx) * kTile, ty0 = (blockIdx.x / ntx) * kTile;
    const int tnx = min(kTile, P.n[0] - tx0), tny = min(kTile, P.n[1] - ty0);
    for (int i = threadIdx.x; i < kTile * (kTile + 1); i += blockDim.x) tile[i] = 0.0f;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s_begin = blockIdx.y * views_per_block;
    const int s_end = min(P.n_views, s_begin + views_per_block);
    // warps take views far apart in angle (warp w: s_begin + w * span + i), so the
    // concurrently updated cells of the tile differ; a block of fewer than 8
    // views gives each view 8 / nv warps, which split its rays in runs of 32
    const int nv = s_end - s_begin;
    const int wpv = nv >= 8 ? 1 : 8 / nv;  // warps per view
    const int span = wpv == 1 ? (nv + 7) / 8 : 1;
    const int slice = warp % wpv;
    for (int i = 0; i < span; ++i) {
        const int s = s_begin + (wpv == 1 ? warp * span + i : warp / wpv);
        if (s >= s_end) break;
        const ViewFrame &V = P.views[s];
        // candidate rays: projections of the tile's corners (cell coordinates)
        float umin = 3.0e38f, umax = -3.0e38f;
        bool bad = false;
        for (int c = 0; c < 4; ++c) {
            const float x = (float)(tx0 + ((c & 1) ? tnx : 0));
            const float y = (float)(ty0 + ((c & 2) ? tny : 0));
            const float u = plane_project_u(V, P.beam, x, y);
            bad |= !(fabsf(u) < 1.0e30f);
            umin = fminf(umin, u);
            umax = fmaxf(umax, u);
        }
        // a corner behind the source or a degenerate view: take every ray
        int u0 = 0, u1 = P.n_u - 1;
        if (!bad && umax - umin < (float)P.n_u) {
            u0 = max(0, (int)floorf(umin) - 1);
            u1 = min(P.n_u - 1, (int)ceilf(umax) + 1);
        }
        for (int iu = u0 + 32 * slice + lane; iu <= u1; iu += 32 * wpv) {
            const long long ray = (long long)s * P.n_u + iu;
            if (!ctp_in(ray, sino_cells(P), kSitePlaneSinoLoad)) continue;
            const float y = sino[ray];
            if (y == 0.0f) continue;
            const PlaneRay R = plane_ray_record(T, ray);
            if (R.k0 > R.k1) continue;
            const int p = R.pad_[0];
            const bool mp = R.sp < 0, mb = R.sb < 0;
            const int np = P.n[p], nbv = P.n[1 - p];
            const int tp0 = p == 0 ? tx0 : ty0, tb0 = p == 0 ? ty0 : tx0;
            const int tpn = p == 0 ? tnx : tny, tbn = p == 0 ? tny : tnx;
            // the tile's slab range and transverse range in the ray's mirrored indices
            const int klo = mp ? np - tp0 - tpn : tp0;
            const int jlo = mb ? nbv - tb0 - tbn : tb0;
            const int ka = max(R.k0, klo), kb = min(R.k1, klo + tpn - 1);
            if (ka > kb) continue;
            // shared-memory address of mirrored cell (k, j): x fastest, row pitch kTile + 1
            const int pitch = kTile + 1;
            const int sp = (p == 0 ? 1 : pitch) * (mp ? -1 : 1);
            const int sb = (p == 0 ? pitch : 1) * (mb ? -1 : 1);
            // natural local index of mirrored k is (mp ? np-1-k : k) - tp0, likewise for j
            const int cp = (p == 0 ? 1 : pitch) * (mp ? np - 1 - tp0 : -tp0);
            const int cb = (p == 0 ? pitch : 1) * (mb ? nbv - 1 - tb0 : -tb0);
            PlaneRay L = R;
            L.addr = cp + cb + sp * R.k0 + sb * R.jb;
            L.sp = sp;
            L.sb = sb;
            TileScatter op{tile, __fmul_rn(R.ell, y), jlo, (unsigned)tbn};
            plane_walk_range(L, ka, kb, op);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTile * kTile; i += blockDim.x) {
        const int ly = i / kTile, lx = i % kTile;
        if (lx < tnx && ly < tny) {
            const float v = tile[ly * (kTile + 1) + lx];
            const long long o = (long long)(ty0 + ly) * P.n[0] + tx0 + lx;
            if (v != 0.0f && ctp_in(o, (long long)P.n[0] * P.n[1], kSitePlaneTileOut))
                atomicAdd(out + o, v);
        }
    }
}

inline size_t plane_buffer_cells(const PlaneLayout &G) { return 2 * (size_t)G.px * G.py; }

// Accumulator copies of the backward: as many as fit 48 MiB (they stay in L2),
// at most 8 and never more than the views.  More copies spread concurrent
// views' reductions over more L2 lines, fewer cost less zero-fill and unpack
// (C2 backward with 2 / 4 / 8 / 16 copies: 0.231 / 0.225 / 0.220 / 0.223 ms).
inline int plane_copies(const RayParams &P, const PlaneLayout &G)
{
    const size_t one = sizeof(float) * plane_buffer_cells(G);
    int c = (int)(((size_t)48 << 20) / (one > 0 ? one : 1));
    c = c > 8 ? 8 : (c < 1 ? 1 : c);
    if (P.n_views > 0 && c > P.n_views) c = P.n_views;
    return c < 1 ? 1 : c;
}

// Builds the per-ray table and the two combined padded buffers (forward:
// halo zeroed once, interiors rewritten per call; backward: zeroed per call).
// Returns 0, 9 (CUDA error) or 11 (scan not eligible for the plane path).
inline int plane_plan_build(const RayParams &P, void **d_rays, float **d_fwd, float **d_bwd,
                            unsigned long long *bytes)
{
    const PlaneLayout G = plane_layout(P);
    if (plane_buffer_cells(G) >= (1ULL << 31)) return 11;
    const long long n_rays = (long long)P.n_views * P.n_u;
    const size_t rbytes = sizeof(PlaneRay) * (size_t)(n_rays > 0 ? n_rays : 1);
    const size_t vbytes = sizeof(float) * plane_buffer_cells(G);
    const size_t bbytes = vbytes * (size_t)plane_copies(P, G);
    int *d_flag = nullptr;
    if (cudaMalloc(d_rays, rbytes) != cudaSuccess || cudaMalloc(d_fwd, vbytes) != cudaSuccess ||
        cudaMalloc(d_bwd, bbytes) != cudaSuccess || cudaMemset(*d_fwd, 0, vbytes) != cudaSuccess ||
        cudaMalloc(&d_flag, sizeof(int)) != cudaSuccess ||
        cudaMemset(d_flag, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(d_flag);
        return 9;
    }
    *bytes += rbytes + vbytes + bbytes;
    if (n_rays > 0) {
        const int threads = 128;
        const long long blocks = (n_rays + threads - 1) / threads;
        plane_setup_kernel<<<(unsigned)blocks, threads>>>(P, G, (PlaneRay *)*d_rays, d_flag);
    }
    int flag = 0;
    const bool ok = cudaGetLastError() == cudaSuccess &&
                    cudaMemcpy(&flag, d_flag, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaFree(d_flag);
    if (!ok) return 9;
    return flag ? 11 : 0;
}

inline dim3 plane_grid(const RayParams &P)
{
    return dim3((P.n_u + kPlaneBlock - 1) / kPlaneBlock, P.view_count, 1);
}

// Chunks per ray: enough threads for about `waves` waves of the whole GPU
// (forward 4; the backward 8, its lockstep chunks measured faster shorter:
// C2 backward with 2 / 4 / 8 chunks 0.228 / 0.216 / 0.212 ms, the forward
// 0.117 / 0.111 / 0.118 ms).
inline int plane_chunks(const RayParams &P, int waves = 4)
{
    const long long rays = (long long)P.n_views * P.n_u;
    const long long want = (long long)waves * 148 * 2048;
    int ch = 1;
    while (ch < 8 && rays * ch < want) ch *= 2;
    return ch;
}

inline dim3 plane_chunk_grid(const RayParams &P)
{
    return dim3((P.n_u + 31) / 32, P.view_count, 1);
}

inline dim3 plane_tgrid(const PlaneLayout &G)
{
    return dim3((G.nx + 31) / 32, (G.ny + 31) / 32, 1);
}

// Stages of a call (see the column path): layout in, walk over P's view range,
// layout out.  Small scans (launch- and latency-bound) use the shared-memory
// tiled backward, which walks all views in one launch (plane_backward_whole).
// Larger ones use fire-and-forget global reductions into the privatised padded
// copies, which measured faster than shared-memory float atomics (C2: 0.46 vs
// 0.66 ms).  mode: 0 = by size, 1 = tiled, 2 = privatised (a plan option).
inline bool plane_backward_tiled(const RayParams &P, int mode)
{
    if (mode == 1) return true;
    if (mode == 2) return false;
    return (long long)P.n_views * P.n_u <= 65536;
}

inline int plane_layout_in(const RayParams &P, float *d_fwd, const float *img, cudaStream_t s)
{
    const PlaneLayout G = plane_layout(P);
    plane_pack_kernel<<<plane_tgrid(G), 256, 0, s>>>(G, img, d_fwd);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int plane_walk_forward(const RayParams &P, const void *d_rays, const float *d_fwd,
                              float *sino, cudaStream_t s)
{
    if (P.view_count <= 0) return 0;
    const PlaneRay *T = (const PlaneRay *)d_rays;
    switch (plane_chunks(P)) {
    case 8: plane_forward_kernel<8><<<plane_chunk_grid(P), 256, 0, s>>>(P, T, d_fwd, sino); break;
    case 4: plane_forward_kernel<4><<<plane_chunk_grid(P), 128, 0, s>>>(P, T, d_fwd, sino); break;
    case 2: plane_forward_kernel<2><<<plane_chunk_grid(P), 64, 0, s>>>(P, T, d_fwd, sino); break;
    default: plane_forward_kernel<1><<<plane_chunk_grid(P), 32, 0, s>>>(P, T, d_fwd, sino); break;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

// Privatised-accumulator backward: prepare, walk view ranges, layout out.  (A
// layout out that zeroed the copies as it read them, in place of the
// zero-fill, measured slower: C2 0.223 -> 0.313 ms.)
inline int plane_backward_prepare(const RayParams &P, float *d_bwd, cudaStream_t s)
{
    const PlaneLayout G = plane_layout(P);
    const size_t bytes = sizeof(float) * plane_buffer_cells(G) * plane_copies(P, G);
    return cudaMemsetAsync(d_bwd, 0, bytes, s) == cudaSuccess ? 0 : 9;
}

inline int plane_walk_backward(const RayParams &P, const void *d_rays, const float *sino,
                               float *d_bwd, cudaStream_t s)
{
    if (P.view_count <= 0 || P.n_u <= 0) return 0;
    const PlaneLayout G = plane_layout(P);
    const int copies = plane_copies(P, G);
    const long long copy_cells = (long long)plane_buffer_cells(G);
    const PlaneRay *T = (const PlaneRay *)d_rays;
    const dim3 g = plane_chunk_grid(P);
    switch (plane_chunks(P, 8)) {
    case 8: plane_backward_kernel<8><<<g, 256, 0, s>>>(P, T, sino, d_bwd, copies, copy_cells); break;
    case 4: plane_backward_kernel<4><<<g, 128, 0, s>>>(P, T, sino, d_bwd, copies, copy_cells); break;
    case 2: plane_backward_kernel<2><<<g, 64, 0, s>>>(P, T, sino, d_bwd, copies, copy_cells); break;
    default: plane_backward_kernel<1><<<g, 32, 0, s>>>(P, T, sino, d_bwd, copies, copy_cells); break;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int plane_layout_out(const RayParams &P, const float *d_bwd, float *img, cudaStream_t s)
{
    const PlaneLayout G = plane_layout(P);
    plane_unpack_kernel<<<plane_tgrid(G), 256, 0, s>>>(G, d_bwd, img, plane_copies(P, G),
                                                        (long long)plane_buffer_cells(G));
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

// Small scans: zero the output, one block per (32 x 32 tile, view group), all
// views.  (A one-launch variant -- one block per 8 x 8 tile over every view,
// storing its tile -- measured slower on the 64 x 64 scan: 0.048 against
// 0.022 ms; a block then walks all 90 views serially.)
inline int plane_backward_whole(const RayParams &P, const void *d_rays, const float *sino,
                                float *img, cudaStream_t s)
{
    if (cudaMemsetAsync(img, 0, sizeof(float) * (size_t)P.n[0] * P.n[1], s) != cudaSuccess)
        return 9;
    if ((long long)P.n_views * P.n_u == 0) return 0;
    // view groups: enough blocks for about four per SM, down to one view per
    // block on small images (C1 with one warp per view: 1 / 2 / 4 / 8 views per
    // block 16.5 / 16.9 / 17.1 / 19.1 us per call, the extra tile flushes
    // cheaper than serial views; 12.1 us with a view's rays split over the
    // block's 8 warps)
    const int tiles = ((P.n[0] + kTile - 1) / kTile) * ((P.n[1] + kTile - 1) / kTile);
    int groups = (4 * 148 + tiles - 1) / tiles;
    groups = max(1, min(groups, P.n_views));
    const int vpb = (P.n_views + groups - 1) / groups;
    groups = (P.n_views + vpb - 1) / vpb;
    plane_backward_tiled_kernel<<<dim3(tiles, groups), 256, 0, s>>>(
        P, (const PlaneRay *)d_rays, sino, img, vpb);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

inline int plane_count(const RayParams &P, const void *d_rays, unsigned long long *d_total,
                       cudaStream_t s)
{
    plane_count_kernel<<<plane_grid(P), kPlaneBlock, 0, s>>>(P, (const PlaneRay *)d_rays, d_total);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

}  // namespace ctp
