// C ABI of the Siddon projector pair: validation, plans, launches.
//
// Host side of the boundary declared in include/ctp.h.  Validation follows the
// pages' error set for frame vectors (non-finite, coincident source/detector,
// the 1e6 and 1e15 magnitude limits; diffct tests/test_surface_geometry_cudasim.py,
// release diff 2.4.1 -> 2.4.2, the failure/message parametrisation) and the native
// spacing bounds ([1e-6, 1e6], max/min ratio <= 1e4; diffct CHANGELOG 2.4.4).
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ctp.h"
#include "ctp_column.cuh"
#include "ctp_fdk.cuh"
#include "ctp_geometry.cuh"
#include "ctp_plane.cuh"
#include "ctp_internal.h"
#include "ctp_ray.cuh"

struct ctp_plan {
    int device = 0;
    int path = CTP_PATH_RAY;
    int ndim = 3, beam = 1;
    int n_views = 0, n_u = 0, n_v = 0;
    int n[3] = {0, 0, 0};
    double spacing[3] = {0, 0, 0};
    double origin[3] = {0, 0, 0};
    double pitch_u = 1, pitch_v = 1, offset_u = 0, offset_v = 0;
    long long n_rays = 0, n_cells = 0;
    std::vector<ctp::ViewFrame> frames;     // host copy
    std::vector<float> raw;                 // the caller's frames: src, centre, u, v (n_views x 12)
    ctp::ViewFrame *d_frames = nullptr;     // device copy
    float *d_offsets = nullptr;             // curved detector: pixel offsets (t, s, e)
    int offsets_per_view = 0;               // 1: one (n_v, n_u, 3) table per view
    ctp::ColumnOffsets *d_columns = nullptr;  // curved detector, column path: per column
    unsigned long long *d_counter = nullptr;
    // column and plane paths
    ctp::ColumnPlan col{};
    void *d_table = nullptr;                // ColumnTrace (column) or PlaneRay (plane) table
    float *d_work_fwd = nullptr;            // padded working copy read by the forward
    float *d_work_bwd = nullptr;            // padded accumulator of the backward
    // host-buffer entry points
    float *d_stage_vol = nullptr, *d_stage_sino = nullptr;
    cudaStream_t copy_stream = nullptr;     // sinogram chunks move here, beside the walk
    cudaEvent_t ev_start = nullptr;         // work queued on the caller's stream before a call
    cudaEvent_t ev_chunk[64] = {};          // chunk c walked (forward) or staged (backward)
    // analytical operators
    int fdk_status = CTP_E_GEOMETRY;
    ctp::FdkParams fdk{};
    ctp::FdkView *d_fdk = nullptr;
    float *d_ramp[ctp::kRampKinds] = {};    // ramp kernels (2 n_u - 1) by ctp_ramp value
    bool ramp_odd[ctp::kRampKinds] = {};    // even nonzero taps all zero (Ram-Lak)
    unsigned long long device_bytes = 0;
    ctp_plan_options opt{};                 // work-layout options (all zero: defaults)
};

namespace {

bool finite3(const float *v) { return std::isfinite(v[0]) && std::isfinite(v[1]) && std::isfinite(v[2]); }

double norm3(const double *v) { return std::sqrt(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]); }

void cross3(const double *a, const double *b, double *out)
{
    out[0] = a[1] * b[2] - a[2] * b[1];
    out[1] = a[2] * b[0] - a[0] * b[2];
    out[2] = a[0] * b[1] - a[1] * b[0];
}

int check_device(const ctp_plan_t *plan)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return CTP_E_CUDA;
    return dev == plan->device ? CTP_OK : CTP_E_DEVICE;
}

ctp::RayParams ray_params(const ctp_plan_t *plan)
{
    ctp::RayParams P{};
    P.views = plan->d_frames;
    P.beam = plan->beam;
    P.n_u = plan->n_u;
    P.n_v = plan->n_v;
    P.n_views = plan->n_views;
    for (int a = 0; a < 3; ++a) {
        P.n[a] = plan->n[a];
        P.spacing[a] = plan->spacing[a];
    }
    P.stride[0] = 1;
    P.stride[1] = plan->n[0];
    P.stride[2] = plan->n[0] * plan->n[1];
    P.min_len = (float)(1e-5 * std::fmin(plan->spacing[0],
                                         std::fmin(plan->spacing[1], plan->spacing[2])));
    P.view0 = 0;
    P.view_count = plan->n_views;
    P.offsets = plan->d_offsets;
    P.offsets_per_view = plan->offsets_per_view;
    P.columns = plan->d_columns;
    return P;
}

// Parameters of a launch over views [v0, v0 + nv).
ctp::RayParams view_range(const ctp_plan_t *plan, int v0, int nv)
{
    ctp::RayParams P = ray_params(plan);
    P.view0 = v0;
    P.view_count = nv;
    return P;
}

// Threads of one ray block: 32 (u) x 4 (v) for 3-D scans, 128 (u) for single-row detectors.
int launch_ray(const ctp::RayParams &P, int which, const float *in, float *out,
               unsigned long long *counter, cudaStream_t s)
{
    if (P.view_count <= 0) return CTP_OK;
    if (P.n_v == 1) {
        dim3 grid((P.n_u + 127) / 128, P.view_count, 1), block(128);
        if (which == 0) ctp::ray_forward_kernel<128, 1><<<grid, block, 0, s>>>(P, in, out);
        else if (which == 1) ctp::ray_backward_kernel<128, 1><<<grid, block, 0, s>>>(P, in, out);
        else ctp::ray_count_kernel<128, 1><<<grid, block, 0, s>>>(P, counter);
    } else {
        dim3 grid((P.n_u + 31) / 32, P.view_count, (P.n_v + 3) / 4), block(128);
        if (which == 0) ctp::ray_forward_kernel<32, 4><<<grid, block, 0, s>>>(P, in, out);
        else if (which == 1) ctp::ray_backward_kernel<32, 4><<<grid, block, 0, s>>>(P, in, out);
        else ctp::ray_count_kernel<32, 4><<<grid, block, 0, s>>>(P, counter);
    }
    return cudaGetLastError() == cudaSuccess ? CTP_OK : CTP_E_CUDA;
}

// Stages of the two operators, shared by the device- and host-buffer entry
// points.  Forward: forward_in (layout of the volume) then forward_walk over
// view ranges.  Backward: backward_in (zero the accumulator), backward_walk over
// view ranges, backward_out (fold the accumulator into the output volume).
// The walks index the sinogram by absolute view, so a range's launch reads or
// writes only that range's rows.
int forward_in(const ctp_plan_t *plan, const float *vol, cudaStream_t s)
{
    const ctp::RayParams P = ray_params(plan);
    if (plan->path == CTP_PATH_COLUMN)
        return ctp::column_layout_in(P, plan->d_work_fwd, vol, s) ? CTP_E_CUDA : CTP_OK;
    if (plan->path == CTP_PATH_PLANE)
        return ctp::plane_layout_in(P, plan->d_work_fwd, vol, s) ? CTP_E_CUDA : CTP_OK;
    return CTP_OK;
}

int forward_walk(const ctp_plan_t *plan, int v0, int nv, const float *vol, float *sino,
                 cudaStream_t s)
{
    const ctp::RayParams P = view_range(plan, v0, nv);
    if (plan->path == CTP_PATH_COLUMN)
        return ctp::column_walk_forward(P, plan->col, plan->d_table, plan->d_work_fwd, sino, s)
                   ? CTP_E_CUDA : CTP_OK;
    if (plan->path == CTP_PATH_PLANE)
        return ctp::plane_walk_forward(P, plan->d_table, plan->d_work_fwd, sino, s) ? CTP_E_CUDA
                                                                                    : CTP_OK;
    return launch_ray(P, 0, vol, sino, nullptr, s);
}

// Small 2-D scans take a single tiled launch over all views instead.
bool backward_whole(const ctp_plan_t *plan)
{
    return plan->path == CTP_PATH_PLANE &&
           ctp::plane_backward_tiled(ray_params(plan), plan->opt.plane_backward);
}

int backward_in(const ctp_plan_t *plan, float *vol, cudaStream_t s)
{
    const ctp::RayParams P = ray_params(plan);
    if (plan->path == CTP_PATH_COLUMN)
        return ctp::column_backward_prepare(P, plan->d_work_bwd, s) ? CTP_E_CUDA : CTP_OK;
    if (plan->path == CTP_PATH_PLANE)
        return ctp::plane_backward_prepare(P, plan->d_work_bwd, s) ? CTP_E_CUDA : CTP_OK;
    return cudaMemsetAsync(vol, 0, sizeof(float) * plan->n_cells, s) == cudaSuccess ? CTP_OK
                                                                                     : CTP_E_CUDA;
}

int backward_walk(const ctp_plan_t *plan, int v0, int nv, const float *sino, float *vol,
                  cudaStream_t s)
{
    const ctp::RayParams P = view_range(plan, v0, nv);
    if (plan->path == CTP_PATH_COLUMN)
        return ctp::column_walk_backward(P, plan->col, plan->d_table, sino, plan->d_work_bwd, s)
                   ? CTP_E_CUDA : CTP_OK;
    if (plan->path == CTP_PATH_PLANE)
        return ctp::plane_walk_backward(P, plan->d_table, sino, plan->d_work_bwd, s) ? CTP_E_CUDA
                                                                                     : CTP_OK;
    return launch_ray(P, 1, sino, vol, nullptr, s);
}

int backward_out(const ctp_plan_t *plan, float *vol, cudaStream_t s)
{
    const ctp::RayParams P = ray_params(plan);
    if (plan->path == CTP_PATH_COLUMN)
        return ctp::column_layout_out(P, plan->d_work_bwd, vol, s) ? CTP_E_CUDA : CTP_OK;
    if (plan->path == CTP_PATH_PLANE)
        return ctp::plane_layout_out(P, plan->d_work_bwd, vol, s) ? CTP_E_CUDA : CTP_OK;
    return CTP_OK;
}

void free_plan(ctp_plan_t *p)
{
    if (!p) return;
    cudaDeviceSynchronize();
    cudaFree(p->d_frames);
    cudaFree(p->d_offsets);
    cudaFree(p->d_columns);
    cudaFree(p->d_counter);
    cudaFree(p->d_table);
    cudaFree(p->d_work_fwd);
    cudaFree(p->d_work_bwd);
    cudaFree(p->d_stage_vol);
    cudaFree(p->d_stage_sino);
    cudaFree(p->d_fdk);
    for (float *h : p->d_ramp) cudaFree(h);
    if (p->copy_stream) cudaStreamDestroy(p->copy_stream);
    if (p->ev_start) cudaEventDestroy(p->ev_start);
    for (cudaEvent_t e : p->ev_chunk)
        if (e) cudaEventDestroy(e);
    delete p;
}

int validate(const ctp_geometry *g, const ctp_volume *v)
{
    if (g->ndim != 2 && g->ndim != 3) return CTP_E_OPTION;
    if (g->beam != CTP_PARALLEL && g->beam != CTP_DIVERGENT) return CTP_E_OPTION;
    if (v->nx < 1 || v->ny < 1 || v->nz < 1 || v->nx > 32768 || v->ny > 32768 || v->nz > 32768)
        return CTP_E_SHAPE;
    if ((long long)v->nx * v->ny * v->nz >= (1LL << 31)) return CTP_E_SHAPE;
    if (g->n_views < 0 || g->n_u < 1 || g->n_v < 1 || g->n_views > 65535) return CTP_E_SHAPE;
    if ((g->n_v + 3) / 4 > 65535) return CTP_E_SHAPE;
    if ((long long)g->n_views * g->n_u * g->n_v >= (1LL << 40)) return CTP_E_SHAPE;
    if (g->ndim == 2 && (v->nz != 1 || g->n_v != 1)) return CTP_E_SHAPE;
    const double sp[3] = {v->dx, v->dy, v->dz};
    const double org[3] = {v->ox, v->oy, v->oz};
    for (int a = 0; a < 3; ++a)
        if (!std::isfinite(sp[a]) || !std::isfinite(org[a])) return CTP_E_NONFINITE;
    if (!std::isfinite(g->pitch_u) || !std::isfinite(g->pitch_v) || !std::isfinite(g->offset_u) ||
        !std::isfinite(g->offset_v))
        return CTP_E_NONFINITE;
    // 2-D scans ignore dz (one cell along z); only the in-plane pitches are bound.
    const int naxes = g->ndim == 2 ? 2 : 3;
    double smin = 1e300, smax = 0;
    for (int a = 0; a < naxes; ++a) {
        if (!(sp[a] >= 1e-6 && sp[a] <= 1e6)) return CTP_E_SPACING;
        smin = std::fmin(smin, sp[a]);
        smax = std::fmax(smax, sp[a]);
    }
    if (g->ndim == 2 && !(sp[2] > 0.0)) return CTP_E_SPACING;
    if (smax / smin > 1e4) return CTP_E_SPACING;
    if (!(g->pitch_u > 0.0) || !(g->pitch_v > 0.0)) return CTP_E_SHAPE;
    if (g->offsets_per_view != 0 && g->offsets_per_view != 1) return CTP_E_OPTION;
    if (g->pixel_offsets) {
        const long long tables = g->offsets_per_view ? g->n_views : 1;
        for (long long q = 0; q < 3LL * g->n_u * g->n_v * tables; ++q)
            if (!std::isfinite(g->pixel_offsets[q])) return CTP_E_NONFINITE;
    }
    if (g->n_views == 0) return CTP_OK;
    if (!g->src || !g->det_centre || !g->det_u || !g->det_v) return CTP_E_NULL;

    const double centre[3] = {v->ox + 0.5 * v->nx * v->dx, v->oy + 0.5 * v->ny * v->dy,
                              v->oz + 0.5 * v->nz * v->dz};
    for (int s = 0; s < g->n_views; ++s) {
        const float *S = g->src + 3 * s, *C = g->det_centre + 3 * s;
        const float *U = g->det_u + 3 * s, *V = g->det_v + 3 * s;
        if (!finite3(S) || !finite3(C) || !finite3(U) || !finite3(V)) return CTP_E_NONFINITE;
        double Sd[3], Cd[3], Ud[3], Vd[3], nrm[3];
        for (int a = 0; a < 3; ++a) {
            Sd[a] = S[a];
            Cd[a] = C[a];
            Ud[a] = U[a];
            Vd[a] = V[a];
        }
        cross3(Ud, Vd, nrm);
        if (!(norm3(Ud) > 0) || !(norm3(Vd) > 0) || !(norm3(nrm) > 1e-6 * norm3(Ud) * norm3(Vd)))
            return CTP_E_AXES;
        // magnitude limits on positions relative to the volume centre
        const double *pts[2] = {Sd, Cd};
        for (int q = 0; q < 2; ++q) {
            if (q == 0 && g->beam == CTP_PARALLEL) continue;
            for (int a = 0; a < 3; ++a)
                if (std::fabs(pts[q][a] - centre[a]) > 1e15) return CTP_E_FAR;
            for (int a = 0; a < 3; ++a)
                if (std::fabs(pts[q][a] - centre[a]) > 1e6 * smax) return CTP_E_NEAR;
        }
        if (g->beam == CTP_PARALLEL) {
            if (!(norm3(Sd) > 0)) return CTP_E_AXES;
            const double dn = std::fabs(Sd[0] * nrm[0] + Sd[1] * nrm[1] + Sd[2] * nrm[2]);
            if (!(dn > 1e-9 * norm3(Sd) * norm3(nrm))) return CTP_E_COINCIDENT;
        } else {
            // the source must not lie in the detector plane (some pixel would coincide)
            double SC[3] = {Sd[0] - Cd[0], Sd[1] - Cd[1], Sd[2] - Cd[2]};
            const double dn = std::fabs(SC[0] * nrm[0] + SC[1] * nrm[1] + SC[2] * nrm[2]);
            if (!(dn > 1e-9 * norm3(nrm) * (norm3(SC) + 1e-300))) return CTP_E_COINCIDENT;
        }
    }
    return CTP_OK;
}

// Tables of the analytical operators (small: one FdkView per view and the two
// ramp kernels).  A scan outside their class only records CTP_E_GEOMETRY.
int fdk_setup(ctp_plan_t *p, const ctp_geometry *g, const ctp_volume *v)
{
    if (g->pixel_offsets) {
        p->fdk_status = CTP_E_GEOMETRY;  // flat detectors only
        return CTP_OK;
    }
    std::vector<ctp::FdkView> views;
    const int n[3] = {v->nx, v->ny, v->nz};
    const double d[3] = {v->dx, v->dy, v->dz}, o[3] = {v->ox, v->oy, v->oz};
    const int st = ctp::fdk_build(g->ndim, g->beam, g->n_views, g->n_u, g->n_v, g->src,
                                  g->det_centre, g->det_u, g->det_v, g->pitch_u, g->pitch_v,
                                  g->offset_u, g->offset_v, n, d, o, views, p->fdk);
    if (st != 0) {
        p->fdk_status = CTP_E_GEOMETRY;
        return CTP_OK;
    }
    const size_t vbytes = sizeof(ctp::FdkView) * views.size();
    if (cudaMalloc(&p->d_fdk, vbytes) != cudaSuccess ||
        cudaMemcpy(p->d_fdk, views.data(), vbytes, cudaMemcpyHostToDevice) != cudaSuccess)
        return CTP_E_CUDA;
    p->device_bytes += vbytes;
    p->fdk.views = p->d_fdk;
    if (g->n_u <= ctp::kFilterMaxU) {
        for (int kind = 0; kind < ctp::kRampKinds; ++kind) {
            std::vector<float> h;
            ctp::fdk_ramp_kernel(g->n_u, g->pitch_u, kind, h);
            p->ramp_odd[kind] = ctp::ramp_taps_odd(h, g->n_u);
            const size_t hb = sizeof(float) * h.size();
            if (cudaMalloc(&p->d_ramp[kind], hb) != cudaSuccess ||
                cudaMemcpy(p->d_ramp[kind], h.data(), hb, cudaMemcpyHostToDevice) != cudaSuccess)
                return CTP_E_CUDA;
            p->device_bytes += hb;
        }
    }
    p->fdk_status = CTP_OK;
    return CTP_OK;
}

// Per-view frame of a flat detector in cell coordinates (float64): the source
// (divergent) or ray direction (parallel) a, pixel (0, 0) p00 and the pixel
// steps du, dv along u and v.  ctp_plan and ctp_forward_static both take their
// frames from here.
void flat_view_frame(const ctp_geometry *g, const ctp_volume *v, int s, ctp::ViewFrame *F)
{
    const double spacing[3] = {v->dx, v->dy, v->dz};
    const double origin[3] = {v->ox, v->oy, v->oz};
    const double cu = 0.5 * (g->n_u - 1) - g->offset_u;
    const double cv = 0.5 * (g->n_v - 1) - g->offset_v;
    const float *S = g->src + 3 * s, *C = g->det_centre + 3 * s;
    const float *U = g->det_u + 3 * s, *V = g->det_v + 3 * s;
    for (int a = 0; a < 3; ++a) {
        const double d = spacing[a], o = origin[a];
        const double pu = g->pitch_u * (double)U[a];
        const double pv = g->pitch_v * (double)V[a];
        // pixel (0, 0) = centre - cu * pitch_u * u - cv * pitch_v * v
        const double p00 = (double)C[a] - cu * pu - cv * pv;
        F->a[a] = g->beam == CTP_DIVERGENT ? ((double)S[a] - o) / d : (double)S[a] / d;
        F->p00[a] = (p00 - o) / d;
        F->du[a] = pu / d;
        F->dv[a] = pv / d;
        F->dn[a] = 0.0;
    }
}

// Per-view frame of a curved detector: pixel = centre + t u + s v + e n with
// per-pixel offsets in physical units; p00 holds the centre, du / dv / dn the
// unit axes and the unit normal n = u x v / |u x v|, all in cell coordinates.
void curved_view_frame(const ctp_geometry *g, const ctp_volume *v, int s, ctp::ViewFrame *F)
{
    const double spacing[3] = {v->dx, v->dy, v->dz};
    const double origin[3] = {v->ox, v->oy, v->oz};
    const float *S = g->src + 3 * s, *C = g->det_centre + 3 * s;
    const float *U = g->det_u + 3 * s, *V = g->det_v + 3 * s;
    const double Ud[3] = {U[0], U[1], U[2]}, Vd[3] = {V[0], V[1], V[2]};
    double N[3];
    cross3(Ud, Vd, N);
    const double nn = norm3(N);
    for (int a = 0; a < 3; ++a) {
        const double d = spacing[a], o = origin[a];
        F->a[a] = g->beam == CTP_DIVERGENT ? ((double)S[a] - o) / d : (double)S[a] / d;
        F->p00[a] = ((double)C[a] - o) / d;
        F->du[a] = Ud[a] / d;
        F->dv[a] = Vd[a] / d;
        F->dn[a] = N[a] / nn / d;
    }
}

int validate_options(const ctp_plan_options *o)
{
    if (!o) return CTP_OK;
    const bool ok = o->rows_forward >= 0 && o->rows_forward <= 4 && o->rows_backward >= 0 &&
                    o->rows_backward <= 4 &&
                    (o->backward_rows_adjacent == 0 || o->backward_rows_adjacent == 1) &&
                    o->plane_backward >= 0 && o->plane_backward <= 2 && o->host_chunks >= 0 &&
                    o->host_chunks <= 64 && (o->geometry_walk == 0 || o->geometry_walk == 1) &&
                    o->forward_ahead >= 0 && o->forward_ahead <= 2 &&
                    o->forward_views_first >= 0 && o->forward_views_first <= 2;
    return ok ? CTP_OK : CTP_E_OPTION;
}

int fdk_check(const ctp_plan_t *plan)
{
    const int st = check_device(plan);
    return st != CTP_OK ? st : plan->fdk_status;
}

}  // namespace

extern "C" {

const char *ctp_status_string(int status)
{
    switch (status) {
    case CTP_OK: return "ok";
    case CTP_E_NULL: return "a required pointer is NULL";
    case CTP_E_SHAPE: return "sizes out of range";
    case CTP_E_NONFINITE: return "geometry and grid values must be finite";
    case CTP_E_COINCIDENT: return "source and detector must differ";
    case CTP_E_NEAR: return "frame coordinates must lie within 1e6 voxel widths of the volume";
    case CTP_E_FAR: return "frame coordinates must be below 1e15 in magnitude";
    case CTP_E_SPACING: return "spacing must be in [1e-6, 1e6] with max/min <= 1e4";
    case CTP_E_AXES: return "detector axes must be non-zero and not parallel";
    case CTP_E_CUDA: return "CUDA runtime error";
    case CTP_E_DEVICE: return "current CUDA device differs from the plan's";
    case CTP_E_OPTION: return "unknown ndim, beam or path";
    case CTP_E_LIMIT: return "request exceeds a fixed limit of this entry point";
    case CTP_E_GEOMETRY:
        return "scan outside the analytical operators' class (3-D needs v = +-z, u horizontal)";
    default: return "unknown status";
    }
}

int ctp_check_violations(unsigned long long *count, long long *index, long long *extent,
                         int *site)
{
    if (!count || !index || !extent || !site) return CTP_E_NULL;
#ifdef CTP_CHECK
    ctp::CheckState h{};
    const ctp::CheckState zero{};
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&h, ctp::ctp_check_state, sizeof h) != cudaSuccess ||
        cudaMemcpyToSymbol(ctp::ctp_check_state, &zero, sizeof zero) != cudaSuccess)
        return CTP_E_CUDA;
    *count = h.count;
    *index = h.index;
    *extent = h.extent;
    *site = h.site;
    return CTP_OK;
#else
    *count = 0;
    *index = *extent = 0;
    *site = 0;
    return CTP_E_OPTION;
#endif
}

int ctp_plan(const ctp_geometry *geom, const ctp_volume *vol, int path, ctp_plan_t **out)
{
    return ctp_plan_ex(geom, vol, path, nullptr, out);
}

int ctp_plan_ex(const ctp_geometry *geom, const ctp_volume *vol, int path,
                const ctp_plan_options *options, ctp_plan_t **out)
{
    if (!out) return CTP_E_NULL;
    *out = nullptr;
    if (!geom || !vol) return CTP_E_NULL;
    if (path != CTP_PATH_AUTO && path != CTP_PATH_RAY && path != CTP_PATH_COLUMN &&
        path != CTP_PATH_PLANE)
        return CTP_E_OPTION;
    int st = validate_options(options);
    if (st != CTP_OK) return st;
    st = validate(geom, vol);
    if (st != CTP_OK) return st;

    ctp_plan_t *p = new (std::nothrow) ctp_plan_t();
    if (!p) return CTP_E_CUDA;
    if (options) p->opt = *options;
    if (cudaGetDevice(&p->device) != cudaSuccess) {
        delete p;
        return CTP_E_CUDA;
    }
    p->ndim = geom->ndim;
    p->beam = geom->beam;
    p->n_views = geom->n_views;
    p->n_u = geom->n_u;
    p->n_v = geom->n_v;
    p->n[0] = vol->nx;
    p->n[1] = vol->ny;
    p->n[2] = vol->nz;
    p->spacing[0] = vol->dx;
    p->spacing[1] = vol->dy;
    p->spacing[2] = vol->dz;
    p->origin[0] = vol->ox;
    p->origin[1] = vol->oy;
    p->origin[2] = vol->oz;
    p->pitch_u = geom->pitch_u;
    p->pitch_v = geom->pitch_v;
    p->offset_u = geom->offset_u;
    p->offset_v = geom->offset_v;
    p->n_rays = (long long)geom->n_views * geom->n_u * geom->n_v;
    p->raw.assign(12 * (size_t)geom->n_views, 0.0f);
    for (int s = 0; s < geom->n_views; ++s)
        for (int a = 0; a < 3; ++a) {
            p->raw[12 * (size_t)s + a] = geom->src[3 * s + a];
            p->raw[12 * (size_t)s + 3 + a] = geom->det_centre[3 * s + a];
            p->raw[12 * (size_t)s + 6 + a] = geom->det_u[3 * s + a];
            p->raw[12 * (size_t)s + 9 + a] = geom->det_v[3 * s + a];
        }
    p->n_cells = (long long)vol->nx * vol->ny * vol->nz;

    // Per-view frames in cell coordinates, float64.
    p->frames.resize(geom->n_views > 0 ? geom->n_views : 1);
    bool v_is_z = geom->ndim == 3;
    const bool curved = geom->pixel_offsets != nullptr;
    for (int s = 0; s < geom->n_views; ++s) {
        if (curved) curved_view_frame(geom, vol, s, &p->frames[s]);
        else flat_view_frame(geom, vol, s, &p->frames[s]);
        const float *V = geom->det_v + 3 * s;
        if (!(V[0] == 0.0f && V[1] == 0.0f && V[2] != 0.0f)) v_is_z = false;
    }
    // A curved detector runs on the column path when its columns are straight
    // vertical lines of evenly spaced pixels (tangent and depth offsets the same
    // in every row, vertical offsets affine in the row to 1e-6 of the column's
    // span): circular / helical scans with cylindrical detectors.  Other curved
    // detectors run on the ray path; the plane path assumes the pitch grid.
    // With one table per view, every view's columns are checked and tabled.
    std::vector<ctp::ColumnOffsets> colq;
    p->offsets_per_view = curved && geom->offsets_per_view ? 1 : 0;
    const int tables = p->offsets_per_view ? geom->n_views : 1;
    if (curved) {
        bool columnar = geom->ndim == 3 && geom->n_v >= 2;
        for (int t = 0; t < tables && columnar; ++t)
            for (int iu = 0; iu < geom->n_u && columnar; ++iu) {
                const float *q0 = geom->pixel_offsets + 3LL * geom->n_u * geom->n_v * t + 3LL * iu;
                const float *q1 = q0 + 3LL * geom->n_u;
                const double s0 = q0[1], ds = (double)q1[1] - (double)q0[1];
                const double span = std::fabs(ds) * (geom->n_v - 1);
                for (int iv = 1; iv < geom->n_v && columnar; ++iv) {
                    const float *q = q0 + 3LL * geom->n_u * iv;
                    columnar = q[0] == q0[0] && q[2] == q0[2] &&
                               std::fabs((double)q[1] - (s0 + ds * iv)) <= 1e-6 * span;
                }
                colq.push_back(ctp::ColumnOffsets{q0[0], q0[2], s0, ds});
            }
        if (!columnar) {
            colq.clear();
            v_is_z = false;
        }
        if ((path == CTP_PATH_COLUMN && !v_is_z) || path == CTP_PATH_PLANE) {
            free_plan(p);
            return CTP_E_OPTION;
        }
    }

    int chosen = path;
    if (chosen == CTP_PATH_AUTO)
        chosen = curved ? (v_is_z ? CTP_PATH_COLUMN : CTP_PATH_RAY)
                        : (geom->ndim == 2 ? CTP_PATH_PLANE
                                           : (v_is_z ? CTP_PATH_COLUMN : CTP_PATH_RAY));
    if ((chosen == CTP_PATH_COLUMN && (!v_is_z || geom->ndim != 3)) ||
        (chosen == CTP_PATH_PLANE && geom->ndim != 2)) {
        free_plan(p);
        return CTP_E_OPTION;
    }
    p->path = chosen;

    size_t fbytes = sizeof(ctp::ViewFrame) * p->frames.size();
    if (cudaMalloc(&p->d_frames, fbytes) != cudaSuccess ||
        cudaMemcpy(p->d_frames, p->frames.data(), fbytes, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&p->d_counter, sizeof(unsigned long long)) != cudaSuccess) {
        free_plan(p);
        return CTP_E_CUDA;
    }
    p->device_bytes = fbytes + sizeof(unsigned long long);
    if (curved) {
        const size_t ob = sizeof(float) * 3 * (size_t)geom->n_u * geom->n_v * (size_t)tables;
        if (cudaMalloc(&p->d_offsets, ob) != cudaSuccess ||
            cudaMemcpy(p->d_offsets, geom->pixel_offsets, ob, cudaMemcpyHostToDevice) !=
                cudaSuccess) {
            free_plan(p);
            return CTP_E_CUDA;
        }
        p->device_bytes += ob;
        if (chosen == CTP_PATH_COLUMN) {
            const size_t cb = sizeof(ctp::ColumnOffsets) * colq.size();
            if (cudaMalloc(&p->d_columns, cb) != cudaSuccess ||
                cudaMemcpy(p->d_columns, colq.data(), cb, cudaMemcpyHostToDevice) !=
                    cudaSuccess) {
                free_plan(p);
                return CTP_E_CUDA;
            }
            p->device_bytes += cb;
        }
    }
    if (chosen == CTP_PATH_COLUMN || chosen == CTP_PATH_PLANE) {
        // every view's source and detector centre at one height (a circular
        // scan): then views first for the column forward's blocks
        bool level = true;
        for (int v = 1; v < p->n_views && level; ++v)
            level = p->raw[12 * (size_t)v + 2] == p->raw[2] && p->raw[12 * (size_t)v + 5] == p->raw[5];
        const int views_first = p->opt.forward_views_first == 0 ? (level ? 2 : 1)
                                                                 : p->opt.forward_views_first;
        if (chosen == CTP_PATH_COLUMN)
            st = ctp::column_plan_build(ray_params(p), p->opt.rows_forward, p->opt.rows_backward,
                                        p->opt.backward_rows_adjacent != 0,
                                        p->opt.forward_ahead, views_first == 2, &p->col,
                                        &p->d_table, &p->d_work_fwd,
                                        &p->d_work_bwd, &p->device_bytes);
        else
            st = ctp::plane_plan_build(ray_params(p), &p->d_table, &p->d_work_fwd,
                                       &p->d_work_bwd, &p->device_bytes);
        if (st == CTP_E_OPTION && path == CTP_PATH_AUTO) {
            // column: some rows cross more than one z plane per slab; plane: some
            // rays leave the slice plane.  Use the ray path.
            cudaFree(p->d_table);
            cudaFree(p->d_work_fwd);
            cudaFree(p->d_work_bwd);
            cudaFree(p->d_columns);
            p->d_table = nullptr;
            p->d_work_fwd = nullptr;
            p->d_work_bwd = nullptr;
            p->d_columns = nullptr;
            p->device_bytes = fbytes + sizeof(unsigned long long) +
                              (curved ? sizeof(float) * 3 * (size_t)geom->n_u * geom->n_v *
                                            (size_t)tables
                                      : 0);
            p->path = CTP_PATH_RAY;
            st = CTP_OK;
        }
        if (st != CTP_OK) {
            free_plan(p);
            return st;
        }
    }
    if ((st = fdk_setup(p, geom, vol)) != CTP_OK) {
        free_plan(p);
        return st;
    }
    *out = p;
    return CTP_OK;
}

void ctp_destroy(ctp_plan_t *plan) { free_plan(plan); }

int ctp_plan_info_get(const ctp_plan_t *plan, ctp_plan_info *info)
{
    if (!plan || !info) return CTP_E_NULL;
    info->path = plan->path;
    info->device = plan->device;
    info->n_rays = plan->n_rays;
    info->n_cells = plan->n_cells;
    info->device_bytes = plan->device_bytes;
    return CTP_OK;
}

int ctp_forward(const ctp_plan_t *plan, const float *vol_dev, float *sino_dev, void *stream)
{
    if (!plan) return CTP_E_NULL;
    if (plan->n_rays > 0 && (!vol_dev || !sino_dev)) return CTP_E_NULL;
    int st = check_device(plan);
    if (st != CTP_OK) return st;
    if (plan->n_rays == 0) return CTP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = forward_in(plan, vol_dev, s)) != CTP_OK) return st;
    return forward_walk(plan, 0, plan->n_views, vol_dev, sino_dev, s);
}

int ctp_backward(const ctp_plan_t *plan, const float *sino_dev, float *vol_dev, void *stream)
{
    if (!plan || !vol_dev || (plan->n_rays > 0 && !sino_dev)) return CTP_E_NULL;
    int st = check_device(plan);
    if (st != CTP_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (backward_whole(plan))
        return ctp::plane_backward_whole(ray_params(plan), plan->d_table, sino_dev, vol_dev, s)
                   ? CTP_E_CUDA : CTP_OK;
    if ((st = backward_in(plan, vol_dev, s)) != CTP_OK) return st;
    if (plan->n_rays > 0 && (st = backward_walk(plan, 0, plan->n_views, sino_dev, vol_dev, s)) != CTP_OK)
        return st;
    return backward_out(plan, vol_dev, s);
}

int ctp_segment_count(const ctp_plan_t *plan, unsigned long long *out, void *stream)
{
    if (!plan || !out) return CTP_E_NULL;
    int st = check_device(plan);
    if (st != CTP_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    *out = 0;
    if (plan->n_rays == 0) return CTP_OK;
    if (cudaMemsetAsync(plan->d_counter, 0, sizeof(unsigned long long), s) != cudaSuccess)
        return CTP_E_CUDA;
    const ctp::RayParams P = ray_params(plan);
    if (plan->path == CTP_PATH_COLUMN)
        st = ctp::column_count(P, plan->col, plan->d_table, plan->d_counter, s);
    else if (plan->path == CTP_PATH_PLANE)
        st = ctp::plane_count(P, plan->d_table, plan->d_counter, s);
    else
        st = launch_ray(P, 2, nullptr, nullptr, plan->d_counter, s);
    if (st != CTP_OK) return CTP_E_CUDA;
    if (cudaMemcpyAsync(out, plan->d_counter, sizeof(unsigned long long), cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return CTP_E_CUDA;
    return CTP_OK;
}

static int ensure_stage(ctp_plan_t *plan)
{
    if (!plan->d_stage_vol) {
        if (cudaMalloc(&plan->d_stage_vol, sizeof(float) * plan->n_cells) != cudaSuccess)
            return CTP_E_CUDA;
        plan->device_bytes += sizeof(float) * plan->n_cells;
    }
    if (!plan->d_stage_sino && plan->n_rays > 0) {
        if (cudaMalloc(&plan->d_stage_sino, sizeof(float) * plan->n_rays) != cudaSuccess)
            return CTP_E_CUDA;
        plan->device_bytes += sizeof(float) * plan->n_rays;
    }
    if (!plan->copy_stream) {
        if (cudaStreamCreateWithFlags(&plan->copy_stream, cudaStreamNonBlocking) != cudaSuccess)
            return CTP_E_CUDA;
        if (cudaEventCreateWithFlags(&plan->ev_start, cudaEventDisableTiming) != cudaSuccess)
            return CTP_E_CUDA;
        for (cudaEvent_t &e : plan->ev_chunk)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                return CTP_E_CUDA;
    }
    return CTP_OK;
}

// Number of view chunks the host-buffer entry points pipeline: one per 64 MiB
// of sinogram, at most 8 (each chunk's walk still fills the GPU many times
// over), at most one per view.  The plan option host_chunks (1..64) overrides.
static int host_chunks(const ctp_plan_t *plan)
{
    long long c = (long long)(sizeof(float) * (unsigned long long)plan->n_rays >> 26);
    if (c > 8) c = 8;
    if (plan->opt.host_chunks >= 1) c = plan->opt.host_chunks;
    if (c > plan->n_views) c = plan->n_views;
    return c < 1 ? 1 : (int)c;
}

static int chunk_begin(const ctp_plan_t *plan, int c, int chunks)
{
    return (int)((long long)plan->n_views * c / chunks);
}

// Ends a failed host-buffer call: copies already queued still read or write the
// caller's buffers, so wait for them before returning.
static int host_fail(ctp_plan_t *plan, cudaStream_t s, int st)
{
    cudaStreamSynchronize(plan->copy_stream);
    cudaStreamSynchronize(s);
    return st;
}

// Forward over host buffers.  The volume goes up on the caller's stream; the
// walk runs in view chunks on the caller's stream and each finished chunk's
// sinogram rows go down on the plan's copy stream while the next chunk walks.
int ctp_forward_host(ctp_plan_t *plan, const float *vol_host, float *sino_host, void *stream)
{
    if (!plan || !vol_host || !sino_host) return CTP_E_NULL;
    int st = check_device(plan);
    if (st != CTP_OK) return st;
    if (plan->n_rays == 0) return CTP_OK;
    if ((st = ensure_stage(plan)) != CTP_OK) return st;
    cudaStream_t s = (cudaStream_t)stream, cs = plan->copy_stream;
    const size_t row = (size_t)plan->n_u * plan->n_v;     // sinogram floats of one view
    // the copy stream starts after whatever the caller queued on s before this call
    if (cudaEventRecord(plan->ev_start, s) != cudaSuccess ||
        cudaStreamWaitEvent(cs, plan->ev_start, 0) != cudaSuccess)
        return host_fail(plan, s, CTP_E_CUDA);
    if (cudaMemcpyAsync(plan->d_stage_vol, vol_host, sizeof(float) * plan->n_cells,
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
        return host_fail(plan, s, CTP_E_CUDA);
    if ((st = forward_in(plan, plan->d_stage_vol, s)) != CTP_OK) return host_fail(plan, s, st);
    const int chunks = host_chunks(plan);
    // all walks first: with pageable host memory a device-to-host copy returns
    // only once it is done, and the walks queued behind it would wait for it
    for (int c = 0; c < chunks; ++c) {
        const int v0 = chunk_begin(plan, c, chunks), v1 = chunk_begin(plan, c + 1, chunks);
        if ((st = forward_walk(plan, v0, v1 - v0, plan->d_stage_vol, plan->d_stage_sino, s)) !=
                CTP_OK ||
            cudaEventRecord(plan->ev_chunk[c], s) != cudaSuccess)
            return host_fail(plan, s, st != CTP_OK ? st : CTP_E_CUDA);
    }
    for (int c = 0; c < chunks; ++c) {
        const int v0 = chunk_begin(plan, c, chunks), v1 = chunk_begin(plan, c + 1, chunks);
        if (cudaStreamWaitEvent(cs, plan->ev_chunk[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(sino_host + row * v0, plan->d_stage_sino + row * v0,
                            sizeof(float) * row * (v1 - v0), cudaMemcpyDeviceToHost,
                            cs) != cudaSuccess)
            return host_fail(plan, s, CTP_E_CUDA);
    }
    if (cudaStreamSynchronize(cs) != cudaSuccess) return host_fail(plan, s, CTP_E_CUDA);
    return CTP_OK;
}

// Backward over host buffers.  Each view chunk's sinogram rows go up on the
// plan's copy stream and that chunk's walk waits only for them; the volume
// comes down on the caller's stream at the end.
int ctp_backward_host(ctp_plan_t *plan, const float *sino_host, float *vol_host, void *stream)
{
    if (!plan || !vol_host || (!sino_host && plan->n_rays > 0)) return CTP_E_NULL;
    int st = check_device(plan);
    if (st != CTP_OK) return st;
    if ((st = ensure_stage(plan)) != CTP_OK) return st;
    cudaStream_t s = (cudaStream_t)stream, cs = plan->copy_stream;
    const size_t row = (size_t)plan->n_u * plan->n_v;
    float *vol = plan->d_stage_vol;
    if (backward_whole(plan)) {
        if (plan->n_rays > 0 &&
            cudaMemcpyAsync(plan->d_stage_sino, sino_host, sizeof(float) * plan->n_rays,
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return host_fail(plan, s, CTP_E_CUDA);
        const float *sino = plan->n_rays > 0 ? plan->d_stage_sino : vol;
        if (ctp::plane_backward_whole(ray_params(plan), plan->d_table, sino, vol, s))
            return host_fail(plan, s, CTP_E_CUDA);
    } else {
        if (cudaEventRecord(plan->ev_start, s) != cudaSuccess ||
            cudaStreamWaitEvent(cs, plan->ev_start, 0) != cudaSuccess)
            return host_fail(plan, s, CTP_E_CUDA);
        if ((st = backward_in(plan, vol, s)) != CTP_OK) return host_fail(plan, s, st);
        const int chunks = plan->n_rays > 0 ? host_chunks(plan) : 0;
        for (int c = 0; c < chunks; ++c) {
            const int v0 = chunk_begin(plan, c, chunks), v1 = chunk_begin(plan, c + 1, chunks);
            if (cudaMemcpyAsync(plan->d_stage_sino + row * v0, sino_host + row * v0,
                                sizeof(float) * row * (v1 - v0), cudaMemcpyHostToDevice,
                                cs) != cudaSuccess ||
                cudaEventRecord(plan->ev_chunk[c], cs) != cudaSuccess ||
                cudaStreamWaitEvent(s, plan->ev_chunk[c], 0) != cudaSuccess)
                return host_fail(plan, s, CTP_E_CUDA);
            if ((st = backward_walk(plan, v0, v1 - v0, plan->d_stage_sino, vol, s)) != CTP_OK)
                return host_fail(plan, s, st);
        }
        if ((st = backward_out(plan, vol, s)) != CTP_OK) return host_fail(plan, s, st);
    }
    if (cudaMemcpyAsync(vol_host, vol, sizeof(float) * plan->n_cells, cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return host_fail(plan, s, CTP_E_CUDA);
    return CTP_OK;
}

int ctp_parker_weights(const ctp_plan_t *plan, float *weight_dev, void *stream)
{
    if (!plan) return CTP_E_NULL;
    if (plan->n_views > 0 && !weight_dev) return CTP_E_NULL;
    int st = check_device(plan);
    if (st != CTP_OK) return st;
    if (plan->beam != CTP_DIVERGENT || plan->d_offsets) return CTP_E_GEOMETRY;
    if (plan->n_views == 0) return CTP_OK;
    std::vector<float> src(3 * (size_t)plan->n_views), cen(src.size()), u(src.size());
    for (int k = 0; k < plan->n_views; ++k)
        for (int a = 0; a < 3; ++a) {
            src[3 * k + a] = plan->raw[12 * (size_t)k + a];
            cen[3 * k + a] = plan->raw[12 * (size_t)k + 3 + a];
            u[3 * k + a] = plan->raw[12 * (size_t)k + 6 + a];
        }
    const double iso[2] = {plan->origin[0] + 0.5 * plan->n[0] * plan->spacing[0],
                           plan->origin[1] + 0.5 * plan->n[1] * plan->spacing[1]};
    std::vector<float> w;
    ctp::fdk_parker(plan->n_views, plan->n_u, src.data(), cen.data(), u.data(), plan->pitch_u,
                    plan->offset_u, iso, w);
    cudaStream_t s = (cudaStream_t)stream;
    // the host vector dies with this call: copy, then wait for the copy
    if (cudaMemcpyAsync(weight_dev, w.data(), sizeof(float) * w.size(), cudaMemcpyHostToDevice,
                        s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return CTP_E_CUDA;
    return CTP_OK;
}

int ctp_ramp_filter(const ctp_plan_t *plan, const float *sino_dev, float *out_dev,
                    const float *view_weight_dev, const float *pixel_weight_dev, int ramp,
                    int transpose, void *stream)
{
    if (!plan) return CTP_E_NULL;
    if (plan->n_rays > 0 && (!sino_dev || !out_dev)) return CTP_E_NULL;
    if (ramp < CTP_RAMLAK || ramp > CTP_HANN) return CTP_E_OPTION;
    int st = fdk_check(plan);
    if (st != CTP_OK) return st;
    if (!plan->d_ramp[ramp]) return CTP_E_LIMIT;
    return ctp::fdk_filter(plan->fdk, plan->d_ramp[ramp], plan->ramp_odd[ramp], sino_dev, out_dev,
                           view_weight_dev,
                           pixel_weight_dev, transpose ? 1 : 0, (cudaStream_t)stream)
               ? CTP_E_CUDA : CTP_OK;
}

int ctp_weighted_backproject(const ctp_plan_t *plan, const float *sino_dev, float *vol_dev,
                             void *stream)
{
    if (!plan || !vol_dev || (plan->n_rays > 0 && !sino_dev)) return CTP_E_NULL;
    int st = fdk_check(plan);
    if (st != CTP_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (plan->n_rays == 0)
        return cudaMemsetAsync(vol_dev, 0, sizeof(float) * plan->n_cells, s) == cudaSuccess
                   ? CTP_OK : CTP_E_CUDA;
    return ctp::fdk_gather(plan->fdk, sino_dev, vol_dev, s) ? CTP_E_CUDA : CTP_OK;
}

int ctp_weighted_backproject_transpose(const ctp_plan_t *plan, const float *vol_dev,
                                       float *sino_dev, void *stream)
{
    if (!plan || !vol_dev || (plan->n_rays > 0 && !sino_dev)) return CTP_E_NULL;
    int st = fdk_check(plan);
    if (st != CTP_OK) return st;
    if (plan->n_rays == 0) return CTP_OK;
    return ctp::fdk_scatter(plan->fdk, vol_dev, sino_dev, (cudaStream_t)stream) ? CTP_E_CUDA
                                                                                : CTP_OK;
}

static ctp::GeomParams geom_params(const ctp_plan_t *plan)
{
    ctp::GeomParams Q;
    Q.cu = (float)(0.5 * (plan->n_u - 1) - plan->offset_u);
    Q.cv = (float)(0.5 * (plan->n_v - 1) - plan->offset_v);
    Q.pitch_u = (float)plan->pitch_u;
    Q.pitch_v = (float)plan->pitch_v;
    Q.pitch_ud = plan->pitch_u;
    Q.pitch_vd = plan->pitch_v;
    return Q;
}

int ctp_geometry_vjp(const ctp_plan_t *plan, const float *vol_dev, const float *weight_dev,
                     double *grad_dev, void *stream)
{
    if (!plan) return CTP_E_NULL;
    if (plan->n_views > 0 && !grad_dev) return CTP_E_NULL;
    if (plan->n_rays > 0 && (!vol_dev || !weight_dev)) return CTP_E_NULL;
    int st = check_device(plan);
    if (st != CTP_OK) return st;
    if (plan->n_views == 0) return CTP_OK;
    const ctp::GeomParams Q = geom_params(plan);
    cudaStream_t s = (cudaStream_t)stream;
    // the column walk takes flat detectors; curved ones run the ray walk
    if (plan->path == CTP_PATH_COLUMN && plan->opt.geometry_walk == 0 && !plan->d_offsets) {
        // the column walk reads the plan's padded z-fastest working copy
        if ((st = forward_in(plan, vol_dev, s)) != CTP_OK) return st;
        return ctp::column_geometry_vjp(ray_params(plan), Q, (const ctp::ColumnTrace *)plan->d_table,
                                        plan->d_work_fwd, weight_dev, grad_dev,
                                        plan->col.fwd_views_first, s)
                   ? CTP_E_CUDA : CTP_OK;
    }
    return ctp::geometry_vjp(ray_params(plan), Q, vol_dev, weight_dev, grad_dev, s) ? CTP_E_CUDA
                                                                                   : CTP_OK;
}

int ctp_surface_vjp(const ctp_plan_t *plan, const float *vol_dev, const float *weight_dev,
                    double *grad_dev, void *stream)
{
    if (!plan) return CTP_E_NULL;
    // the output is empty only for per-view tables of an empty scan
    const bool empty_out = plan->offsets_per_view && plan->n_views == 0;
    if ((!grad_dev && !empty_out) || (plan->n_rays > 0 && (!vol_dev || !weight_dev)))
        return CTP_E_NULL;
    int st = check_device(plan);
    if (st != CTP_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (plan->n_rays == 0)  // nothing to sum (a per-view table has no views to write)
        return plan->offsets_per_view ||
                       cudaMemsetAsync(grad_dev, 0,
                                       sizeof(double) * 3 * (size_t)plan->n_u * plan->n_v, s) ==
                           cudaSuccess
                   ? CTP_OK : CTP_E_CUDA;
    return ctp::surface_vjp(ray_params(plan), geom_params(plan), vol_dev, weight_dev, grad_dev, s)
               ? CTP_E_CUDA : CTP_OK;
}

int ctp_fdk(const ctp_plan_t *plan, const float *sino_dev, float *work_dev, float *vol_dev,
            const float *view_weight_dev, const float *pixel_weight_dev, int ramp, void *stream)
{
    if (!plan || !vol_dev || (plan->n_rays > 0 && (!sino_dev || !work_dev))) return CTP_E_NULL;
    int st = ctp_ramp_filter(plan, sino_dev, work_dev, view_weight_dev, pixel_weight_dev, ramp, 0,
                             stream);
    if (st != CTP_OK) return st;
    return ctp_weighted_backproject(plan, work_dev, vol_dev, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free forward projection.
//
// For callers that may not allocate device memory once they run: an application
// whose device memory belongs to its own pool allocator (a raw cudaMalloc there
// would take memory behind the pool's back and can fail when the pool has
// reserved the rest), or a loop that must not take cudaMalloc / cudaFree's
// implicit device synchronisation.  ctp_plan allocates its tables; this entry
// point keeps its only scratch -- the per-view frame table of the ray path --
// in a fixed file-scope device array instead.
// ---------------------------------------------------------------------------
namespace {

constexpr int kStaticMaxViews = 4096;   // 4096 frames x 120 B = 480 KiB per device
constexpr int kStaticMaxDevices = 64;
constexpr int kStaticChunk = 32;        // frames staged per host-to-device copy

// Shared by every call on a device and held by every device that loads the
// library until the process exits; keeps the last call's frames.
static __device__ __align__(256) ctp::ViewFrame g_static_frames[kStaticMaxViews];

// Driver calls that identify the current context, fetched through the runtime
// (the library does not link the driver library itself).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

struct StaticLookup {
    std::mutex lock;
    bool fetched = false;
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
    unsigned long long ctx_id[kStaticMaxDevices] = {};  // 0: not looked up yet
    void *addr[kStaticMaxDevices] = {};
};

StaticLookup &static_lookup()
{
    static StaticLookup L;
    return L;
}

// Unique id of the current context (0 when it cannot be told).
unsigned long long current_context_id(StaticLookup &L)
{
    if (!L.fetched) {
        L.fetched = true;
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            L.get_current = (CtxGetCurrentFn)fn;
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            L.get_id = (CtxGetIdFn)fn;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!L.get_current || !L.get_id || L.get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        L.get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_static_frames on the current device (host code may not
// use the symbol itself as a device pointer).  Looked up once per device and
// context: a context that was reset and recreated gets a fresh lookup.  When
// the context cannot be identified, every call looks the address up.
int static_frames_address(int device, ctp::ViewFrame **out)
{
    StaticLookup &L = static_lookup();
    std::lock_guard<std::mutex> guard(L.lock);
    unsigned long long id = current_context_id(L);
    if (id != 0 && L.ctx_id[device] == id) {
        *out = static_cast<ctp::ViewFrame *>(L.addr[device]);
        return CTP_OK;
    }
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_frames) != cudaSuccess || !ptr) return CTP_E_CUDA;
    if (id == 0) id = current_context_id(L);  // the lookup made the context current
    L.ctx_id[device] = id;
    L.addr[device] = ptr;
    *out = static_cast<ctp::ViewFrame *>(ptr);
    return CTP_OK;
}

}  // namespace

extern "C" int ctp_forward_static(const ctp_geometry *geom, const ctp_volume *vol,
                                  const float *vol_dev, float *sino_dev, void *stream)
{
    if (!geom || !vol) return CTP_E_NULL;
    int st = validate(geom, vol);
    if (st != CTP_OK) return st;
    if (geom->pixel_offsets) return CTP_E_OPTION;  // flat detectors only
    if (geom->n_views > kStaticMaxViews) return CTP_E_LIMIT;
    if (geom->n_views == 0) return CTP_OK;
    if (!vol_dev || !sino_dev) return CTP_E_NULL;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return CTP_E_CUDA;
    if (device < 0 || device >= kStaticMaxDevices) return CTP_E_LIMIT;
    ctp::ViewFrame *frames = nullptr;
    if ((st = static_frames_address(device, &frames)) != CTP_OK) return st;

    cudaStream_t s = (cudaStream_t)stream;
    ctp::ViewFrame chunk[kStaticChunk];
    for (int s0 = 0; s0 < geom->n_views; s0 += kStaticChunk) {
        const int n = geom->n_views - s0 < kStaticChunk ? geom->n_views - s0 : kStaticChunk;
        for (int q = 0; q < n; ++q) flat_view_frame(geom, vol, s0 + q, &chunk[q]);
        // pageable source: the copy may wait for the stream's earlier work, and it
        // returns once `chunk` has been staged, so the buffer can be refilled
        if (cudaMemcpyAsync(frames + s0, chunk, sizeof(ctp::ViewFrame) * n,
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return CTP_E_CUDA;
    }

    ctp::RayParams P{};
    P.views = frames;
    P.beam = geom->beam;
    P.n_u = geom->n_u;
    P.n_v = geom->n_v;
    P.n_views = geom->n_views;
    P.n[0] = vol->nx;
    P.n[1] = vol->ny;
    P.n[2] = vol->nz;
    P.spacing[0] = vol->dx;
    P.spacing[1] = vol->dy;
    P.spacing[2] = vol->dz;
    P.stride[0] = 1;
    P.stride[1] = vol->nx;
    P.stride[2] = vol->nx * vol->ny;
    P.min_len = (float)(1e-5 * std::fmin(vol->dx, std::fmin(vol->dy, vol->dz)));
    P.view0 = 0;
    P.view_count = geom->n_views;
    if (geom->n_v == 1) {
        dim3 grid((geom->n_u + 127) / 128, geom->n_views, 1);
        ctp::ray_forward_kernel<128, 1><<<grid, 128, 0, s>>>(P, vol_dev, sino_dev);
    } else {
        dim3 grid((geom->n_u + 31) / 32, geom->n_views, (geom->n_v + 3) / 4);
        ctp::ray_forward_kernel<32, 4><<<grid, 128, 0, s>>>(P, vol_dev, sino_dev);
    }
    return cudaGetLastError() == cudaSuccess ? CTP_OK : CTP_E_CUDA;
}
