// Internal types shared by the host plan code and the device kernels.
#pragma once

#include <cstdint>

namespace ctp {

// Per-view frame in CELL coordinates (x, y, z): world X maps to (X - o) / d.
// Divergent: a = source.  Parallel: a = ray direction (cell units).
// Flat detector: pixel (iu, iv) = p00 + iu * du + iv * dv.  Curved detector
// (per-pixel offsets (t, s, e)): pixel = p00 + t du + s dv + e dn with p00 the
// detector centre and du, dv, dn the unit axes and normal per unit length.
// Built on the host in float64.
struct ViewFrame {
    double a[3];
    double p00[3];
    double du[3];
    double dv[3];
    double dn[3];
};

// Curved detector with column structure: column iu's tangent and depth offsets
// (the same in every row), the vertical offset of row 0 and the step per row.
struct ColumnOffsets {
    double t, e, s0, ds;
};

// Launch-time constants of the ray path.
struct RayParams {
    const ViewFrame *views;
    int beam;             // 0 parallel, 1 divergent
    int n_u, n_v, n_views;
    int n[3];             // cells along x, y, z
    int stride[3];        // element stride of x, y, z in the (nz, ny, nx) buffer
    double spacing[3];    // dx, dy, dz
    float min_len;        // segment counter: pieces longer than this (physical units)
    int view0;            // first view of a launch (grid row y handles view view0 + y)
    int view_count;       // views of a launch
    const float *offsets; // curved detector: per-pixel offsets (t, s, e); else null
    int offsets_per_view; // 0: offsets (n_v, n_u, 3) shared; 1: (n_views, n_v, n_u, 3)
    const ColumnOffsets *columns;  // curved detector on the column path: per column
                                   // (per view and column with per-view tables); else null
};

// Bounds-checked debug build (compiled with -DCTP_CHECK): the projector walks
// test the index of every global load, store and reduction -- and the tiled
// backward of every shared-memory reduction -- against its buffer's extent
// before the access.  An index outside is counted in ctp_check_state (with the
// first offending index, its buffer's extent and the access site) and the
// access is skipped, so a wrong index shows up as a count, never as a fault.
// In normal builds ctp_in is the constant true and the tests vanish.
enum CheckSite {
    kSiteRayGather = 1, kSiteRayScatter, kSiteRaySinoStore, kSiteRaySinoLoad,
    kSiteColumnGather = 10, kSiteColumnScatter, kSiteColumnSinoStore, kSiteColumnSinoLoad,
    kSiteColumnLayoutIn, kSiteColumnLayoutOut,
    kSitePlaneGather = 20, kSitePlaneScatter, kSitePlaneSinoStore, kSitePlaneSinoLoad,
    kSitePlaneTile, kSitePlaneTileOut
};

#ifdef CTP_CHECK
struct CheckState {
    unsigned long long count;
    long long index, extent;
    int site, pad_;
};
__device__ CheckState ctp_check_state;

__device__ __forceinline__ bool ctp_in(long long i, long long n, int site)
{
    if (i >= 0 && i < n) return true;
    if (atomicAdd(&ctp_check_state.count, 1ull) == 0ull) {
        ctp_check_state.index = i;
        ctp_check_state.extent = n;
        ctp_check_state.site = site;
    }
    return false;
}
#else
__device__ __forceinline__ constexpr bool ctp_in(long long, long long, int) { return true; }
#endif

// The (t, s, e) offsets of pixel (iu, iv) of view `view` (curved detectors).
__host__ __device__ __forceinline__ const float *pixel_offsets_of(const RayParams &P, int view,
                                                                 int iu, int iv)
{
    const long long pix = (long long)iv * P.n_u + iu;
    return P.offsets + 3 * (P.offsets_per_view ? (long long)view * P.n_u * P.n_v + pix : pix);
}

// Elements of the sinogram buffer (n_views, n_v, n_u).
__host__ __device__ __forceinline__ long long sino_cells(const RayParams &P)
{
    return (long long)P.n_views * P.n_v * P.n_u;
}

}  // namespace ctp
