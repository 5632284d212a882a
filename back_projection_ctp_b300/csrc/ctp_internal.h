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
    const float *offsets; // curved detector: (n_v, n_u, 3) per-pixel offsets; else null
    const ColumnOffsets *columns;  // curved detector on the column path: per column; else null
};

}  // namespace ctp
