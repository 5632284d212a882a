/*
 * ctp.h -- C ABI of the B300 (sm_103a) ray-driven Siddon projector pair.
 *
 * The library computes, for every detector ray R of a scan and a volume f of
 * axis-aligned constant cells,
 *
 *     forward    p(R)    = sum over cells c of |R n c| * f(c)
 *     backward   g(c)    = sum over rays  R of |R n c| * y(R)
 *
 * where |R n c| is the physical length of the ray inside the cell.  The two
 * are an exact adjoint pair of the cell-constant Siddon model ("Matched
 * operators", diffct README, release diff 2.1.0 -> 2.2.1; "Siddon path sum;
 * matched adjoint", docs/video/README.md, release diff 2.4.1 -> 2.4.2), with
 * per-axis voxel spacing in physical length units (diffct CHANGELOG 2.4.4,
 * "Added": native per-axis voxel spacing).
 *
 * Conventions (all calls):
 *   - World axes x, y, z.  Volume buffers are float32, C-contiguous with shape
 *     (nz, ny, nx): x fastest ("(D, H, W)" tensor order).  Cell (i, j, k)
 *     covers [o + i d, o + (i+1) d) per axis, o = (ox, oy, oz).
 *   - Sinogram buffers are float32, C-contiguous (n_views, n_v, n_u): u fastest.
 *   - Detector pixel (iu, iv) of view s sits at
 *         det_centre[s] + (iu - (n_u-1)/2 + offset_u) * pitch_u * det_u[s]
 *                       + (iv - (n_v-1)/2 + offset_v) * pitch_v * det_v[s].
 *     Divergent beams (fan in 2-D, cone in 3-D): the ray is the segment from
 *     src[s] to the pixel.  Parallel beams: src[s] is the ray direction and the
 *     ray is the whole line through the pixel.  Each view has its own frame
 *     (per-view trajectory tuple, diffct README "Arbitrary trajectories").
 *   - A ray lying exactly in a cell-face plane counts in the cell on the + side.
 *   - 2-D scans are 3-D scans with nz = 1 and n_v = 1.
 *
 * Ownership: the caller owns every volume / sinogram buffer (device pointers
 * unless a name says _host); the library never frees or keeps them ("caller-owned
 * float32 buffers", diffct release diff 2.4.1 -> 2.4.2, kernels/surface_geometry.py
 * docstring; project_into / backproject_into, CHANGELOG 2.2.0).  A plan owns its
 * copy of the geometry and its device tables and scratch.  Calls are asynchronous
 * on the given stream unless stated; a NULL stream is the legacy default stream.
 *
 * Errors: every entry point returns a ctp_status; no C++ exception crosses the
 * ABI.  Validation happens on the host in ctp_plan before any device work
 * (validation errors surface before numerical work, CHANGELOG 2.4.0 "Fixed").
 */
#ifndef CTP_H
#define CTP_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ctp_status {
    CTP_OK = 0,
    CTP_E_NULL = 1,        /* a required pointer is NULL */
    CTP_E_SHAPE = 2,       /* sizes out of range (see ctp_plan) */
    CTP_E_NONFINITE = 3,   /* a frame vector, pitch, offset, spacing or origin is not finite */
    CTP_E_COINCIDENT = 4,  /* source and detector must differ (or parallel ray along the detector) */
    CTP_E_NEAR = 5,        /* frame coordinates beyond 1e6 voxel widths of the volume */
    CTP_E_FAR = 6,         /* frame coordinates beyond 1e15 in magnitude */
    CTP_E_SPACING = 7,     /* spacing outside [1e-6, 1e6] or max/min ratio above 1e4 */
    CTP_E_AXES = 8,        /* detector axes zero or parallel; parallel ray direction zero */
    CTP_E_CUDA = 9,        /* a CUDA runtime call failed */
    CTP_E_DEVICE = 10,     /* called with a different current device than the plan's */
    CTP_E_OPTION = 11,     /* unknown beam / ndim / path value or plan option */
    CTP_E_LIMIT = 12,      /* request beyond a fixed size limit of this entry point */
    CTP_E_GEOMETRY = 13    /* scan outside the analytical operators' class (see ctp_fdk) */
} ctp_status;

typedef enum ctp_beam { CTP_PARALLEL = 0, CTP_DIVERGENT = 1 } ctp_beam;

/* Traversal path.  AUTO picks PLANE for 2-D scans (rays in the slice plane),
 * COLUMN for 3-D scans whose detector v axis is exactly +-z in every view (then
 * all rays of a detector column share one xy trace; curved detectors qualify
 * when their columns are straight, see pixel_offsets), else RAY; it falls back
 * to RAY when a scan does not meet PLANE's or COLUMN's conditions (rays leaving
 * the slice; rows crossing more than one z plane per slab).  An explicit PLANE
 * or COLUMN request for a scan outside its class returns CTP_E_OPTION.  All
 * paths compute the same operator; they differ in work layout only. */
typedef enum ctp_path {
    CTP_PATH_AUTO = 0,
    CTP_PATH_RAY = 1,
    CTP_PATH_COLUMN = 2,
    CTP_PATH_PLANE = 3
} ctp_path;

typedef struct ctp_geometry {
    int ndim;                 /* 2 or 3 */
    int beam;                 /* ctp_beam */
    int n_views, n_u, n_v;    /* n_v = 1 for 2-D; n_views may be 0 (empty scan) */
    const float *src;         /* HOST (n_views, 3): source, or unit ray direction (PARALLEL) */
    const float *det_centre;  /* HOST (n_views, 3) */
    const float *det_u;       /* HOST (n_views, 3) unit u axis */
    const float *det_v;       /* HOST (n_views, 3) unit v axis (2-D: any vector not along u) */
    double pitch_u, pitch_v;  /* detector pitch (physical units) */
    double offset_u, offset_v;/* detector-centre offset in pixels */
    const float *pixel_offsets; /* NULL: flat detector (the pitch grid above).  Else a
                                 curved detector: HOST (n_v, n_u, 3) per-pixel (t, s, e),
                                 shared by all views: pixel (iu, iv) of view k sits at
                                 det_centre + t det_u + s det_v + e n, n = the unit
                                 normal (det_u x det_v) / |det_u x det_v| (the pages'
                                 surface composition: point = centre + tangent u +
                                 vertical v + depth n, release diff 2.4.1 -> 2.4.2,
                                 kernels/surface_geometry.py compose_surface); pitches
                                 and offsets are then unused.  3-D scans whose every
                                 view has det_v = +-z and whose columns are straight
                                 (t and e the same in every row, s affine in the row
                                 to 1e-6 of the column's span: cylindrical detectors)
                                 may take the column path; others take the ray path;
                                 the plane path is refused.  ctp_forward_static and
                                 the analytical operators refuse curved detectors
                                 (CTP_E_OPTION / CTP_E_GEOMETRY); ctp_geometry_vjp
                                 and ctp_surface_vjp take them.
                                 Offsets must be finite (CTP_E_NONFINITE). */
    int offsets_per_view;     /* 0: pixel_offsets is one (n_v, n_u, 3) table shared by
                                 all views; 1: one table per view, (n_views, n_v, n_u,
                                 3) (the pages sample surfaces in view and pixel
                                 batches: each view may see its own surface).  With
                                 per-view tables the column path needs every view's
                                 columns straight.  Other values: CTP_E_OPTION. */
} ctp_geometry;

typedef struct ctp_volume {
    int nx, ny, nz;           /* cells; nz = 1 for 2-D */
    double dx, dy, dz;        /* spacing; each in [1e-6, 1e6], max/min <= 1e4 */
    double ox, oy, oz;        /* world position of the min corner of cell (0, 0, 0);
                                 a centred volume has o = -n * d / 2 */
} ctp_volume;

typedef struct ctp_plan ctp_plan_t;

/*
 * Work-layout options of a plan.  None changes what the operators compute;
 * they select among work layouts that compute the same operator (used to test
 * each layout and to measure them against each other).  Zero in every field
 * (or a NULL pointer to ctp_plan_ex) is the measured default.
 *   rows_forward, rows_backward  column path: detector rows per thread of the
 *                 forward walk / of the backward walk and the segment counter,
 *                 1 to 4 (0: 4 and 2, halved on detectors under 96 / 48 rows).
 *   backward_rows_adjacent  column path with 2 rows per backward thread: 1 =
 *                 each reduction instruction covers 32 adjacent rows; 0 = a
 *                 thread's two rows are interleaved across lanes (default).
 *   plane_backward  plane path: 0 = by scan size (shared-memory tiles in view
 *                 groups up to 65536 rays, else privatised global reductions);
 *                 1 = always tiled; 2 = always privatised.
 *   host_chunks   host-buffer calls: number of view chunks the walk and the
 *                 sinogram copies are pipelined in, 1 to 64 (0: one per 64 MiB
 *                 of sinogram, at most 8); never more than the views.
 *   geometry_walk ctp_geometry_vjp on column-path plans: 0 = the column walk,
 *                 1 = the ray walk (other plans always take the ray walk).
 *   forward_ahead column path: the forward loads each row's next cell one slab
 *                 ahead in the slabs where its warp is inside the grid; 0 = when
 *                 its blocks run columns first (forward_views_first) and the
 *                 padded working copy is larger than the device's L2, 1 =
 *                 never, 2 = always.
 *   forward_views_first  column path: the blocks of the forward (and of the
 *                 column geometry walk) run views before detector columns (the
 *                 resident blocks then hold few columns at many angles, a thin
 *                 shell of the volume); 0 = when every view's source and
 *                 detector centre lie at one height (circular scans), 1 =
 *                 never, 2 = always.
 * Values outside these ranges make ctp_plan_ex return CTP_E_OPTION.
 */
typedef struct ctp_plan_options {
    int rows_forward;
    int rows_backward;
    int backward_rows_adjacent;
    int plane_backward;
    int host_chunks;
    int geometry_walk;
    int forward_ahead;
    int forward_views_first;
} ctp_plan_options;

typedef struct ctp_plan_info {
    int path;                         /* ctp_path actually used */
    int device;                       /* CUDA device the plan lives on */
    long long n_rays;                 /* n_views * n_v * n_u */
    long long n_cells;                /* nx * ny * nz */
    unsigned long long device_bytes;  /* device memory owned by the plan */
} ctp_plan_info;

/*
 * ctp_plan -- validate a scan and build a plan on the current CUDA device.
 * geom, vol: host structs, read only during the call (all frame arrays are
 * copied).  path: a ctp_path.  *out receives the plan (NULL on error).
 * Limits: 1 <= nx, ny, nz <= 32768 with nx*ny*nz < 2^31; n_u, n_v >= 1,
 * n_views >= 0, n_views*n_v*n_u < 2^40, n_views <= 65535, ceil(n_v/4) <= 65535.
 * Errors: CTP_E_NULL, CTP_E_OPTION, CTP_E_SHAPE, CTP_E_NONFINITE, CTP_E_SPACING,
 * CTP_E_AXES, CTP_E_COINCIDENT, CTP_E_NEAR, CTP_E_FAR (the validation set of the
 * pages' tests: "finite", "must differ", "1e6", "1e15"), CTP_E_CUDA.
 * Synchronous: allocates and fills the plan's device tables.
 */
int ctp_plan(const ctp_geometry *geom, const ctp_volume *vol, int path, ctp_plan_t **out);

/* ctp_plan with work-layout options (host struct, read during the call; NULL =
 * all defaults, the same plan as ctp_plan).  Errors as ctp_plan, plus
 * CTP_E_OPTION for an option out of range. */
int ctp_plan_ex(const ctp_geometry *geom, const ctp_volume *vol, int path,
                const ctp_plan_options *options, ctp_plan_t **out);

/* Release a plan (NULL is ignored).  Synchronises the device before freeing. */
void ctp_destroy(ctp_plan_t *plan);

/* Plan facts; info is a host struct. */
int ctp_plan_info_get(const ctp_plan_t *plan, ctp_plan_info *info);

/*
 * ctp_forward -- p = A f.  vol_dev: device float32 (nz, ny, nx), read only.
 * sino_dev: device float32 (n_views, n_v, n_u), fully overwritten (rays that
 * miss the volume get 0).  stream: a cudaStream_t (NULL = default stream).
 * The two buffers must not overlap.  For a plan without rays both pointers may
 * be NULL (nothing is done).  The column and plane paths walk padded working
 * copies of the volume that the plan owns, so device calls on one plan must be
 * ordered (one stream, or events between streams); different plans are
 * independent.  Errors: CTP_E_NULL, CTP_E_DEVICE, CTP_E_CUDA.
 */
int ctp_forward(const ctp_plan_t *plan, const float *vol_dev, float *sino_dev, void *stream);

/*
 * ctp_backward -- g = A^T y.  sino_dev: device float32 (n_views, n_v, n_u), read
 * only.  vol_dev: device float32 (nz, ny, nx), fully overwritten (zeroed, then
 * accumulated with float32 atomics, so the summation order -- not the set of
 * terms -- varies between calls).  sino_dev may be NULL for a plan without
 * rays (vol_dev is then zeroed).  Errors as ctp_forward.
 */
int ctp_backward(const ctp_plan_t *plan, const float *sino_dev, float *vol_dev, void *stream);

/*
 * ctp_segment_count -- number of (ray, cell) pieces longer than 1e-5 of the
 * smallest cell width that the plan's traversal visits in one pass (the same for
 * forward and backward).  The threshold drops only the rounding-sized pieces of
 * rays that cross a cell edge or corner exactly.  *out is a host value; the call
 * waits for the stream.  Diagnostics and throughput units.
 */
int ctp_segment_count(const ctp_plan_t *plan, unsigned long long *out, void *stream);

/*
 * Host-buffer variants (end-to-end): copy the input from host memory, run the
 * operator, copy the result back, and return once the result is in host memory.
 * Results equal the device calls' (the forward bit for bit, the backward up to
 * its atomics' summation order).  Host buffers may be pageable or pinned; with
 * pinned buffers the sinogram transfer overlaps the walk: the walk runs in view
 * chunks on `stream` (one chunk per 64 MiB of sinogram, at most 8; the plan
 * option host_chunks overrides) and each chunk's
 * sinogram rows move on a second stream owned by the plan -- down as soon as the
 * chunk is walked (forward), up just before it is walked (backward).  The
 * volume moves on `stream`.  The plan allocates one device volume, one device
 * sinogram, the copy stream and its events on the first host-buffer call and
 * reuses them; these calls cannot be captured into a CUDA graph.  Calls on one
 * plan must not run concurrently.  Errors as ctp_forward; after an error the
 * call has waited for every copy it queued.
 */
int ctp_forward_host(ctp_plan_t *plan, const float *vol_host, float *sino_host, void *stream);
int ctp_backward_host(ctp_plan_t *plan, const float *sino_host, float *vol_host, void *stream);

/*
 * ctp_forward_static -- p = A f without any allocation, for callers that may not
 * allocate device memory while they run: applications whose device memory is
 * owned by their own pool allocator (a raw cudaMalloc would bypass the pool's
 * budget and can fail once the pool has reserved the rest), and loops that must
 * not take the implicit device synchronisation of cudaMalloc / cudaFree.  The
 * pages have no counterpart; the result equals ctp_forward of a RAY-path plan
 * of the same scan (the per-view frames come from the same host function).
 * geom, vol: host structs as for ctp_plan (validated the same way, same error
 * codes).  vol_dev / sino_dev: device float32 buffers as for ctp_forward (may be
 * NULL when n_views is 0), on the current device.  stream: a cudaStream_t
 * (NULL = default stream).
 * Scratch: the per-view frame table lives in a fixed device array of
 * 4096 views (480 KiB) that every device loading the library holds until exit;
 * n_views above 4096 returns CTP_E_LIMIT, and so does a current device ordinal
 * of 64 or more.  The first call on a device (and the first after its context
 * was reset and recreated) looks the array's device address up
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * The frames are converted on the host into a buffer on the call's stack and
 * copied with cudaMemcpyAsync from that pageable memory: the copy may make the
 * host wait for the stream's earlier work, and the call returns only once the
 * frames have left the buffer.  Every call rewrites the frames it uses and
 * reads nothing left by earlier calls; calls that overlap on the GPU (other
 * streams, other host threads) share the array and race.  Calls no
 * cudaMalloc / cudaFree.
 */
int ctp_forward_static(const ctp_geometry *geom, const ctp_volume *vol, const float *vol_dev,
                       float *sino_dev, void *stream);

/*
 * Analytical FBP / FDK operators on the plan's geometry (diffct release diff
 * 2.1.0 -> 2.2.1, README "Analytical helpers" and "Differentiable FBP and FDK";
 * diffct/analytical.py: voxel-driven weighted gathers with the analytical
 * constant 1/(2 pi) or SDD/(2 pi SID), and their dedicated transposes; the
 * per-view SDD/(2 pi SID) of release diff 2.4.3 -> 2.4.4).  The pages give the
 * structure and the constants; the rest is the textbook flat-detector FBP:
 *
 *   isocentre  the volume centre; n_s the unit detector normal pointing away
 *              from the source (parallel: along the rays); SDD_s = (c_s - a_s).n_s,
 *              SID_s = (iso - a_s).n_s, a_s = src[s], c_s = det_centre[s].
 *   ramp       q[s,iv,i] = post * pitch_u * sum_j h[i-j] * pre * p[s,iv,j] along u,
 *              h the inverse transform of |omega| (radians per unit length) times
 *              a window (ctp_ramp: none = Ram-Lak, sinc = Shepp-Logan, cosine,
 *              Hamming, Hann; the pages' list of ramp filters), tau = pitch_u.
 *              Forward: pre = SDD_s / |pixel - a_s| (cosine weight; parallel 1),
 *              post = view_weight[s].  Transpose: pre and post swapped.
 *   gather     g(x) = sum_s k_s (SID_s / U_s(x))^2 I(q_s; u_s(x), v_s(x)): x the
 *              voxel centre, (u_s, v_s) the pixel coordinates where the ray from
 *              the source through x (parallel: along the rays) meets the detector
 *              plane (the inverse of the pixel-centre convention above), U_s(x) =
 *              (x - a_s).n_s the depth, I bilinear interpolation with zeros
 *              outside the detector (2-D: linear along u), k_s = SDD_s/(2 pi SID_s)
 *              (parallel: 1/(2 pi), weight 1).  Voxels at or behind a source get
 *              nothing from that view.
 *   transpose  the exact transpose of the gather (same stencil, float atomics).
 *
 * With view weights pi / n_views (a full 2 pi scan: half the angular step),
 * ctp_fdk reconstructs the image whose line integrals are the sinogram.
 *
 * Supported scans: every 2-D scan, and 3-D scans whose every view has the
 * detector v axis along +-z and the u axis horizontal (circular and helical cone
 * or parallel beams), with each divergent view's isocentre in front of its source;
 * others return CTP_E_GEOMETRY from these calls (the plan itself is still valid for
 * the projector pair).  ctp_ramp_filter needs n_u <= 16384 (else CTP_E_LIMIT).
 *
 * Buffers: device float32, layouts as above; view_weight_dev: device float32
 * (n_views), or NULL for all ones; pixel_weight_dev: device float32 (n_views,
 * n_u), or NULL for all ones, multiplied into the forward filter's pre-weight
 * (and the transpose's post-weight) -- e.g. ctp_parker_weights.  ramp: a ctp_ramp.
 * transpose: 0 or 1.  ctp_ramp_filter may run in place (out_dev == sino_dev).
 * ctp_weighted_backproject overwrites vol_dev; ctp_weighted_backproject_transpose
 * overwrites sino_dev (zeroed, then accumulated with float atomics).  ctp_fdk =
 * ramp filter of sino_dev into work_dev (n_views, n_v, n_u floats; may equal
 * sino_dev, which is then overwritten) followed by the gather into vol_dev.
 * Errors: CTP_E_NULL, CTP_E_DEVICE, CTP_E_OPTION (unknown ramp), CTP_E_GEOMETRY,
 * CTP_E_LIMIT, CTP_E_CUDA.  All are asynchronous on `stream`.
 */
typedef enum ctp_ramp {
    CTP_RAMLAK = 0,       /* |omega| */
    CTP_SHEPP_LOGAN = 1,  /* (2 / tau) |sin(omega tau / 2)| */
    CTP_COSINE = 2,       /* |omega| cos(omega tau / 2) */
    CTP_HAMMING = 3,      /* |omega| (0.54 + 0.46 cos(omega tau)) */
    CTP_HANN = 4          /* |omega| (1 + cos(omega tau)) / 2 */
} ctp_ramp;

int ctp_ramp_filter(const ctp_plan_t *plan, const float *sino_dev, float *out_dev,
                    const float *view_weight_dev, const float *pixel_weight_dev, int ramp,
                    int transpose, void *stream);
int ctp_weighted_backproject(const ctp_plan_t *plan, const float *sino_dev, float *vol_dev,
                             void *stream);
int ctp_weighted_backproject_transpose(const ctp_plan_t *plan, const float *vol_dev,
                                       float *sino_dev, void *stream);
int ctp_fdk(const ctp_plan_t *plan, const float *sino_dev, float *work_dev, float *vol_dev,
            const float *view_weight_dev, const float *pixel_weight_dev, int ramp, void *stream);

/*
 * ctp_parker_weights -- Parker's short-scan weights (the pages' analytical
 * helpers list Parker weights) of a circular divergent scan about the vertical
 * axis through the volume centre, for pixel_weight_dev of the calls above:
 * weight_dev[k][i] (device float32, n_views x n_u) = sin^2(pi/4 beta / (G - g))
 * for beta < 2 (G - g), sin^2(pi/4 (pi + 2 G - beta) / (G + g)) for
 * beta > pi - 2 g, 1 between and 0 outside [0, pi + 2 G]: beta = view k's source
 * azimuth from view 0 in the scan's turning sense, g = the signed fan angle of
 * column i (xy plane, central ray to the column's ray, in the turning sense),
 * G = the largest |g| of view 0.  A ray's and its conjugate's weights sum to
 * one; with them, view weights equal to the angular step (not half of it)
 * reconstruct a scan of pi + 2 G.  Computed on the host in float64 and copied;
 * the call waits for the copy.  Errors: CTP_E_NULL, CTP_E_DEVICE,
 * CTP_E_GEOMETRY (parallel beam or curved detector), CTP_E_CUDA.
 */
int ctp_parker_weights(const ctp_plan_t *plan, float *weight_dev, void *stream);

/*
 * ctp_geometry_vjp -- first-order geometry gradients of the projection
 * ("first-order source / centre / axis gradients", diffct release diff
 * 2.4.1 -> 2.4.2, docs/video/README.md; trajectory tensors that require
 * gradients receive geometry gradients, release diff 2.1.0 -> 2.2.1, README
 * "Arbitrary trajectories"):
 *
 *     grad[s][0..2]  = sum over rays R of view s of w[R] * dp(R)/d src[s]
 *     grad[s][3..5]  = ... d det_centre[s],   grad[s][6..8] = ... d det_u[s],
 *     grad[s][9..11] = ... d det_v[s]
 *
 * with p = A vol the path sums of the plan's scan.  For the line X0 + t r
 * (divergent: X0 = source, r = pixel - source, t in [0, 1]; parallel: X0 =
 * pixel, r = src) p = |r| sum_j (t_{j+1} - t_j) f_j; every crossing of a grid
 * plane x_a = const at t_k (value outside the grid 0; the ray's own end points
 * are not crossings) contributes -(f_before - f_after) |r| (dX0_a + t_k dr_a) / r_a,
 * and the length scale contributes p r.dr / |r|^2; pixel = centre + alpha u +
 * beta v (flat detectors: the pitch grid), or centre + t u + s v + e n with n =
 * u x v / |u x v| (curved detectors: the pixel's offsets), whose u and v
 * gradients also carry the normal's derivative: with g = dp/d pixel and h =
 * (g - (n.g) n) / |u x v|, dp/du = t g + e v x h and dp/dv = s g - e u x h.
 * The gradient of the backprojection <A^T y, h> with respect to the geometry is
 * the same call with vol = h and w = y.  Rays through a cell edge or corner are
 * kinks of p; the jump goes to one of the coincident crossings.
 * vol_dev: device float32 (nz, ny, nx).  weight_dev: device float32
 * (n_views, n_v, n_u).  grad_dev: device float64 (n_views, 12), overwritten.
 * Column-path plans of flat detectors run the sums over the column walk on the
 * plan's working copy of vol_dev (ordered with the plan's other calls, as
 * ctp_forward); other plans run the ray path's walk (the plan option
 * geometry_walk = 1 selects it for column plans too).  Asynchronous on
 * `stream`.  Errors: CTP_E_NULL, CTP_E_DEVICE, CTP_E_CUDA.
 */
int ctp_geometry_vjp(const ctp_plan_t *plan, const float *vol_dev, const float *weight_dev,
                     double *grad_dev, void *stream);

/*
 * ctp_surface_vjp -- first-order gradients with respect to the detector
 * surface: every pixel's offsets (t, s, e) along det_u, det_v and the unit
 * normal n = det_u x det_v / |det_u x det_v|, shared by all views (the pages'
 * curved detectors: "Projection and matched backprojection support first-order
 * surface gradients", diffct release diff 2.1.0 -> 2.2.1, README "Curved
 * detectors"; the point centre + tangent u + vertical v + depth n, release diff
 * 2.4.1 -> 2.4.2, kernels/surface_geometry.py compose_surface):
 *
 *     grad[iv][iu][m] = sum over views s of w[s][iv][iu] * (dp/d pixel) . (u_s, v_s, n_s)[m]
 *
 * with dp/d pixel the end-point derivative of ctp_geometry_vjp.  Flat detectors
 * are included: their offsets are the pitch grid (e = 0), and the result is the
 * gradient with respect to moving each pixel along the view's axes.
 * With one offset table per view (offsets_per_view = 1) every view's pixel has
 * its own gradient: grad_dev is (n_views, n_v, n_u, 3), no sum over views.
 * vol_dev: device float32 (nz, ny, nx); weight_dev: device float32 (n_views,
 * n_v, n_u); grad_dev: device float64 (n_v, n_u, 3), overwritten (every
 * pixel's sums are one thread's: deterministic, no atomics).  Runs the
 * ray path's walk on vol_dev on any plan.  Asynchronous on `stream`.  Errors:
 * CTP_E_NULL, CTP_E_DEVICE, CTP_E_CUDA.
 */
int ctp_surface_vjp(const ctp_plan_t *plan, const float *vol_dev, const float *weight_dev,
                    double *grad_dev, void *stream);

/*
 * ctp_check_violations -- the bounds-checked debug build (the library compiled
 * with -DCTP_CHECK, libctp_check.so) tests, before each access, the index of
 * every global load, store and reduction of the projector walks (ray, column
 * and plane paths, their sinogram reads and writes, the column path's layout
 * transposes), every shared-memory reduction of the tiled 2-D backward, the
 * weighted backprojection's and its transpose's loads, stores and reductions
 * and the geometry-gradient walks' loads and outputs against the buffer's
 * extent; an access outside is skipped and counted.  This
 * call waits for the device, returns the count since the previous call, the
 * first offending index, its buffer's extent and the access site (the CheckSite
 * values of the library's sources), and resets them.  All four pointers are
 * host outputs.  Errors: CTP_E_NULL; CTP_E_OPTION in normal builds (outputs
 * zeroed); CTP_E_CUDA.
 */
int ctp_check_violations(unsigned long long *count, long long *index, long long *extent,
                         int *site);

/* Static English text of a status code. */
const char *ctp_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* CTP_H */
