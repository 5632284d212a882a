"""Float64 oracle of the analytical FBP / FDK operators -- TEST INFRASTRUCTURE ONLY.

Same rules as the rest of ``oracle/``: only ``tests/``, the package's smoke check
and the benchmark's CPU legs may import it; it never loads the product library
and shares no code with it.  Plain numpy in float64 (the float32 frames are
promoted exactly), vectorised over voxels or pixels, one view at a time.

What the pages fix (diffct release pages, my.diffend.io):

* the analytical helpers: ramp filters (Ram-Lak, Shepp-Logan among them), fan /
  cone weights, and FBP / FDK backprojection (diffct 2.1.0 -> 2.2.1, README
  "Analytical helpers" / "Differentiable FBP and FDK");
* a voxel-driven weighted gather -- one thread per output voxel -- whose
  analytical constant is 1 / (2 pi) for parallel beams and SDD / (2 pi SID) for
  fan and cone beams, per view (diffct 2.1.0 -> 2.2.1, ``diffct/analytical.py``,
  ``_analytical_transpose_raw``; diffct 2.4.3 -> 2.4.4, ``diffct/analytical.py``,
  the per-view ``sdd_n / (2 pi sid_n)`` scale and the parallel gather's final
  ``1 / (2 pi)``);
* a dedicated transpose of that gather that moves the same interpolation
  stencil the other way ("Their backward kernels transpose the actual
  interpolation stencil", README "Differentiable FBP and FDK").

Readings where the pages are silent (the textbook fan / cone FBP with a flat
detector, written in physical detector units):

* isocentre = the volume centre; n = unit detector normal pointing away from the
  source (parallel: along the rays); SDD_k = (c_k - a_k).n_k,
  SID_k = (iso - a_k).n_k;
* pixel coordinates of a detector point P: u = (P - c).u* / pitch_u + (n_u-1)/2
  - offset_u, v likewise with v*, where (u*, v*) is the dual basis of the
  detector axes in the detector plane (the inverse of the pixel-centre formula
  the projector uses);
* gather: g(x) = sum_k s_k W_k(x) I(q_k; u_k(x), v_k(x)) with x the voxel centre,
  (u_k, v_k) where the source ray through x (parallel: the ray along the beam)
  meets the detector, W_k = (SID_k / U_k(x))^2 with depth U_k = (x - a_k).n_k
  (parallel: 1; voxels with U_k <= 0 get nothing from view k), s_k as above, and
  I the bilinear interpolation of view k's rows with zeros outside the detector
  (2-D scans: linear along u, v ignored);
* filter: q[k, iv, i] = w_k * tau * sum_j h[i - j] * cw[k, iv, j] * p[k, iv, j]
  with tau = pitch_u, cw = SDD_k / |P_pix - a_k| the cosine of the ray to the
  normal (parallel: 1), w_k caller-given view weights (full 2 pi scans: pi / K,
  i.e. half the angular step), and h the ramp kernel with frequency response
  |omega| in radians per unit length times a window (none: Ram-Lak; sinc:
  Shepp-Logan; cosine, Hamming, Hann).

With these, g = gather(filter(p)) is the textbook FBP / FDK estimate of the
image whose line integrals are p.  What pins it (``tests/test_oracle_fdk_pins.py``):
the kernels' frequency responses, exact reproduction of sinograms that are
linear in the pixel indices (with the projection point and depth computed by an
independent linear solve), the adjoint identity between the gather and the
separately written scatter, and reconstructions of discs and balls from their
closed-form line integrals.
"""

from __future__ import annotations

import math

import numpy as np

RAMLAK, SHEPP_LOGAN, COSINE, HAMMING, HANN = 0, 1, 2, 3, 4


def _frames(scan):
    return [a.astype(np.float64) for a in scan.arrays]


def view_geometry(scan):
    """Per-view float64 quantities: unit normal ``n``, dual axes ``us``/``vs``,
    ``sdd``, ``sid`` (divergent; zeros for parallel) and the scale ``s``."""
    a, c, u, v = _frames(scan)
    n = np.cross(u, v)
    n /= np.linalg.norm(n, axis=1, keepdims=True)
    if scan.beam == "divergent":
        side = np.einsum("ij,ij->i", c - a, n)
    else:
        side = np.einsum("ij,ij->i", a, n)
    n *= np.where(side < 0, -1.0, 1.0)[:, None]
    triple = np.einsum("ij,ij->i", np.cross(u, v), n)
    us = np.cross(v, n) / triple[:, None]
    vs = np.cross(n, u) / triple[:, None]
    if scan.beam == "divergent":
        iso = volume_centre(scan)
        sdd = np.einsum("ij,ij->i", c - a, n)
        sid = np.einsum("ij,ij->i", iso[None, :] - a, n)
        s = sdd / (2.0 * math.pi * sid)
    else:
        sdd = np.zeros(scan.n_views)
        sid = np.zeros(scan.n_views)
        s = np.full(scan.n_views, 1.0 / (2.0 * math.pi))
    return {"a": a, "c": c, "u": u, "v": v, "n": n, "us": us, "vs": vs, "sdd": sdd,
            "sid": sid, "s": s}


def volume_centre(scan):
    D, H, W = scan.shape
    dz, dy, dx = scan.spacing
    o = np.asarray(scan.origin, np.float64)
    return o + 0.5 * np.array([W * dx, H * dy, D * dz])


def voxel_centres(scan, voxels=None):
    """World (x, y, z) of voxel centres, shape (N, 3); ``voxels`` (N, 3) of (k, j, i)
    picks some (default: all, in (D, H, W) C order)."""
    D, H, W = scan.shape
    dz, dy, dx = scan.spacing
    ox, oy, oz = scan.origin
    if voxels is None:
        k, j, i = np.meshgrid(np.arange(D), np.arange(H), np.arange(W), indexing="ij")
        k, j, i = k.ravel(), j.ravel(), i.ravel()
    else:
        voxels = np.asarray(voxels).reshape(-1, 3)
        k, j, i = voxels[:, 0], voxels[:, 1], voxels[:, 2]
    return np.stack([ox + (i + 0.5) * dx, oy + (j + 0.5) * dy, oz + (k + 0.5) * dz], axis=1)


def project(scan, G, view, X):
    """Pixel coordinates (u, v) and weight W of points X (N, 3) in one view.
    Points behind the source (depth <= 0) get W = 0 and u = v = nan."""
    a, c, n = G["a"][view], G["c"][view], G["n"][view]
    if scan.beam == "divergent":
        d = X - a
        depth = d @ n
        ok = depth > 0
        t = np.where(ok, G["sdd"][view] / np.where(ok, depth, 1.0), np.nan)
        P = a + t[:, None] * d
        W = np.where(ok, (G["sid"][view] / np.where(ok, depth, 1.0)) ** 2, 0.0)
    else:
        r = a / np.linalg.norm(a)
        s = ((c - X) @ n) / (r @ n)
        P = X + s[:, None] * r
        W = np.ones(X.shape[0])
    rel = P - c
    u = rel @ G["us"][view] / scan.pitch_u + 0.5 * (scan.n_u - 1) - scan.offset_u
    if scan.ndim == 2:
        v = np.zeros_like(u)
    else:
        v = rel @ G["vs"][view] / scan.pitch_v + 0.5 * (scan.n_v - 1) - scan.offset_v
    return u, v, W


def _stencil(scan, u, v):
    """Bilinear stencil: list of (row, col, weight, valid) arrays; zero padding."""
    i0 = np.floor(np.nan_to_num(u, nan=-10.0)).astype(np.int64)
    fu = np.nan_to_num(u, nan=-10.0) - i0
    cols = [(i0, 1.0 - fu), (i0 + 1, fu)]
    if scan.ndim == 2:
        rows = [(np.zeros_like(i0), np.ones_like(fu))]
    else:
        j0 = np.floor(np.nan_to_num(v, nan=-10.0)).astype(np.int64)
        fv = np.nan_to_num(v, nan=-10.0) - j0
        rows = [(j0, 1.0 - fv), (j0 + 1, fv)]
    out = []
    for r, wr in rows:
        for col, wc in cols:
            ok = (r >= 0) & (r < scan.n_v) & (col >= 0) & (col < scan.n_u) & np.isfinite(u)
            out.append((np.where(ok, r, 0), np.where(ok, col, 0), wr * wc, ok))
    return out


def weighted_backproject(scan, q, voxels=None):
    """The gather g(x) = sum_k s_k W_k(x) I(q_k; u_k(x), v_k(x)), float64.
    Returns the whole volume (D, H, W), or values at ``voxels`` (N, 3) of (k, j, i)."""
    q = np.asarray(q, np.float64).reshape(scan.n_views, scan.n_v, scan.n_u)
    G = view_geometry(scan)
    X = voxel_centres(scan, voxels)
    g = np.zeros(X.shape[0])
    for k in range(scan.n_views):
        u, v, W = project(scan, G, k, X)
        val = np.zeros(X.shape[0])
        for r, col, w, ok in _stencil(scan, u, v):
            val += np.where(ok, w * q[k, r, col], 0.0)
        g += G["s"][k] * W * val
    return g.reshape(scan.shape) if voxels is None else g


def weighted_backproject_transpose(scan, vol):
    """The exact transpose of :func:`weighted_backproject`: every voxel's value,
    times s_k W_k, is scattered onto its bilinear stencil in each view."""
    vol = np.asarray(vol, np.float64).reshape(-1)
    G = view_geometry(scan)
    X = voxel_centres(scan)
    out = np.zeros((scan.n_views, scan.n_v, scan.n_u))
    for k in range(scan.n_views):
        u, v, W = project(scan, G, k, X)
        amount = G["s"][k] * W * vol
        for r, col, w, ok in _stencil(scan, u, v):
            np.add.at(out[k], (r[ok], col[ok]), (w * amount)[ok])
    return out


def _band_limited_ramp(x, tau):
    """g(x) = (1 / 2 pi) * integral over |omega| <= pi / tau of |omega| exp(i omega x tau),
    the band-limited ramp at a (possibly fractional) sample offset x."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    zero = x == 0
    xs = np.where(zero, 1.0, x)
    out[:] = (math.pi * np.sin(math.pi * xs) / xs + (np.cos(math.pi * xs) - 1.0) / xs ** 2) / (
        math.pi * tau * tau)
    out[zero] = math.pi / (2.0 * tau * tau)
    return out


def ramp_kernel(n_u, tau, kind=RAMLAK):
    """Spatial ramp kernel h[m], m = -(n_u-1) .. n_u-1 (index m + n_u - 1), in the
    convention where tau * sum_m h[m] exp(-i omega m tau) -> H(omega) for
    |omega| <= pi / tau, with H = |omega| times a window (the pages name Ram-Lak,
    Shepp-Logan, cosine, Hamming and Hann):
        Ram-Lak      |omega|
        Shepp-Logan  (2 / tau) |sin(omega tau / 2)|  = |omega| sinc
        cosine       |omega| cos(omega tau / 2)
        Hamming      |omega| (0.54 + 0.46 cos(omega tau))
        Hann         |omega| (1 + cos(omega tau)) / 2
    Each is the inverse transform of H: the band-limited ramp g at the sample
    offsets, or its half-sample / one-sample shifts for the cosine windows."""
    m = np.arange(-(n_u - 1), n_u, dtype=np.float64)
    g = lambda x: _band_limited_ramp(x, tau)  # noqa: E731
    if kind == RAMLAK:
        h = g(m)
    elif kind == SHEPP_LOGAN:
        h = -4.0 / (math.pi * tau * tau * (4.0 * m * m - 1.0))
    elif kind == COSINE:
        h = 0.5 * (g(m - 0.5) + g(m + 0.5))
    elif kind == HAMMING:
        h = 0.54 * g(m) + 0.23 * (g(m - 1.0) + g(m + 1.0))
    elif kind == HANN:
        h = 0.5 * g(m) + 0.25 * (g(m - 1.0) + g(m + 1.0))
    else:
        raise ValueError(f"unknown filter {kind}")
    return h


def cosine_weights(scan):
    """cw[k, iv, iu] = SDD_k / |P_pix - a_k| (divergent), 1 (parallel)."""
    shape = (scan.n_views, scan.n_v, scan.n_u)
    if scan.beam != "divergent":
        return np.ones(shape)
    G = view_geometry(scan)
    iu = np.arange(scan.n_u) - 0.5 * (scan.n_u - 1) + scan.offset_u
    iv = np.arange(scan.n_v) - 0.5 * (scan.n_v - 1) + scan.offset_v
    if scan.ndim == 2:
        iv = np.zeros_like(iv)
    out = np.empty(shape)
    for k in range(scan.n_views):
        P = (G["c"][k][None, None, :]
             + (iu * scan.pitch_u)[None, :, None] * G["u"][k][None, None, :]
             + (iv * scan.pitch_v)[:, None, None] * G["v"][k][None, None, :])
        out[k] = G["sdd"][k] / np.linalg.norm(P - G["a"][k], axis=2)
    return out


def _toeplitz(scan, kind):
    h = ramp_kernel(scan.n_u, scan.pitch_u, kind)
    idx = np.arange(scan.n_u)
    return h[(idx[:, None] - idx[None, :]) + scan.n_u - 1]   # T[i, j] = h[i - j]


def filter_sinogram(scan, p, view_weight=None, kind=RAMLAK):
    """q = w_k * tau * (h * (cw . p)) along u, float64, shape (n_views, n_v, n_u)."""
    p = np.asarray(p, np.float64).reshape(scan.n_views, scan.n_v, scan.n_u)
    w = np.ones(scan.n_views) if view_weight is None else np.asarray(view_weight, np.float64)
    T = _toeplitz(scan, kind)
    pw = cosine_weights(scan) * p
    q = scan.pitch_u * (pw @ T.T)
    return q * w[:, None, None]


def filter_sinogram_transpose(scan, q, view_weight=None, kind=RAMLAK):
    """Transpose of :func:`filter_sinogram`: cw . (tau * T^T (w_k q))."""
    q = np.asarray(q, np.float64).reshape(scan.n_views, scan.n_v, scan.n_u)
    w = np.ones(scan.n_views) if view_weight is None else np.asarray(view_weight, np.float64)
    T = _toeplitz(scan, kind)
    return cosine_weights(scan) * (scan.pitch_u * ((q * w[:, None, None]) @ T))


def parker(beta, gamma, big_gamma):
    """Parker's short-scan weight of the ray with scan angle beta in [0, pi + 2 Gamma]
    and signed fan angle gamma (counter-clockwise from the central ray, the scan
    turning counter-clockwise), half fan angle Gamma (Parker 1982, as the pages'
    "Parker weights"): the weights of a ray and of its conjugate
    (beta + pi + 2 gamma, -gamma) sum to one."""
    beta = np.asarray(beta, np.float64)
    gamma = np.asarray(gamma, np.float64)
    g = big_gamma
    w = np.ones(np.broadcast(beta, gamma).shape)
    lo = beta < 2 * (g - gamma)
    hi = beta > math.pi - 2 * gamma
    with np.errstate(divide="ignore", invalid="ignore"):
        w = np.where(lo, np.sin(0.25 * math.pi * beta / (g - gamma)) ** 2, w)
        w = np.where(hi, np.sin(0.25 * math.pi * (math.pi + 2 * g - beta) / (g + gamma)) ** 2, w)
    w = np.where((beta < 0) | (beta > math.pi + 2 * g), 0.0, w)
    return w


def scan_angles(scan):
    """Per view the scan angle beta (source azimuth about the vertical axis through
    the volume centre, from view 0 in the direction the scan turns), per view and
    detector column the signed fan angle gamma in the xy plane (from the central
    ray -- source to axis -- to the column's ray, counter-clockwise in the
    turning sense), and the half fan angle Gamma (largest |gamma| of view 0)."""
    a, c, u, v = _frames(scan)
    iso = volume_centre(scan)
    rel = a[:, :2] - iso[None, :2]
    az = np.unwrap(np.arctan2(rel[:, 1], rel[:, 0]))
    sense = 1.0 if scan.n_views < 2 or az[1] >= az[0] else -1.0
    beta = sense * (az - az[0])
    iu = (np.arange(scan.n_u) - 0.5 * (scan.n_u - 1) + scan.offset_u) * scan.pitch_u
    P = c[:, None, :] + iu[None, :, None] * u[:, None, :]
    d = (P - a[:, None, :])[:, :, :2]
    ctr = -rel[:, None, :] / np.linalg.norm(rel, axis=1)[:, None, None]
    cross = ctr[..., 0] * d[..., 1] - ctr[..., 1] * d[..., 0]
    dot = (ctr * d).sum(-1)
    gamma = sense * np.arctan2(cross, dot)
    return beta, gamma, float(np.abs(gamma[0]).max())


def parker_weights(scan):
    """(n_views, n_u) Parker weights of a circular short scan (see :func:`parker`)."""
    beta, gamma, big = scan_angles(scan)
    return parker(beta[:, None], gamma, big)


def filter_sinogram_pw(scan, p, view_weight=None, pixel_weight=None, kind=RAMLAK):
    """:func:`filter_sinogram` with per-(view, column) weights applied before the
    convolution (Parker weights, or any learned weights)."""
    p = np.asarray(p, np.float64).reshape(scan.n_views, scan.n_v, scan.n_u)
    if pixel_weight is not None:
        p = p * np.asarray(pixel_weight, np.float64)[:, None, :]
    return filter_sinogram(scan, p, view_weight, kind)


def fdk(scan, p, view_weight=None, kind=RAMLAK):
    """Filtered backprojection: weighted_backproject(filter_sinogram(p))."""
    return weighted_backproject(scan, filter_sinogram(scan, p, view_weight, kind))
