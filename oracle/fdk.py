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
  |omega| in radians per unit length (Ram-Lak) or |omega| |sinc| (Shepp-Logan).

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

RAMLAK, SHEPP_LOGAN = 0, 1


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


def ramp_kernel(n_u, tau, kind=RAMLAK):
    """Spatial ramp kernel h[m], m = -(n_u-1) .. n_u-1 (index m + n_u - 1), in the
    convention where tau * sum_m h[m] exp(-i omega m tau) -> |omega| (Ram-Lak) or
    (2 / tau) |sin(omega tau / 2)| (Shepp-Logan) for |omega| <= pi / tau."""
    m = np.arange(-(n_u - 1), n_u, dtype=np.float64)
    if kind == RAMLAK:
        h = np.zeros_like(m)
        h[m == 0] = math.pi / (2.0 * tau * tau)
        odd = (np.abs(m) % 2) == 1
        h[odd] = -2.0 / (math.pi * m[odd] ** 2 * tau * tau)
    elif kind == SHEPP_LOGAN:
        h = -4.0 / (math.pi * tau * tau * (4.0 * m * m - 1.0))
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


def fdk(scan, p, view_weight=None, kind=RAMLAK):
    """Filtered backprojection: weighted_backproject(filter_sinogram(p))."""
    return weighted_backproject(scan, filter_sinogram(scan, p, view_weight, kind))
