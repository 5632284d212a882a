"""Pins of the oracle's curved-detector gradients against central finite
differences of its float64 forward projection.

* ``geometry_vjp`` on a curved detector: pixel = centre + t u + s v + e n with n
  the unit normal of (u, v), so the u and v gradients carry the normal's
  derivative (dn = (I - n n^T) d(u x v) / |u x v|).
* ``surface_vjp``: the gradient with respect to every pixel's offsets (t, s, e),
  shared by all views (the pages' curved detectors support first-order surface
  gradients: diffct 2.1.0 -> 2.2.1, README "Curved detectors"; the surface point
  centre + tangent u + vertical v + depth n: diffct 2.4.1 -> 2.4.2,
  kernels/surface_geometry.py ``compose_surface``), for flat detectors their
  pitch grid.
"""

import numpy as np
import pytest

from geom_helpers import random_frames

H = 2.0 ** -18   # exact on float32 values below 4 (perturbations of frames and offsets)


def _scan(oracle, beam, frames, n_u, n_v, shape, spacing, offsets=None, pu=0.25, pv=0.22,
          ou=0.0, ov=0.0):
    D, Hh, W = shape
    dz, dy, dx = spacing
    origin = (-0.5 * W * dx, -0.5 * Hh * dy, -0.5 * D * dz)
    return oracle.Scan(beam, *frames, n_u, n_v, pu, pv, shape, spacing, origin, ou, ov,
                       pixel_offsets=offsets)


def _curved_offsets(rng, n_u, n_v, pu, pv):
    """A bent detector: the pitch grid with jittered tangent / vertical offsets
    and depths of up to +-0.3 (all below 4 in magnitude)."""
    iu = np.arange(n_u) - 0.5 * (n_u - 1)
    iv = np.arange(n_v) - 0.5 * (n_v - 1)
    t = np.broadcast_to(iu[None, :] * pu, (n_v, n_u))
    s = np.broadcast_to(iv[:, None] * pv, (n_v, n_u))
    off = np.stack([t + rng.uniform(-0.03, 0.03, (n_v, n_u)),
                    s + rng.uniform(-0.03, 0.03, (n_v, n_u)),
                    0.3 * np.sin(0.7 * t) + rng.uniform(-0.05, 0.05, (n_v, n_u))], -1)
    return off.astype(np.float32)


def _weights(oracle, scan, rng):
    """N(0,1) ray weights, zero on rays within 1e-3 cell of a kink (a cell edge
    or corner, where the path sum has no derivative and a central difference
    of step 2^-18 straddles the jump)."""
    w = rng.standard_normal(scan.n_rays).astype(np.float32)
    return np.where(oracle.kinks(scan, tol=1e-3).ravel(), np.float32(0), w)


def _objective(oracle, scan, vol, w):
    return float(np.dot(oracle.forward(scan, vol).ravel(), w.astype(np.float64)))


@pytest.mark.parametrize("beam", ["divergent", "parallel"])
def test_curved_geometry_vjp_matches_central_differences(oracle_mod, beam):
    rng = np.random.default_rng(81 if beam == "divergent" else 82)
    src, cen, U, V = random_frames(rng, 2, beam, radius=3.0, det_dist=2.5, tilt=0.3)
    # axes neither unit nor orthogonal (|u x v| = 1.35): every factor of the
    # normal's derivative shows
    U2 = (1.5 * U).astype(np.float32)
    V2 = (0.9 * V + 0.3 * U2).astype(np.float32)
    frames = (src, cen, U2, V2)
    shape, spacing = (5, 6, 7), (0.21, 0.19, 0.23)
    n_u, n_v = 9, 7
    off = _curved_offsets(rng, n_u, n_v, 0.25, 0.22)
    scan = _scan(oracle_mod, beam, frames, n_u, n_v, shape, spacing, off)
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    w = _weights(oracle_mod, scan, rng)
    g = oracle_mod.geometry_vjp(scan, vol, w)
    worst = 0.0
    for view in range(scan.n_views):
        for part in range(4):
            for ax in range(3):
                vals = []
                for sgn in (1.0, -1.0):
                    fr = [a.copy() for a in scan.arrays]
                    fr[part][view, ax] = np.float32(fr[part][view, ax] + sgn * H)
                    sc = _scan(oracle_mod, beam, fr, n_u, n_v, shape, spacing, off)
                    vals.append(_objective(oracle_mod, sc, vol, w))
                fd = (vals[0] - vals[1]) / (2 * H)
                worst = max(worst, abs(fd - g[view, part, ax]))
    assert worst <= 1e-5 * np.abs(g).max(), (worst, np.abs(g).max())
    # the normal's derivative matters here: the u / v gradients differ from the
    # pitch-grid chain (t, s times d p / d pixel alone)
    assert np.abs(g[:, 2:]).max() > 0


@pytest.mark.parametrize("beam", ["divergent", "parallel"])
@pytest.mark.parametrize("curved", [True, False])
def test_surface_vjp_matches_central_differences(oracle_mod, beam, curved):
    rng = np.random.default_rng(83 + 2 * int(curved) + (beam == "parallel"))
    frames = random_frames(rng, 3, beam, radius=3.0, det_dist=2.5, tilt=0.3)
    shape, spacing = (5, 6, 7), (0.21, 0.19, 0.23)
    n_u, n_v, pu, pv = 8, 6, 0.25, 0.1875   # dyadic: the pitch grid is exact as float32 offsets
    off = _curved_offsets(rng, n_u, n_v, pu, pv) if curved else None
    scan = _scan(oracle_mod, beam, frames, n_u, n_v, shape, spacing, off, pu, pv)
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    w = _weights(oracle_mod, scan, rng)
    g = oracle_mod.surface_vjp(scan, vol, w)
    assert g.shape == (n_v, n_u, 3)
    # the flat detector's pitch grid written out as offsets moves the same pixels
    base = off if curved else np.stack(np.broadcast_arrays(
        ((np.arange(n_u) - 0.5 * (n_u - 1)) * pu)[None, :],
        ((np.arange(n_v) - 0.5 * (n_v - 1)) * pv)[:, None],
        np.zeros((n_v, 1))), -1).astype(np.float32)
    if not curved:
        sc = _scan(oracle_mod, beam, frames, n_u, n_v, shape, spacing, base, pu, pv)
        np.testing.assert_allclose(oracle_mod.surface_vjp(sc, vol, w), g, rtol=1e-12,
                                   atol=1e-12 * np.abs(g).max())
    worst = 0.0
    for iv in range(n_v):
        for iu in range(n_u):
            for m in range(3):
                vals = []
                for sgn in (1.0, -1.0):
                    o2 = base.copy()
                    o2[iv, iu, m] = np.float32(o2[iv, iu, m] + sgn * H)
                    sc = _scan(oracle_mod, beam, frames, n_u, n_v, shape, spacing, o2, pu, pv)
                    vals.append(_objective(oracle_mod, sc, vol, w))
                fd = (vals[0] - vals[1]) / (2 * H)
                worst = max(worst, abs(fd - g[iv, iu, m]))
    assert worst <= 1e-5 * np.abs(g).max(), (worst, np.abs(g).max())


def test_flat_detector_as_offsets_gives_the_same_geometry_vjp(oracle_mod):
    """The pitch grid written as explicit offsets (depth 0) is the same detector:
    the frame gradients agree (the normal's derivative then vanishes with e)."""
    rng = np.random.default_rng(87)
    frames = random_frames(rng, 4, "divergent", radius=3.0, det_dist=2.5, tilt=0.3)
    shape, spacing = (6, 5, 7), (0.2, 0.22, 0.19)
    n_u, n_v, pu, pv = 10, 8, 0.25, 0.1875  # dyadic: the pitch grid is exact as float32 offsets
    off = np.stack(np.broadcast_arrays(((np.arange(n_u) - 4.5) * pu)[None, :],
                                       ((np.arange(n_v) - 3.5) * pv)[:, None],
                                       np.zeros((n_v, 1))), -1).astype(np.float32)
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    flat = _scan(oracle_mod, "divergent", frames, n_u, n_v, shape, spacing, None, pu, pv)
    curved = _scan(oracle_mod, "divergent", frames, n_u, n_v, shape, spacing, off, pu, pv)
    w = rng.standard_normal(flat.n_rays).astype(np.float32)
    a = oracle_mod.geometry_vjp(flat, vol, w)
    b = oracle_mod.geometry_vjp(curved, vol, w)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-11 * np.abs(a).max())


# ------------------------------------------------------ one offset table per view
def _per_view_case(oracle, rng, beam="divergent", K=3, n_u=8, n_v=6):
    frames = random_frames(rng, K, beam, radius=3.0, det_dist=2.5, tilt=0.3)
    off = np.stack([_curved_offsets(rng, n_u, n_v, 0.25, 0.1875) for _ in range(K)])
    shape, spacing = (5, 6, 7), (0.21, 0.19, 0.23)
    scan = _scan(oracle, beam, frames, n_u, n_v, shape, spacing, off, 0.25, 0.1875)
    return frames, off, shape, spacing, scan


def test_per_view_offsets_are_the_views_own_detectors(oracle_mod):
    """A table per view (the pages sample surfaces in view batches): every view
    projects as a one-view scan with that view's table would, and identical
    tables reproduce the shared-table scan."""
    rng = np.random.default_rng(88)
    frames, off, shape, spacing, scan = _per_view_case(oracle_mod, rng)
    assert scan.offsets_per_view
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    p = oracle_mod.forward(scan, vol)
    for k in range(scan.n_views):
        one = _scan(oracle_mod, "divergent", [f[k:k + 1] for f in frames], 8, 6, shape, spacing,
                    off[k], 0.25, 0.1875)
        np.testing.assert_array_equal(p[k], oracle_mod.forward(one, vol)[0])
    same = np.repeat(off[:1], scan.n_views, axis=0)
    a = oracle_mod.forward(_scan(oracle_mod, "divergent", frames, 8, 6, shape, spacing, same,
                                 0.25, 0.1875), vol)
    b = oracle_mod.forward(_scan(oracle_mod, "divergent", frames, 8, 6, shape, spacing, off[0],
                                 0.25, 0.1875), vol)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("beam", ["divergent", "parallel"])
def test_per_view_surface_vjp_matches_central_differences(oracle_mod, beam):
    rng = np.random.default_rng(89 if beam == "divergent" else 90)
    frames, off, shape, spacing, scan = _per_view_case(oracle_mod, rng, beam)
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    w = _weights(oracle_mod, scan, rng)
    g = oracle_mod.surface_vjp(scan, vol, w)
    assert g.shape == (scan.n_views, 6, 8, 3)
    worst = 0.0
    for k in range(scan.n_views):
        for iv in range(6):
            for iu in range(8):
                for m in range(3):
                    vals = []
                    for sgn in (1.0, -1.0):
                        o2 = off.copy()
                        o2[k, iv, iu, m] = np.float32(o2[k, iv, iu, m] + sgn * H)
                        sc = _scan(oracle_mod, beam, frames, 8, 6, shape, spacing, o2, 0.25,
                                   0.1875)
                        vals.append(_objective(oracle_mod, sc, vol, w))
                    fd = (vals[0] - vals[1]) / (2 * H)
                    worst = max(worst, abs(fd - g[k, iv, iu, m]))
    assert worst <= 1e-5 * np.abs(g).max(), (worst, np.abs(g).max())
    # summed over views it is the gradient of a table shared by all views
    shared = _scan(oracle_mod, beam, frames, 8, 6, shape, spacing, off[0], 0.25, 0.1875)
    per = _scan(oracle_mod, beam, frames, 8, 6, shape, spacing,
                np.repeat(off[:1], scan.n_views, axis=0), 0.25, 0.1875)
    w2 = _weights(oracle_mod, shared, rng)
    np.testing.assert_allclose(oracle_mod.surface_vjp(per, vol, w2).sum(0),
                               oracle_mod.surface_vjp(shared, vol, w2), rtol=1e-12, atol=1e-12)


def test_per_view_geometry_vjp_matches_central_differences(oracle_mod):
    rng = np.random.default_rng(91)
    frames, off, shape, spacing, scan = _per_view_case(oracle_mod, rng, K=2)
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    w = _weights(oracle_mod, scan, rng)
    g = oracle_mod.geometry_vjp(scan, vol, w)
    worst = 0.0
    for view in range(scan.n_views):
        for part in range(4):
            for ax in range(3):
                vals = []
                for sgn in (1.0, -1.0):
                    fr = [a.copy() for a in scan.arrays]
                    fr[part][view, ax] = np.float32(fr[part][view, ax] + sgn * H)
                    sc = _scan(oracle_mod, "divergent", fr, 8, 6, shape, spacing, off, 0.25,
                               0.1875)
                    vals.append(_objective(oracle_mod, sc, vol, w))
                fd = (vals[0] - vals[1]) / (2 * H)
                worst = max(worst, abs(fd - g[view, part, ax]))
    assert worst <= 1e-5 * np.abs(g).max(), (worst, np.abs(g).max())
