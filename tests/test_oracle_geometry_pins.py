"""Pins of the oracle's geometry gradients (``oracle.geometry_vjp``) against
things other than itself: central finite differences of the float64 forward
projection, and the invariance of a chord under sliding the ray's end points
along the ray.

First-order source / centre / axis gradients of the projector are a feature of
the pages (diffct 2.4.1 -> 2.4.2, docs/video/README.md, shot "Geometry";
diffct 2.1.0 -> 2.2.1, README "Arbitrary trajectories": trajectory tensors
that require gradients receive geometry gradients).
"""

import numpy as np
import pytest

from geom_helpers import random_frames


def _scan(oracle, beam, frames, n_u, n_v, pu, pv, shape, spacing, ou=0.0, ov=0.0):
    D, H, W = shape
    dz, dy, dx = spacing
    origin = (-0.5 * W * dx, -0.5 * H * dy, -0.5 * D * dz)
    return oracle.Scan(beam, *frames, n_u, n_v, pu, pv, shape, spacing, origin, ou, ov)


@pytest.mark.parametrize("beam", ["divergent", "parallel"])
def test_geometry_vjp_matches_central_differences(oracle_mod, beam):
    rng = np.random.default_rng(31 if beam == "divergent" else 32)
    frames = random_frames(rng, 3, beam, radius=3.0, det_dist=2.5, tilt=0.3)
    shape, spacing = (5, 6, 7), (0.21, 0.19, 0.23)
    scan = _scan(oracle_mod, beam, frames, 11, 9, 0.25, 0.22, shape, spacing, 0.3, -0.2)
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    w = rng.standard_normal(scan.n_rays).astype(np.float32)
    g = oracle_mod.geometry_vjp(scan, vol, w)
    h = 2.0 ** -18   # exact on float32 frame values below 4
    worst = 0.0
    for view in range(scan.n_views):
        for part in range(4):
            for ax in range(3):
                vals = []
                for sgn in (1.0, -1.0):
                    fr = [a.copy() for a in scan.arrays]
                    fr[part][view, ax] = np.float32(fr[part][view, ax] + sgn * h)
                    sc = _scan(oracle_mod, beam, fr, 11, 9, 0.25, 0.22, shape, spacing, 0.3,
                               -0.2)
                    vals.append(float(np.dot(oracle_mod.forward(sc, vol).ravel(), w.astype(np.float64))))
                fd = (vals[0] - vals[1]) / (2 * h)
                worst = max(worst, abs(fd - g[view, part, ax]))
    assert worst <= 1e-5 * np.abs(g).max(), (worst, np.abs(g).max())


def test_sliding_end_points_along_the_ray_changes_nothing(oracle_mod):
    """One ray per view, both end points outside the volume: moving the source or
    the pixel along the ray leaves the chord sums unchanged, so the gradients
    are orthogonal to the ray direction."""
    rng = np.random.default_rng(33)
    src, cen, U, V = random_frames(rng, 6, "divergent", radius=4.0, det_dist=3.0, tilt=0.2)
    cen = cen + rng.uniform(-0.3, 0.3, cen.shape).astype(np.float32)
    scan = _scan(oracle_mod, "divergent", (src, cen, U, V), 1, 1, 1.0, 1.0, (6, 5, 7),
                 (0.2, 0.25, 0.18))
    vol = rng.uniform(0.0, 1.0, (6, 5, 7)).astype(np.float32)
    g = oracle_mod.geometry_vjp(scan, vol, np.ones(scan.n_rays, np.float32))
    r = cen.astype(np.float64) - src.astype(np.float64)
    r /= np.linalg.norm(r, axis=1, keepdims=True)
    scale = np.abs(g).max()
    assert scale > 0
    assert np.abs(np.einsum("ij,ij->i", g[:, 0], r)).max() <= 1e-9 * scale
    assert np.abs(np.einsum("ij,ij->i", g[:, 1], r)).max() <= 1e-9 * scale


def test_uniform_volume_gradient_is_the_box_chord_gradient(oracle_mod):
    """f = 1: p is the chord of the grid's box, whose gradient comes only from the
    entry and exit planes; checked by central differences of the closed-form
    chord (slab method), independent of the oracle's traversal."""
    rng = np.random.default_rng(34)
    src, cen, U, V = random_frames(rng, 4, "divergent", radius=4.0, det_dist=3.0, tilt=0.2)
    shape, spacing = (6, 5, 7), (0.2, 0.25, 0.18)
    scan = _scan(oracle_mod, "divergent", (src, cen, U, V), 3, 2, 0.3, 0.3, shape, spacing)
    g = oracle_mod.geometry_vjp(scan, np.ones(shape, np.float32), np.ones(scan.n_rays, np.float32))
    lo = np.array(scan.origin)
    hi = lo + np.array(shape[::-1]) * np.array(spacing[::-1])

    def chords(frames):
        s, c, u, v = (a.astype(np.float64) for a in frames)
        total = np.zeros(len(s))
        for iv in range(2):
            for iu in range(3):
                P = c + ((iu - 1.0) * 0.3) * u + ((iv - 0.5) * 0.3) * v
                r = P - s
                t0 = (lo[None, :] - s) / r
                t1 = (hi[None, :] - s) / r
                a0 = np.maximum(np.minimum(t0, t1).max(1), 0.0)
                a1 = np.minimum(np.maximum(t0, t1).min(1), 1.0)
                total += np.maximum(a1 - a0, 0.0) * np.linalg.norm(r, axis=1)
        return total

    h = 1e-6
    base = [a.astype(np.float64) for a in (src, cen, U, V)]
    for part in range(4):
        for ax in range(3):
            plus = [a.copy() for a in base]
            minus = [a.copy() for a in base]
            plus[part][:, ax] += h
            minus[part][:, ax] -= h
            fd = (chords(plus) - chords(minus)) / (2 * h)
            np.testing.assert_allclose(g[:, part, ax], fd, rtol=1e-6, atol=1e-7)


def test_kink_flags_on_hand_built_rays(oracle_mod):
    """Unit cells: a ray through the edge x = 1, y = 1 (the diagonal of the xy
    plane at z = 0.5) is a kink; the same ray shifted by 0.3 in y is not; a ray
    entering through the box edge x = 0, y = 0 is one too."""
    def scan_of(src, cen):
        z = np.float32
        fr = (np.array([src], z), np.array([cen], z), np.array([[0, 0, 1]], z),
              np.array([[1, -1, 0]], z) / np.float32(np.sqrt(2)))
        return oracle_mod.Scan("divergent", *fr, 1, 1, 1.0, 1.0, (3, 3, 3), (1.0, 1.0, 1.0),
                               (0.0, 0.0, 0.0))
    assert oracle_mod.kinks(scan_of((-1.0, -1.0, 0.5), (4.0, 4.0, 0.5))).all()
    assert not oracle_mod.kinks(scan_of((-1.0, -0.7, 0.5), (4.0, 4.3, 0.5))).any()
    assert oracle_mod.kinks(scan_of((-1.0, -1.0, 1.5), (4.0, 4.0, 1.5))).all()


def test_kink_flags_source_on_a_plane(oracle_mod):
    """A divergent ray starting inside the grid exactly on a plane is a kink;
    starting 0.25 cell off it is not."""
    def scan_of(src):
        z = np.float32
        fr = (np.array([src], z), np.array([[5.0, 1.3, 1.6]], z), np.array([[0, 1, 0]], z),
              np.array([[0, 0, 1]], z))
        return oracle_mod.Scan("divergent", *fr, 1, 1, 1.0, 1.0, (3, 3, 3), (1.0, 1.0, 1.0),
                               (0.0, 0.0, 0.0))
    assert oracle_mod.kinks(scan_of((1.0, 1.4, 1.55))).all()
    assert not oracle_mod.kinks(scan_of((1.25, 1.4, 1.55))).any()
