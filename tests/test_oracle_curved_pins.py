"""Pins of the oracle's curved-detector rays (per-pixel offsets; the pages'
surface composition: point = centre + tangent u + vertical v + depth n, diffct
2.4.1 -> 2.4.2, kernels/surface_geometry.py ``compose_surface``)."""

import numpy as np

from geom_helpers import chord, random_frames


def _flat_offsets(n_u, n_v, pu, pv, ou, ov):
    iu = (np.arange(n_u) - 0.5 * (n_u - 1) + ou) * pu
    iv = (np.arange(n_v) - 0.5 * (n_v - 1) + ov) * pv
    t, s = np.meshgrid(iu, iv)
    return np.stack([t, s, np.zeros_like(t)], -1).astype(np.float32)


def _cylinder_offsets(n_u, n_v, radius, dgamma, pv):
    """Pixels on a cylinder of the given radius around the source line: angle
    gamma per column, straight rows."""
    g = (np.arange(n_u) - 0.5 * (n_u - 1)) * dgamma
    s = (np.arange(n_v) - 0.5 * (n_v - 1)) * pv
    G, S = np.meshgrid(g, s)
    t = radius * np.sin(G)
    e = radius * (1.0 - np.cos(G))   # towards the source along the normal
    return np.stack([t, S, e], -1).astype(np.float32)


def test_flat_offsets_reproduce_the_pitch_grid(oracle_mod):
    rng = np.random.default_rng(71)
    frames = random_frames(rng, 3, "divergent", radius=30.0, det_dist=20.0, tilt=0.3)
    shape, spacing = (6, 7, 8), (1.1, 0.9, 1.2)
    origin = (-4.8, -3.15, -3.3)
    # dyadic pitches and offsets: the float32 offset table holds the grid exactly
    flat = oracle_mod.Scan("divergent", *frames, 13, 11, 1.25, 1.125, shape, spacing, origin,
                           0.5, -0.25)
    off = _flat_offsets(13, 11, 1.25, 1.125, 0.5, -0.25)
    curved = oracle_mod.Scan("divergent", *frames, 13, 11, 1.0, 1.0, shape, spacing, origin,
                             0.0, 0.0, 3, off)
    vol = rng.uniform(0, 1, shape).astype(np.float32)
    np.testing.assert_allclose(oracle_mod.forward(curved, vol), oracle_mod.forward(flat, vol),
                               rtol=1e-12, atol=1e-12)


def test_cylindrical_detector_box_chords(oracle_mod):
    """f = 1 on a sub-box: every ray's path sum is its chord through the sub-box,
    computed by clipping rays built here (normal from an SVD null space)."""
    rng = np.random.default_rng(72)
    src, cen, U, V = random_frames(rng, 4, "divergent", radius=25.0, det_dist=20.0, tilt=0.2)
    n_u, n_v = 15, 9
    off = _cylinder_offsets(n_u, n_v, 45.0, 0.03, 1.1)
    shape, spacing = (7, 8, 9), (1.0, 0.8, 1.2)
    origin = (-5.4, -3.2, -3.5)
    scan = oracle_mod.Scan("divergent", src, cen, U, V, n_u, n_v, 1.0, 1.0, shape, spacing,
                           origin, 0.0, 0.0, 3, off)
    vol = np.zeros(shape, np.float32)
    vol[1:6, 2:7, 1:8] = 1.0
    p = oracle_mod.forward(scan, vol).reshape(scan.sino_shape)
    lo = np.array(origin) + np.array([1, 2, 1]) * np.array(spacing[::-1])
    hi = np.array(origin) + np.array([8, 7, 6]) * np.array(spacing[::-1])
    for k in range(4):
        u, v = U[k].astype(np.float64), V[k].astype(np.float64)
        n = np.linalg.svd(np.stack([u, v]))[2][-1]
        if np.dot(np.cross(u, v), n) < 0:
            n = -n
        n /= np.linalg.norm(n)
        o = off.astype(np.float64).reshape(-1, 3)
        P = cen[k].astype(np.float64) + o[:, :1] * u + o[:, 1:2] * v + o[:, 2:3] * n
        S = np.repeat(src[k:k + 1].astype(np.float64), len(P), 0)
        want = chord(S, P - S, np.zeros(len(P)), np.ones(len(P)), lo, hi)
        np.testing.assert_allclose(p[k].ravel(), want, rtol=1e-11, atol=1e-11)
