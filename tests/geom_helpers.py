"""Test-side helpers: random scans and an independent numpy chord-length routine.

Nothing here calls the oracle or the CUDA library.  The chord routine clips a
line against ONE axis-aligned box (slab method); it never walks cells, so it
checks the oracle's traversal (crossing merge, midpoint cell lookup, lengths)
from outside.
"""

import numpy as np


def pixel_rays(beam, src, det_centre, det_u, det_v, n_u, n_v, pitch_u, pitch_v,
               offset_u=0.0, offset_v=0.0):
    """(X0, r, tlo, thi) for every ray, view-major then v then u, in float64 from
    the float32 frames: pixel = centre + a u + b v with
    a = (iu - (n_u-1)/2 + offset_u) pitch_u, b = (iv - (n_v-1)/2 + offset_v) pitch_v."""
    src, det_centre, det_u, det_v = (np.asarray(x, dtype=np.float32).astype(np.float64)
                                     for x in (src, det_centre, det_u, det_v))
    iu = np.arange(n_u, dtype=np.float64)
    iv = np.arange(n_v, dtype=np.float64)
    a = (iu - 0.5 * (n_u - 1) + offset_u) * pitch_u
    b = (iv - 0.5 * (n_v - 1) + offset_v) * pitch_v
    P = (det_centre[:, None, None, :] + a[None, None, :, None] * det_u[:, None, None, :]
         + b[None, :, None, None] * det_v[:, None, None, :])
    P = P.reshape(-1, 3)
    nview = src.shape[0]
    rep = n_u * n_v
    S = np.repeat(src, rep, axis=0)
    if beam == "divergent":
        return S, P - S, np.zeros(len(P)), np.ones(len(P))
    return P, S, np.full(len(P), -np.inf), np.full(len(P), np.inf)


def chord(X0, r, tlo, thi, lo, hi):
    """Length of X0 + t r, t in [tlo, thi], inside the box [lo, hi] (per-ray arrays)."""
    a0 = tlo.copy()
    a1 = thi.copy()
    inside = np.ones(len(X0), dtype=bool)
    with np.errstate(divide="ignore", invalid="ignore"):
        for ax in range(3):
            zero = r[:, ax] == 0.0
            t0 = (lo[ax] - X0[:, ax]) / r[:, ax]
            t1 = (hi[ax] - X0[:, ax]) / r[:, ax]
            a0 = np.where(zero, a0, np.maximum(a0, np.minimum(t0, t1)))
            a1 = np.where(zero, a1, np.minimum(a1, np.maximum(t0, t1)))
            inside &= ~zero | ((X0[:, ax] >= lo[ax]) & (X0[:, ax] < hi[ax]))
    L = np.where(inside & (a1 > a0), (a1 - a0), 0.0) * np.linalg.norm(r, axis=1)
    return L


def random_frames(rng, n_views, beam, radius, det_dist, tilt=0.3):
    """Random per-view frames around the origin: source (or direction) on a sphere,
    detector facing it with slightly tilted axes."""
    src = np.zeros((n_views, 3))
    cen = np.zeros((n_views, 3))
    U = np.zeros((n_views, 3))
    V = np.zeros((n_views, 3))
    for k in range(n_views):
        d = rng.standard_normal(3)
        d /= np.linalg.norm(d)
        a = rng.standard_normal(3)
        u = np.cross(d, a)
        u /= np.linalg.norm(u)
        v = np.cross(d, u)
        ang = rng.uniform(-tilt, tilt)
        u, v = np.cos(ang) * u + np.sin(ang) * v, -np.sin(ang) * u + np.cos(ang) * v
        if beam == "divergent":
            src[k] = radius * d
            cen[k] = -det_dist * d + rng.uniform(-1, 1, 3) * 0.5
        else:
            src[k] = -d
            cen[k] = rng.uniform(-1, 1, 3) * 0.5
        U[k], V[k] = u, v
    return [x.astype(np.float32) for x in (src, cen, U, V)]
