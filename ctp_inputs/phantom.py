"""Voxelised random-ellipse / random-ellipsoid phantoms and N(0,1) sinograms.

A voxel's value is the sum of the intensities of the shapes that contain the
voxel CENTRE (no supersampling), plus optional U[0, noise] per voxel.  Shape
parameters are drawn from ``numpy.random.default_rng(w.seed_phantom)`` in a
fixed order; the sinogram fed to backprojection is N(0,1) float32 from
``default_rng(w.seed_sino)``.
"""

from __future__ import annotations

import numpy as np

from .workloads import Workload


def _random_rotation(rng, n):
    """Uniform random rotations from normalised Gaussian quaternions."""
    q = rng.standard_normal((n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    a, b, c, d = q.T
    R = np.empty((n, 3, 3))
    R[:, 0, 0] = a * a + b * b - c * c - d * d
    R[:, 0, 1] = 2 * (b * c - a * d)
    R[:, 0, 2] = 2 * (b * d + a * c)
    R[:, 1, 0] = 2 * (b * c + a * d)
    R[:, 1, 1] = a * a - b * b + c * c - d * d
    R[:, 1, 2] = 2 * (c * d - a * b)
    R[:, 2, 0] = 2 * (b * d - a * c)
    R[:, 2, 1] = 2 * (c * d + a * b)
    R[:, 2, 2] = a * a - b * b - c * c + d * d
    return R


def shapes(w: Workload):
    """The phantom's shape list: centres (n, ndim) world (x, y[, z]), semi-axes,
    rotation matrices (n, ndim, ndim) whose columns are the shape's axes, intensities."""
    rng = np.random.default_rng(w.seed_phantom)
    n, nd = w.n_shapes, w.ndim
    half = np.asarray(w.centre_range[:nd], dtype=np.float64)
    centres = rng.uniform(-1.0, 1.0, size=(n, nd)) * half
    lo, hi = w.semi_axis_range
    semi = rng.uniform(lo, hi, size=(n, nd))
    if nd == 2:
        ang = rng.uniform(0.0, np.pi, size=n)
        c, s = np.cos(ang), np.sin(ang)
        R = np.stack([np.stack([c, -s], 1), np.stack([s, c], 1)], 1)
    else:
        R = _random_rotation(rng, n)
    intensity = rng.uniform(0.0, 1.0, size=n)
    return centres, semi, R, intensity


def _axis_centres(n, d, o):
    return o + (np.arange(n, dtype=np.float64) + 0.5) * d


def phantom(w: Workload) -> np.ndarray:
    """Float32 volume of shape (D, H, W)."""
    D, H, W = w.shape
    dz, dy, dx = w.spacing
    ox, oy, oz = w.origin
    xs, ys, zs = _axis_centres(W, dx, ox), _axis_centres(H, dy, oy), _axis_centres(D, dz, oz)
    vol = np.zeros((D, H, W), dtype=np.float64)
    centres, semi, R, intensity = shapes(w)
    for n in range(w.n_shapes):
        # Axis-aligned half extent of the rotated shape: sqrt(sum_j (R_ij s_j)^2).
        ext = np.sqrt(((R[n] * semi[n][None, :]) ** 2).sum(axis=1))
        lo = centres[n] - ext
        hi = centres[n] + ext
        ix = np.nonzero((xs >= lo[0]) & (xs <= hi[0]))[0]
        iy = np.nonzero((ys >= lo[1]) & (ys <= hi[1]))[0]
        if ix.size == 0 or iy.size == 0:
            continue
        X = (xs[ix] - centres[n][0])
        Y = (ys[iy] - centres[n][1])
        if w.ndim == 2:
            # local coordinates q = R^T (p - c)
            q0 = R[n][0, 0] * X[None, :] + R[n][1, 0] * Y[:, None]
            q1 = R[n][0, 1] * X[None, :] + R[n][1, 1] * Y[:, None]
            inside = (q0 / semi[n][0]) ** 2 + (q1 / semi[n][1]) ** 2 <= 1.0
            vol[0, iy[0]:iy[-1] + 1, ix[0]:ix[-1] + 1] += intensity[n] * inside
        else:
            iz = np.nonzero((zs >= lo[2]) & (zs <= hi[2]))[0]
            if iz.size == 0:
                continue
            Z = (zs[iz] - centres[n][2])
            acc = np.zeros((iz.size, iy.size, ix.size))
            for a in range(3):
                qa = (R[n][0, a] * X[None, None, :] + R[n][1, a] * Y[None, :, None]
                      + R[n][2, a] * Z[:, None, None])
                acc += (qa / semi[n][a]) ** 2
            sl = (slice(iz[0], iz[-1] + 1), slice(iy[0], iy[-1] + 1), slice(ix[0], ix[-1] + 1))
            vol[sl] += intensity[n] * (acc <= 1.0)
    if w.noise > 0:
        rng = np.random.default_rng(w.seed_phantom + 7919)
        vol += rng.uniform(0.0, w.noise, size=vol.shape)
    return np.ascontiguousarray(vol, dtype=np.float32)


def sinogram_noise(w: Workload) -> np.ndarray:
    """Float32 N(0,1) sinogram of shape (n_views, n_v, n_u)."""
    rng = np.random.default_rng(w.seed_sino)
    return rng.standard_normal(size=w.sino_shape, dtype=np.float32)
