"""Seeded random small scans for the parity tests (inputs only: frames, grid
and detector; no projector arithmetic): beam type, arbitrary or vertical
detector axes (column path), circular arcs with the source inside or outside the
grid, 2-D slices (plane path), grid sizes from one cell upwards, anisotropic
spacing, detector sizes, pitches and offsets."""

import numpy as np

from geom_helpers import random_frames

N_CASES = 40


def random_scan(seed):
    """(beam, ndim, frames, n_u, n_v, pitch_u, pitch_v, offset_u, offset_v, shape,
    spacing) of random scan `seed`."""
    rng = np.random.default_rng(7000 + seed)
    kind = ["arbitrary", "vertical", "vertical", "slice"][seed % 4]
    beam = "divergent" if rng.uniform() < 0.7 else "parallel"
    shape = tuple(int(x) for x in rng.integers(1, 14, 3))
    spacing = tuple(float(x) for x in rng.uniform(0.5, 2.0, 3))
    K = int(rng.integers(1, 9))
    n_u, n_v = int(rng.integers(1, 40)), int(rng.integers(1, 30))
    pu, pv = float(rng.uniform(0.3, 2.0)), float(rng.uniform(0.3, 2.0))
    ou, ov = float(rng.uniform(-2, 2)), float(rng.uniform(-2, 2))
    ext = max(n * d for n, d in zip(shape, spacing[::-1]))
    ndim = 3
    if kind == "arbitrary":
        frames = random_frames(rng, K, beam, radius=ext * rng.uniform(0.6, 3.0),
                               det_dist=ext * rng.uniform(0.6, 2.0), tilt=0.5)
    else:
        # circular arc about z with vertical detector columns; the source may sit
        # inside the grid (radius below the half extent)
        b = rng.uniform(0, 2 * np.pi) + np.linspace(0, rng.uniform(0.5, 2 * np.pi), K,
                                                    endpoint=False)
        c, s, z = np.cos(b), np.sin(b), np.zeros_like(b)
        R = ext * rng.uniform(0.3, 3.0)
        zs = rng.uniform(-0.3, 0.3) * ext
        if kind == "slice":
            ndim, n_v, ov, zs = 2, 1, 0.0, 0.0
            shape = (1,) + shape[1:]
            spacing = (1.0,) + spacing[1:]
        if beam == "divergent":
            src = np.stack([R * c, R * s, z + zs], 1)
            cen = np.stack([-0.8 * ext * c, -0.8 * ext * s, z + zs], 1)
        else:
            tilt_z = rng.uniform(-0.3, 0.3) if kind == "vertical" else 0.0
            src = np.stack([c, s, z + tilt_z], 1) / np.sqrt(1 + tilt_z ** 2)
            cen = np.stack([z, z, z + zs], 1)
        frames = [x.astype(np.float32) for x in
                  (src, cen, np.stack([-s, c, z], 1), np.stack([z, z, z + 1.0], 1))]
    return beam, ndim, frames, n_u, n_v, pu, pv, ou, ov, shape, spacing
