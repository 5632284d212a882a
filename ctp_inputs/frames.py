"""Per-view source / detector frames of the three trajectory kinds.

Each view has its own source (or, for parallel beams, unit ray direction),
detector centre and detector axes u, v, as the pages' per-view trajectory tuple
``(src_pos, det_center, det_u_vec[, det_v_vec])`` (diffct 2.1.0 -> 2.2.1,
``analytical.py`` signatures; README "Arbitrary trajectories": "Each view has
its own source, detector centre and detector axes").  The frames are built in
float64 and handed over as float32 vectors; every consumer promotes those same
float32 values.
"""

from __future__ import annotations

import math

import numpy as np

from .workloads import Workload


def view_angles(w: Workload) -> np.ndarray:
    """Rotation angle of each view: uniform over ``w.arc`` with the end excluded."""
    k = np.arange(w.n_views, dtype=np.float64)
    return k * (w.arc / w.n_views)


def frames(w: Workload) -> dict:
    """Float32 arrays of shape (n_views, 3): ``src``, ``det_centre``, ``det_u``, ``det_v``.

    circular (fan / cone): source at SID (cos b, sin b, 0), detector centre at
    -(SDD - SID) (cos b, sin b, 0), u = (-sin b, cos b, 0), v = (0, 0, 1).
    helical: the circular frame with source and detector centre both at
    z = z_start + table_per_turn * b / (2 pi).
    parallel: ``src`` holds the unit ray direction (cos t, sin t, 0), the detector
    line passes through the origin with u = (-sin t, cos t, 0).
    2-D workloads use z = 0 components (v is still (0, 0, 1), unused).
    """
    b = view_angles(w)
    c, s = np.cos(b), np.sin(b)
    zeros = np.zeros_like(b)
    ones = np.ones_like(b)
    det_u = np.stack([-s, c, zeros], axis=1)
    det_v = np.stack([zeros, zeros, ones], axis=1)
    if w.trajectory == "parallel":
        src = np.stack([c, s, zeros], axis=1)
        det_centre = np.zeros((w.n_views, 3))
    elif w.trajectory in ("circular", "helical"):
        z = zeros
        if w.trajectory == "helical":
            z = w.z_start + w.table_per_turn * b / (2 * math.pi)
        src = np.stack([w.sid * c, w.sid * s, z], axis=1)
        det_centre = np.stack([-(w.sdd - w.sid) * c, -(w.sdd - w.sid) * s, z], axis=1)
    else:
        raise ValueError(f"unknown trajectory {w.trajectory!r}")
    out = {"src": src, "det_centre": det_centre, "det_u": det_u, "det_v": det_v}
    return {k: np.ascontiguousarray(v, dtype=np.float32) for k, v in out.items()}
