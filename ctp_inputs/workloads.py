"""The five scan workloads and reduced copies of them for parity tests.

Every workload is a plain record of grid, detector, trajectory and phantom
recipe.  Lengths are physical units (the same unit as the voxel spacing).
Tensor order is kept everywhere: volume shape ``(D, H, W)`` <-> world axes
``(z, y, x)``, spacing ``(dz, dy, dx)`` (diffct 2.4.3 -> 2.4.4, CHANGELOG
2.4.4 "Added": per-axis spacing "in tensor axis order" and "physical length
units").  Volumes are centred on the world origin, as the pages' kernels are
given geometry relative to the volume centre (diffct 2.4.3 -> 2.4.4,
``analytical_execution.py``: ``geometry[0] - centre``).
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    ndim: int                 # 2 or 3
    beam: str                 # "parallel" or "divergent" (fan in 2-D, cone in 3-D)
    trajectory: str           # "parallel", "circular" or "helical"
    shape: tuple              # (D, H, W); D == 1 for 2-D
    spacing: tuple            # (dz, dy, dx)
    n_views: int
    n_u: int
    n_v: int                  # 1 for 2-D
    pitch_u: float
    pitch_v: float
    offset_u: float = 0.0     # detector-centre offset, in pixels
    offset_v: float = 0.0
    arc: float = 2 * math.pi  # total source rotation over all views (radians)
    sid: float = 0.0          # source-to-isocentre distance (divergent beams)
    sdd: float = 0.0          # source-to-detector distance (divergent beams)
    table_per_turn: float = 0.0   # helical table feed per 2*pi
    z_start: float = 0.0          # helical source z at the first view
    n_shapes: int = 8
    centre_range: tuple = ()      # per world axis (x, y[, z]) half-range of centres
    semi_axis_range: tuple = (4.0, 20.0)
    noise: float = 0.0            # U[0, noise] added to every voxel
    seed_phantom: int = 1000
    seed_sino: int = 2000

    # -- derived quantities -------------------------------------------------
    @property
    def origin(self):
        """World position (x, y, z) of the min corner of voxel (0, 0, 0): centred volume."""
        D, H, W = self.shape
        dz, dy, dx = self.spacing
        return (-0.5 * W * dx, -0.5 * H * dy, -0.5 * D * dz)

    @property
    def n_rays(self):
        return self.n_views * self.n_u * self.n_v

    @property
    def n_voxels(self):
        return self.shape[0] * self.shape[1] * self.shape[2]

    @property
    def sino_shape(self):
        return (self.n_views, self.n_v, self.n_u)

    def describe(self):
        return dataclasses.asdict(self)


def _c1():
    # 2-D parallel beam: 64x64, spacing 1.0, 90 views uniform over [0, 180 deg),
    # 96 bins at pitch 1.0, 8 ellipses (centres in [-24, 24], semi-axes in
    # [4, 20], angles U[0, pi), intensities U[0, 1]).
    return Workload(
        name="c1_parallel2d_64", ndim=2, beam="parallel", trajectory="parallel",
        shape=(1, 64, 64), spacing=(1.0, 1.0, 1.0), n_views=90, n_u=96, n_v=1,
        pitch_u=1.0, pitch_v=1.0, arc=math.pi, n_shapes=8,
        centre_range=(24.0, 24.0), semi_axis_range=(4.0, 20.0),
        seed_phantom=1001, seed_sino=2001)


def _c2():
    # 2-D fan beam: 512x512 at spacing 0.5, 720 views over 360 deg, 768 bins at
    # pitch 1.0, SID 1000 / SDD 1500; 20 ellipses with the 64x64 recipe scaled
    # x8 in voxel units (x4 in world units at half the voxel size).
    return Workload(
        name="c2_fan2d_512", ndim=2, beam="divergent", trajectory="circular",
        shape=(1, 512, 512), spacing=(1.0, 0.5, 0.5), n_views=720, n_u=768, n_v=1,
        pitch_u=1.0, pitch_v=1.0, sid=1000.0, sdd=1500.0, n_shapes=20,
        centre_range=(96.0, 96.0), semi_axis_range=(16.0, 80.0),
        seed_phantom=1002, seed_sino=2002)


def _c3():
    # 3-D circular cone beam: 256^3 at spacing 1.0, 360 views, 384x384 at pitch
    # 1.2, SID 600 / SDD 1000, 16 ellipsoids with semi-axes 8..80.
    return Workload(
        name="c3_cone_256", ndim=3, beam="divergent", trajectory="circular",
        shape=(256, 256, 256), spacing=(1.0, 1.0, 1.0), n_views=360, n_u=384, n_v=384,
        pitch_u=1.2, pitch_v=1.2, sid=600.0, sdd=1000.0, n_shapes=16,
        centre_range=(64.0, 64.0, 64.0), semi_axis_range=(8.0, 80.0),
        seed_phantom=1003, seed_sino=2003)


def _c4():
    # 3-D cone beam, anisotropic (dz, dy, dx) = (1.0, 0.8, 0.8): 512^3, 720 views,
    # 768 (u) x 512 (v) at pitch 1.0, SID 800 / SDD 1200, u-offset 3.5 px;
    # 32 ellipsoids plus U[0, 0.01] noise.
    return Workload(
        name="c4_cone_512_aniso", ndim=3, beam="divergent", trajectory="circular",
        shape=(512, 512, 512), spacing=(1.0, 0.8, 0.8), n_views=720, n_u=768, n_v=512,
        pitch_u=1.0, pitch_v=1.0, offset_u=3.5, sid=800.0, sdd=1200.0, n_shapes=32,
        centre_range=(102.4, 102.4, 128.0), semi_axis_range=(12.8, 128.0), noise=0.01,
        seed_phantom=1004, seed_sino=2004)


def _c5():
    # 3-D helical cone beam: 512 x 512 x 256 (x, y, z) at spacing (0.7, 0.7, 1.0),
    # 1440 views over 4 turns, table feed 40 per turn, flat 736 x 64 detector at
    # pitch 1.0, SID 570 / SDD 1040; 24 ellipsoids.
    return Workload(
        name="c5_helical_512x512x256", ndim=3, beam="divergent", trajectory="helical",
        shape=(256, 512, 512), spacing=(1.0, 0.7, 0.7), n_views=1440, n_u=736, n_v=64,
        pitch_u=1.0, pitch_v=1.0, arc=4 * 2 * math.pi, sid=570.0, sdd=1040.0,
        table_per_turn=40.0, z_start=-80.0, n_shapes=24,
        centre_range=(89.6, 89.6, 64.0), semi_axis_range=(11.2, 112.0),
        seed_phantom=1005, seed_sino=2005)


WORKLOADS = {1: _c1(), 2: _c2(), 3: _c3(), 4: _c4(), 5: _c5()}


def get(index: int) -> Workload:
    return WORKLOADS[int(index)]


def scaled(w: Workload, grid: float, views: int | None = None, name: str | None = None,
           ragged: int = 1) -> Workload:
    """A coarser copy of ``w`` with the same physical scan.

    Voxel and detector counts are divided by ``grid`` (then ``ragged`` is added,
    so sizes are not multiples of any tile), spacings and pitches are multiplied
    by the same factor, so extents, distances, cone angles and phantom shapes are
    unchanged.  ``views`` replaces the number of views (same arc).
    """
    D, H, W = w.shape
    dz, dy, dx = w.spacing

    def n(count):
        return max(1, int(round(count / grid)) + ragged)

    nD = 1 if w.ndim == 2 else n(D)
    nH, nW = n(H), n(W)
    sz = 1.0 if w.ndim == 2 else D * dz / nD
    nu = n(w.n_u)
    nv = 1 if w.ndim == 2 else n(w.n_v)
    pu = w.pitch_u * w.n_u / nu
    pv = w.pitch_v if w.ndim == 2 else w.pitch_v * w.n_v / nv
    return dataclasses.replace(
        w, name=name or f"{w.name}_div{grid:g}",
        shape=(nD, nH, nW), spacing=(sz, H * dy / nH, W * dx / nW),
        n_u=nu, n_v=nv, pitch_u=pu, pitch_v=pv,
        offset_u=w.offset_u * w.pitch_u / pu, offset_v=w.offset_v * w.pitch_v / pv,
        n_views=views if views is not None else w.n_views)


def small_cases():
    """Reduced copies of the five workloads that the float64 oracle finishes in
    seconds while still spanning several thread blocks and ragged tails."""
    return {
        1: scaled(WORKLOADS[1], 1.0, views=90, ragged=0, name="c1_full"),
        2: scaled(WORKLOADS[2], 8.0, views=60),
        3: scaled(WORKLOADS[3], 8.0, views=24),
        4: scaled(WORKLOADS[4], 12.0, views=24),
        5: scaled(WORKLOADS[5], 8.0, views=96),
    }
