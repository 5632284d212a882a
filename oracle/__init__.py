"""Float64 CPU oracle for the Siddon projector pair -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library never loads
it, and it never loads the product library: the two share no code; both are
fed from :mod:`ctp_inputs`.

The arithmetic lives in ``siddon_oracle.c`` (plain C, float64, OpenMP over rays
or over owned bands of cells).  This module compiles it with gcc on first use
(or via :func:`build`) and wraps it with ctypes.

Functions and what pins them (the tests under ``tests/test_oracle_*.py``):

* :func:`forward` / :func:`backward` -- textbook parametric Siddon path sum and
  its transpose.  Pinned by chord-length closed forms (uniform boxes, balls),
  the brute-force clip-every-cell path, the supersampled line integral, the
  textbook axis-aligned and diagonal cases, and the float64 adjoint identity.
* :func:`brute_forward`, :func:`brute_count` -- O(cells) per ray; pinned by the
  same closed forms.
* :func:`backward_voxels` -- voxel-driven transpose at chosen voxels; pinned by
  equality with :func:`backward` on small cases.
* :func:`segment_count` -- pieces longer than 1e-5 of the smallest cell width
  (the benchmark's unit); pinned by :func:`brute_count`.
* :func:`ambiguous` -- rays lying on a cell-face plane; pinned on hand-built rays.
* :func:`geometry_vjp` -- first-order gradients of the path sums with respect to
  the per-view frames (flat and curved detectors); pinned by central finite
  differences of :func:`forward` and by the invariance of chords under sliding a
  ray's end points along it.
* :func:`surface_vjp` -- first-order gradients with respect to every pixel's
  offsets along the detector axes and normal; pinned by central finite
  differences of :func:`forward` in the offsets.
* :func:`kinks` -- rays through a cell edge or corner (no geometry derivative);
  pinned on hand-built rays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "siddon_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libctp_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (float64, no fast-math, no FP contraction)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-shared", "-fPIC", "-Wall", "-Wextra", "-Wno-unused-parameter",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Ctx(ctypes.Structure):
    _fields_ = [
        ("beam", ctypes.c_int), ("n_views", ctypes.c_int), ("n_u", ctypes.c_int),
        ("n_v", ctypes.c_int),
        ("src", ctypes.c_void_p), ("det_centre", ctypes.c_void_p),
        ("det_u", ctypes.c_void_p), ("det_v", ctypes.c_void_p),
        ("pitch_u", ctypes.c_double), ("pitch_v", ctypes.c_double),
        ("offset_u", ctypes.c_double), ("offset_v", ctypes.c_double),
        ("n", ctypes.c_int * 3), ("pad_", ctypes.c_int),
        ("d", ctypes.c_double * 3), ("o", ctypes.c_double * 3),
        ("offsets", ctypes.c_void_p), ("offsets_per_view", ctypes.c_int), ("pad2_", ctypes.c_int),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, L, I, D = ctypes.c_void_p, ctypes.c_long, ctypes.c_int, ctypes.c_double
            C = ctypes.POINTER(_Ctx)
            sigs = {
                "ora_forward": [C, P, P, L, L, I],
                "ora_forward_rays": [C, P, P, L, P, I],
                "ora_backward": [C, P, P, L, L, I],
                "ora_segment_count": [C, L, L, I, D, P],
                "ora_brute_forward": [C, P, P, I],
                "ora_brute_count": [C, D, P, I],
                "ora_backward_voxels": [C, P, P, L, P, I],
                "ora_ambiguous": [C, D, P, I],
                "ora_supersampled": [C, P, P, L, L, P, I],
                "ora_trace_ray": [C, L, P, P],
                "ora_geometry_vjp": [C, P, P, P, I],
                "ora_surface_vjp": [C, P, P, P, I],
                "ora_kinks": [C, D, P, I],
            }
            for name, args in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


class Scan:
    """A scan in the oracle's terms: geometry arrays (float32, (n_views, 3)) and
    the volume grid.  ``shape`` is (D, H, W), ``spacing`` (dz, dy, dx), ``origin``
    the world (x, y, z) of the min corner of voxel (0, 0, 0)."""

    def __init__(self, beam, src, det_centre, det_u, det_v, n_u, n_v, pitch_u, pitch_v,
                 shape, spacing, origin, offset_u=0.0, offset_v=0.0, ndim=3, pixel_offsets=None):
        self.beam = beam
        self.ndim = int(ndim)
        self.pitch_u, self.pitch_v = float(pitch_u), float(pitch_v)
        self.offset_u, self.offset_v = float(offset_u), float(offset_v)
        self.arrays = [np.ascontiguousarray(a, dtype=np.float32).reshape(-1, 3)
                       for a in (src, det_centre, det_u, det_v)]
        self.n_views = self.arrays[0].shape[0]
        self.n_u, self.n_v = int(n_u), int(n_v)
        self.shape = tuple(int(s) for s in shape)
        self.spacing = tuple(float(s) for s in spacing)
        self.origin = tuple(float(s) for s in origin)
        c = _Ctx()
        c.beam = 1 if beam == "divergent" else 0
        c.n_views, c.n_u, c.n_v = self.n_views, self.n_u, self.n_v
        c.src, c.det_centre, c.det_u, c.det_v = (a.ctypes.data for a in self.arrays)
        c.pitch_u, c.pitch_v = float(pitch_u), float(pitch_v)
        c.offset_u, c.offset_v = float(offset_u), float(offset_v)
        D, H, W = self.shape
        dz, dy, dx = self.spacing
        c.n[0], c.n[1], c.n[2] = W, H, D
        c.d[0], c.d[1], c.d[2] = dx, dy, dz
        c.o[0], c.o[1], c.o[2] = self.origin
        # curved detector: per-pixel (tangent, vertical, depth) offsets, (n_v, n_u, 3)
        # shared by all views or (n_views, n_v, n_u, 3) one table per view
        self.pixel_offsets = None
        self.offsets_per_view = False
        if pixel_offsets is not None:
            off = np.ascontiguousarray(pixel_offsets, dtype=np.float32)
            self.offsets_per_view = off.size == 3 * self.n_views * self.n_u * self.n_v and \
                off.ndim == 4
            shape = ((self.n_views,) if self.offsets_per_view else ()) + (self.n_v, self.n_u, 3)
            self.pixel_offsets = off.reshape(shape)
            c.offsets = self.pixel_offsets.ctypes.data
            c.offsets_per_view = int(self.offsets_per_view)
        self._ctx = c

    @classmethod
    def from_workload(cls, w, frames):
        return cls(w.beam, frames["src"], frames["det_centre"], frames["det_u"],
                   frames["det_v"], w.n_u, w.n_v, w.pitch_u, w.pitch_v, w.shape,
                   w.spacing, w.origin, w.offset_u, w.offset_v, w.ndim)

    @property
    def n_rays(self):
        return self.n_views * self.n_u * self.n_v

    @property
    def sino_shape(self):
        return (self.n_views, self.n_v, self.n_u)

    def ref(self):
        return ctypes.byref(self._ctx)


def _f32(a, shape=None):
    a = np.ascontiguousarray(a, dtype=np.float32)
    if shape is not None and a.size != int(np.prod(shape)):
        raise ValueError(f"expected {shape}, got {a.shape}")
    return a


def _check(code, name):
    if code != 0:
        raise MemoryError(f"{name} failed ({code})")


def forward(scan: Scan, vol, ray0=0, ray1=None, threads=0):
    """Float64 forward projection of rays [ray0, ray1) (default: all), as (n_rays,)."""
    vol = _f32(vol, scan.shape)
    ray1 = scan.n_rays if ray1 is None else ray1
    out = np.zeros(ray1 - ray0, dtype=np.float64)
    _check(_load().ora_forward(scan.ref(), vol.ctypes.data, out.ctypes.data, ray0, ray1,
                               threads), "ora_forward")
    if ray0 == 0 and ray1 == scan.n_rays:
        return out.reshape(scan.sino_shape)
    return out


def forward_rays(scan: Scan, vol, rays, threads=0):
    vol = _f32(vol, scan.shape)
    rays = np.ascontiguousarray(rays, dtype=np.int64)
    out = np.zeros(rays.size, dtype=np.float64)
    _check(_load().ora_forward_rays(scan.ref(), vol.ctypes.data, rays.ctypes.data, rays.size,
                                    out.ctypes.data, threads), "ora_forward_rays")
    return out


def backward(scan: Scan, sino, ray0=0, ray1=None, threads=0):
    """Float64 backprojection of the rays [ray0, ray1) with values ``sino``
    (length ray1 - ray0), as a (D, H, W) float64 volume."""
    ray1 = scan.n_rays if ray1 is None else ray1
    sino = _f32(sino, (ray1 - ray0,))
    out = np.zeros(scan.shape, dtype=np.float64)
    _check(_load().ora_backward(scan.ref(), sino.ctypes.data, out.ctypes.data, ray0, ray1,
                                threads), "ora_backward")
    return out


def backward_voxels(scan: Scan, sino, voxels, threads=0):
    sino = _f32(sino, scan.sino_shape)
    voxels = np.ascontiguousarray(voxels, dtype=np.int64)
    out = np.zeros(voxels.size, dtype=np.float64)
    _check(_load().ora_backward_voxels(scan.ref(), sino.ctypes.data, voxels.ctypes.data,
                                       voxels.size, out.ctypes.data, threads),
           "ora_backward_voxels")
    return out


SEGMENT_MIN_FRACTION = 1e-5


def segment_min_len(scan: Scan) -> float:
    """Counting threshold: 1e-5 of the smallest cell width.  Pieces shorter than
    this are the degenerate ones of rays crossing a cell edge or corner exactly."""
    return SEGMENT_MIN_FRACTION * min(scan.spacing)


def segment_count(scan: Scan, ray0=0, ray1=None, threads=0, min_len=None) -> int:
    """Pieces longer than ``min_len`` (default :func:`segment_min_len`; 0 counts
    every positive-length piece) over rays [ray0, ray1)."""
    ray1 = scan.n_rays if ray1 is None else ray1
    min_len = segment_min_len(scan) if min_len is None else float(min_len)
    out = ctypes.c_ulonglong(0)
    _check(_load().ora_segment_count(scan.ref(), ray0, ray1, threads, min_len,
                                     ctypes.byref(out)), "ora_segment_count")
    return int(out.value)


def brute_forward(scan: Scan, vol, threads=0):
    vol = _f32(vol, scan.shape)
    out = np.zeros(scan.n_rays, dtype=np.float64)
    _check(_load().ora_brute_forward(scan.ref(), vol.ctypes.data, out.ctypes.data, threads),
           "ora_brute_forward")
    return out.reshape(scan.sino_shape)


def brute_count(scan: Scan, threads=0, min_len=None) -> int:
    min_len = segment_min_len(scan) if min_len is None else float(min_len)
    out = ctypes.c_ulonglong(0)
    _check(_load().ora_brute_count(scan.ref(), min_len, ctypes.byref(out), threads),
           "ora_brute_count")
    return int(out.value)


def ambiguous(scan: Scan, tol=1e-6, threads=0):
    """Boolean (n_views, n_v, n_u): rays lying (numerically) in a cell-face plane."""
    out = np.zeros(scan.n_rays, dtype=np.uint8)
    _check(_load().ora_ambiguous(scan.ref(), float(tol), out.ctypes.data, threads),
           "ora_ambiguous")
    return out.reshape(scan.sino_shape).astype(bool)


def supersampled(scan: Scan, vol, rays, samples, threads=0):
    vol = _f32(vol, scan.shape)
    rays = np.ascontiguousarray(rays, dtype=np.int64)
    out = np.zeros(rays.size, dtype=np.float64)
    _check(_load().ora_supersampled(scan.ref(), vol.ctypes.data, rays.ctypes.data, rays.size,
                                    int(samples), out.ctypes.data, threads),
           "ora_supersampled")
    return out


def trace_ray(scan: Scan, ray: int):
    """(cells, lengths) of one ray's positive-length pieces, in traversal order;
    cells are linear indices (k * ny + j) * nx + i."""
    n = sum(scan.shape) + 8
    cells = np.zeros(n, dtype=np.int64)
    lens = np.zeros(n, dtype=np.float64)
    m = _load().ora_trace_ray(scan.ref(), int(ray), cells.ctypes.data, lens.ctypes.data)
    if m < 0:
        raise MemoryError("ora_trace_ray failed")
    return cells[:m], lens[:m]


def geometry_vjp(scan: Scan, vol, weights, threads=0):
    """Float64 first-order geometry gradient: (n_views, 4, 3) array of
    sum over the view's rays of weights[ray] * d p(ray) / d frame, frames in the
    order src, det_centre, det_u, det_v (the sum of crossing terms written out in
    ``siddon_oracle.c``)."""
    vol = _f32(vol, scan.shape)
    w = _f32(weights, (scan.n_rays,))
    out = np.zeros((scan.n_views, 4, 3), dtype=np.float64)
    _check(_load().ora_geometry_vjp(scan.ref(), vol.ctypes.data, w.ctypes.data,
                                    out.ctypes.data, threads), "ora_geometry_vjp")
    return out


def surface_vjp(scan: Scan, vol, weights, threads=0):
    """Float64 first-order gradient with respect to the detector surface: (n_v,
    n_u, 3) array of sum over views of weights[ray] * d p(ray) / d (t, s, e),
    the pixel's offsets along det_u, det_v and the unit normal det_u x det_v
    (a curved detector's own offsets, or the pitch grid of a flat one); with one
    offset table per view, (n_views, n_v, n_u, 3) without the sum over views."""
    vol = _f32(vol, scan.shape)
    w = _f32(weights, (scan.n_rays,))
    shape = ((scan.n_views,) if scan.offsets_per_view else ()) + (scan.n_v, scan.n_u, 3)
    out = np.zeros(shape, dtype=np.float64)
    _check(_load().ora_surface_vjp(scan.ref(), vol.ctypes.data, w.ctypes.data,
                                   out.ctypes.data, threads), "ora_surface_vjp")
    return out


def kinks(scan: Scan, tol=1e-6, threads=0):
    """Boolean (n_views, n_v, n_u): rays on which two plane crossings of different
    axes coincide within ``tol`` cells (through a cell edge or corner), or whose
    end point inside the grid lies on a plane: the path sum has no geometry
    derivative there."""
    flags = np.zeros(scan.n_rays, dtype=np.uint8)
    _check(_load().ora_kinks(scan.ref(), float(tol), flags.ctypes.data, threads), "ora_kinks")
    return flags.reshape(scan.sino_shape).astype(bool)
