"""Thin ctypes binding of the C ABI in ``include/ctp.h`` -- argument marshalling only.

Every step of the projector runs in ``libctp.so`` (CUDA, sm_103a).  There is no
CPU or PyTorch fallback: if the library cannot be loaded, importing the entry
points raises.  PyTorch is used for device memory and streams only.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libctp.so")
# CTP_LIBRARY_VARIANT=check loads the bounds-checked debug build instead
_CHECK_LIB_PATH = os.path.join(_HERE, "libctp_check.so")
_lib = None
_lock = threading.Lock()

PATHS = {"auto": 0, "ray": 1, "column": 2, "plane": 3}
PATH_NAMES = {v: k for k, v in PATHS.items()}
BEAMS = {"parallel": 0, "divergent": 1}


class CtpError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {ctp_status_string(status)} (status {status})")


class _Geometry(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int), ("beam", ctypes.c_int), ("n_views", ctypes.c_int),
                ("n_u", ctypes.c_int), ("n_v", ctypes.c_int),
                ("src", ctypes.c_void_p), ("det_centre", ctypes.c_void_p),
                ("det_u", ctypes.c_void_p), ("det_v", ctypes.c_void_p),
                ("pitch_u", ctypes.c_double), ("pitch_v", ctypes.c_double),
                ("offset_u", ctypes.c_double), ("offset_v", ctypes.c_double),
                ("pixel_offsets", ctypes.c_void_p), ("offsets_per_view", ctypes.c_int)]


class _Volume(ctypes.Structure):
    _fields_ = [("nx", ctypes.c_int), ("ny", ctypes.c_int), ("nz", ctypes.c_int),
                ("dx", ctypes.c_double), ("dy", ctypes.c_double), ("dz", ctypes.c_double),
                ("ox", ctypes.c_double), ("oy", ctypes.c_double), ("oz", ctypes.c_double)]


class _PlanOptions(ctypes.Structure):
    _fields_ = [("rows_forward", ctypes.c_int), ("rows_backward", ctypes.c_int),
                ("backward_rows_adjacent", ctypes.c_int), ("plane_backward", ctypes.c_int),
                ("host_chunks", ctypes.c_int), ("geometry_walk", ctypes.c_int),
                ("forward_ahead", ctypes.c_int), ("forward_views_first", ctypes.c_int)]


# Work-layout options of a plan (include/ctp.h, ctp_plan_options); keyword values
# accepted by ctp_plan(..., options=...).
PLANE_BACKWARD = {"auto": 0, "tiled": 1, "privatised": 2}
GEOMETRY_WALK = {"auto": 0, "ray": 1}
FORWARD_AHEAD = {"auto": 0, "off": 1, "on": 2}
FORWARD_VIEWS_FIRST = {"auto": 0, "off": 1, "on": 2}


def _plan_options(options):
    if not options:
        return None
    o = _PlanOptions()
    for key, value in options.items():
        if key == "plane_backward":
            value = PLANE_BACKWARD[value] if isinstance(value, str) else value
        elif key == "geometry_walk":
            value = GEOMETRY_WALK[value] if isinstance(value, str) else value
        elif key == "forward_ahead":
            value = FORWARD_AHEAD[value] if isinstance(value, str) else value
        elif key == "forward_views_first":
            value = FORWARD_VIEWS_FIRST[value] if isinstance(value, str) else value
        elif key not in ("rows_forward", "rows_backward", "backward_rows_adjacent",
                         "host_chunks"):
            raise ValueError(f"unknown plan option {key!r}")
        setattr(o, key, int(value))
    return o


class _PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("device", ctypes.c_int), ("n_rays", ctypes.c_longlong),
                ("n_cells", ctypes.c_longlong), ("device_bytes", ctypes.c_ulonglong)]


EXPORTS = ("ctp_plan", "ctp_plan_ex", "ctp_destroy", "ctp_plan_info_get", "ctp_forward", "ctp_backward",
           "ctp_segment_count", "ctp_forward_host", "ctp_backward_host", "ctp_status_string",
           "ctp_forward_static", "ctp_ramp_filter", "ctp_weighted_backproject",
           "ctp_weighted_backproject_transpose", "ctp_fdk", "ctp_geometry_vjp",
           "ctp_parker_weights", "ctp_check_violations", "ctp_surface_vjp")

RAMPS = {"ramlak": 0, "shepp_logan": 1, "cosine": 2, "hamming": 3, "hann": 4}


def load_library(path: str | None = None):
    """Load ``libctp.so`` (building it first when it is absent and nvcc exists);
    with CTP_LIBRARY_VARIANT=check, the bounds-checked ``libctp_check.so``."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        check = os.environ.get("CTP_LIBRARY_VARIANT") == "check"
        lib_path = path or (_CHECK_LIB_PATH if check else _LIB_PATH)
        if not os.path.exists(lib_path):
            from . import build as _build
            _build.build(check=check)
        lib = ctypes.CDLL(lib_path)
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.ctp_plan.argtypes = [ctypes.POINTER(_Geometry), ctypes.POINTER(_Volume), I,
                                 ctypes.POINTER(ctypes.c_void_p)]
        lib.ctp_plan_ex.argtypes = [ctypes.POINTER(_Geometry), ctypes.POINTER(_Volume), I,
                                    ctypes.POINTER(_PlanOptions), ctypes.POINTER(ctypes.c_void_p)]
        lib.ctp_destroy.argtypes = [P]
        lib.ctp_destroy.restype = None
        lib.ctp_plan_info_get.argtypes = [P, ctypes.POINTER(_PlanInfo)]
        for name in ("ctp_forward", "ctp_backward", "ctp_forward_host", "ctp_backward_host"):
            getattr(lib, name).argtypes = [P, P, P, P]
        lib.ctp_segment_count.argtypes = [P, ctypes.POINTER(ctypes.c_ulonglong), P]
        lib.ctp_forward_static.argtypes = [ctypes.POINTER(_Geometry), ctypes.POINTER(_Volume),
                                           P, P, P]
        lib.ctp_ramp_filter.argtypes = [P, P, P, P, P, I, I, P]
        lib.ctp_weighted_backproject.argtypes = [P, P, P, P]
        lib.ctp_weighted_backproject_transpose.argtypes = [P, P, P, P]
        lib.ctp_fdk.argtypes = [P, P, P, P, P, P, I, P]
        lib.ctp_parker_weights.argtypes = [P, P, P]
        lib.ctp_geometry_vjp.argtypes = [P, P, P, P, P]
        lib.ctp_surface_vjp.argtypes = [P, P, P, P, P]
        lib.ctp_check_violations.argtypes = [ctypes.POINTER(ctypes.c_ulonglong),
                                             ctypes.POINTER(ctypes.c_longlong),
                                             ctypes.POINTER(ctypes.c_longlong),
                                             ctypes.POINTER(ctypes.c_int)]
        lib.ctp_status_string.argtypes = [I]
        lib.ctp_status_string.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name not in ("ctp_destroy", "ctp_status_string"):
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def ctp_status_string(status: int) -> str:
    return load_library().ctp_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise CtpError(status, where)


@dataclasses.dataclass
class Geometry:
    """Per-view frames (float32, (n_views, 3)) and detector description."""
    ndim: int
    beam: str
    src: np.ndarray
    det_centre: np.ndarray
    det_u: np.ndarray
    det_v: np.ndarray
    n_u: int
    n_v: int
    pitch_u: float
    pitch_v: float
    offset_u: float = 0.0
    offset_v: float = 0.0
    # curved detector: (n_v, n_u, 3) per-pixel (t, s, e) offsets from det_centre
    # along det_u, det_v and the unit normal det_u x det_v, shared by all views,
    # or (n_views, n_v, n_u, 3) one table per view; None = the pitch grid
    pixel_offsets: np.ndarray | None = None


@dataclasses.dataclass
class Volume:
    """Grid in tensor order: shape (D, H, W), spacing (dz, dy, dx); origin is the
    world (x, y, z) of the min corner of cell (0, 0, 0)."""
    shape: tuple
    spacing: tuple
    origin: tuple


class Plan:
    """Owner of a ``ctp_plan_t``; destroyed with the object."""

    def __init__(self, handle, geometry: Geometry, volume: Volume):
        self._h = handle
        self.geometry = geometry
        self.volume = volume
        info = _PlanInfo()
        _check(load_library().ctp_plan_info_get(handle, ctypes.byref(info)), "ctp_plan_info_get")
        self.path = PATH_NAMES[info.path]
        self.device = info.device
        self.n_rays = int(info.n_rays)
        self.n_cells = int(info.n_cells)
        self.device_bytes = int(info.device_bytes)

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("plan was destroyed")
        return self._h

    @property
    def sino_shape(self):
        g = self.geometry
        return (g.src.shape[0], g.n_v, g.n_u)

    @property
    def vol_shape(self):
        return tuple(self.volume.shape)

    def destroy(self):
        if self._h is not None and _lib is not None:
            _lib.ctp_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _c_scan(geometry: Geometry, volume: Volume):
    """C structs of a scan; the returned arrays must outlive the structs' use."""
    arrays = [np.ascontiguousarray(a, dtype=np.float32).reshape(-1, 3)
              for a in (geometry.src, geometry.det_centre, geometry.det_u, geometry.det_v)]
    g = _Geometry()
    g.ndim, g.beam, g.n_views = int(geometry.ndim), BEAMS[geometry.beam], arrays[0].shape[0]
    g.n_u, g.n_v = int(geometry.n_u), int(geometry.n_v)
    g.src, g.det_centre, g.det_u, g.det_v = (a.ctypes.data for a in arrays)
    g.pitch_u, g.pitch_v = float(geometry.pitch_u), float(geometry.pitch_v)
    g.offset_u, g.offset_v = float(geometry.offset_u), float(geometry.offset_v)
    arrays.append(_pixel_offsets(geometry, g))
    D, H, W = (int(s) for s in volume.shape)
    v = _Volume()
    v.nx, v.ny, v.nz = W, H, D
    v.dz, v.dy, v.dx = (float(s) for s in volume.spacing)
    v.ox, v.oy, v.oz = (float(s) for s in volume.origin)
    return g, v, arrays


def _pixel_offsets(geometry: Geometry, g: _Geometry):
    """Sets g.pixel_offsets (and g.offsets_per_view); returns the array that must
    outlive the call."""
    g.offsets_per_view = 0
    if geometry.pixel_offsets is None:
        g.pixel_offsets = None
        return None
    off = np.ascontiguousarray(geometry.pixel_offsets, dtype=np.float32)
    per = 3 * int(geometry.n_u) * int(geometry.n_v)
    n_views = np.asarray(geometry.src).reshape(-1, 3).shape[0]
    if off.ndim == 4 and off.size == per * n_views:
        g.offsets_per_view = 1
    elif off.size != per:
        raise ValueError("pixel_offsets must hold (n_v, n_u, 3) or (n_views, n_v, n_u, 3) values")
    g.pixel_offsets = off.ctypes.data
    return off


def ctp_forward_static(geometry: Geometry, volume: Volume, vol, sino, stream=None):
    """sino <- A vol with no allocation (per-view frames in a fixed device array of
    at most 4096 views); equals ctp_forward of a "ray" plan of the same scan.
    ``vol`` and ``sino`` must live on the current CUDA device, where the call
    runs."""
    import torch
    cur = torch.cuda.current_device()
    for name, t in (("vol", vol), ("sino", sino)):
        if isinstance(t, torch.Tensor) and t.is_cuda and t.device.index != cur:
            raise ValueError(f"{name} is on cuda:{t.device.index}, the current device is "
                             f"cuda:{cur}")
    g, v, arrays = _c_scan(geometry, volume)
    n_views = arrays[0].shape[0]
    shape_v = tuple(int(s) for s in volume.shape)
    shape_s = (n_views, int(geometry.n_v), int(geometry.n_u))
    _check(load_library().ctp_forward_static(ctypes.byref(g), ctypes.byref(v),
                                             _device_f32(vol, shape_v, "vol"),
                                             _device_f32(sino, shape_s, "sino"),
                                             _stream_ptr(stream)), "ctp_forward_static")
    return sino


def ctp_plan(geometry: Geometry, volume: Volume, path: str = "auto", options=None) -> Plan:
    """Plan a scan on the current CUDA device.  ``options``: None, or a dict of
    work-layout options (``rows_forward``, ``rows_backward``,
    ``backward_rows_adjacent``, ``plane_backward`` ("auto" / "tiled" /
    "privatised"), ``host_chunks``, ``geometry_walk`` ("auto" / "ray")); they
    select among layouts that compute the same operator."""
    lib = load_library()
    opts = _plan_options(options)
    arrays = [np.ascontiguousarray(a, dtype=np.float32).reshape(-1, 3)
              for a in (geometry.src, geometry.det_centre, geometry.det_u, geometry.det_v)]
    n_views = arrays[0].shape[0]
    if any(a.shape[0] != n_views for a in arrays):
        raise ValueError("frame arrays must all have shape (n_views, 3)")
    g = _Geometry()
    g.ndim, g.beam, g.n_views = int(geometry.ndim), BEAMS[geometry.beam], n_views
    g.n_u, g.n_v = int(geometry.n_u), int(geometry.n_v)
    g.src, g.det_centre, g.det_u, g.det_v = (a.ctypes.data for a in arrays)
    g.pitch_u, g.pitch_v = float(geometry.pitch_u), float(geometry.pitch_v)
    g.offset_u, g.offset_v = float(geometry.offset_u), float(geometry.offset_v)
    offsets = _pixel_offsets(geometry, g)  # noqa: F841 (kept alive for the call)
    D, H, W = (int(s) for s in volume.shape)
    dz, dy, dx = (float(s) for s in volume.spacing)
    v = _Volume()
    v.nx, v.ny, v.nz = W, H, D
    v.dx, v.dy, v.dz = dx, dy, dz
    v.ox, v.oy, v.oz = (float(s) for s in volume.origin)
    h = ctypes.c_void_p()
    if opts is None:
        _check(lib.ctp_plan(ctypes.byref(g), ctypes.byref(v), PATHS[path], ctypes.byref(h)),
               "ctp_plan")
    else:
        _check(lib.ctp_plan_ex(ctypes.byref(g), ctypes.byref(v), PATHS[path], ctypes.byref(opts),
                               ctypes.byref(h)), "ctp_plan_ex")
    geometry = dataclasses.replace(geometry, src=arrays[0], det_centre=arrays[1],
                                   det_u=arrays[2], det_v=arrays[3], pixel_offsets=offsets)
    return Plan(h.value, geometry, volume)


def _stream_ptr(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _device_f32(t, shape, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError(f"{name} must be a float32 CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != int(np.prod(shape)):
        raise ValueError(f"{name} must hold {shape} elements, got {tuple(t.shape)}")
    return t.data_ptr()


def ctp_forward(plan: Plan, vol, sino, stream=None):
    """sino <- A vol (both float32 CUDA tensors; sino fully overwritten)."""
    _check(load_library().ctp_forward(plan.handle, _device_f32(vol, plan.vol_shape, "vol"),
                                      _device_f32(sino, plan.sino_shape, "sino"),
                                      _stream_ptr(stream)), "ctp_forward")
    return sino


def ctp_backward(plan: Plan, sino, vol, stream=None):
    """vol <- A^T sino (vol fully overwritten)."""
    _check(load_library().ctp_backward(plan.handle, _device_f32(sino, plan.sino_shape, "sino"),
                                       _device_f32(vol, plan.vol_shape, "vol"),
                                       _stream_ptr(stream)), "ctp_backward")
    return vol


def ctp_segment_count(plan: Plan, stream=None) -> int:
    out = ctypes.c_ulonglong(0)
    _check(load_library().ctp_segment_count(plan.handle, ctypes.byref(out), _stream_ptr(stream)),
           "ctp_segment_count")
    return int(out.value)


def ctp_check_violations() -> tuple[int, int, int, int]:
    """(count, first index, its buffer's extent, access site) of the out-of-range
    accesses since the previous call, in the bounds-checked build; resets them.
    Raises CtpError (CTP_E_OPTION) in normal builds."""
    c, i, e, site = ctypes.c_ulonglong(0), ctypes.c_longlong(0), ctypes.c_longlong(0), ctypes.c_int(0)
    _check(load_library().ctp_check_violations(ctypes.byref(c), ctypes.byref(i), ctypes.byref(e),
                                               ctypes.byref(site)), "ctp_check_violations")
    return int(c.value), int(i.value), int(e.value), int(site.value)


def _host_f32(a, shape, name, writable=False):
    if not isinstance(a, np.ndarray) or a.dtype != np.float32 or not a.flags.c_contiguous:
        raise TypeError(f"{name} must be a C-contiguous float32 numpy array")
    if a.size != int(np.prod(shape)):
        raise ValueError(f"{name} must hold {shape} elements")
    if writable and not a.flags.writeable:
        raise ValueError(f"{name} must be writable")
    return a.ctypes.data


def ctp_forward_host(plan: Plan, vol_host, sino_host, stream=None):
    """End to end: host vol -> device -> A -> host sino (waits for the stream)."""
    _check(load_library().ctp_forward_host(
        plan.handle, _host_f32(vol_host, plan.vol_shape, "vol_host"),
        _host_f32(sino_host, plan.sino_shape, "sino_host", True), _stream_ptr(stream)),
        "ctp_forward_host")
    return sino_host


def ctp_backward_host(plan: Plan, sino_host, vol_host, stream=None):
    _check(load_library().ctp_backward_host(
        plan.handle, _host_f32(sino_host, plan.sino_shape, "sino_host"),
        _host_f32(vol_host, plan.vol_shape, "vol_host", True), _stream_ptr(stream)),
        "ctp_backward_host")
    return vol_host


def ctp_destroy(plan: Plan):
    plan.destroy()


# --------------------------------------------------------------- analytical operators
def _view_weight(plan: Plan, view_weight):
    if view_weight is None:
        return None
    return _device_f32(view_weight, (plan.sino_shape[0],), "view_weight")


def _pixel_weight(plan: Plan, pixel_weight):
    if pixel_weight is None:
        return None
    return _device_f32(pixel_weight, (plan.sino_shape[0], plan.sino_shape[2]), "pixel_weight")


def ctp_ramp_filter(plan: Plan, sino, out, view_weight=None, ramp: str = "ramlak",
                    transpose: bool = False, stream=None, pixel_weight=None):
    """out <- ramp filter along u of the cosine- (and pixel-) weighted sino, times
    the view weights (transpose: the transposed operator).  ``out`` may be
    ``sino``.  pixel_weight: (n_views, n_u), e.g. :func:`ctp_parker_weights`."""
    _check(load_library().ctp_ramp_filter(
        plan.handle, _device_f32(sino, plan.sino_shape, "sino"),
        _device_f32(out, plan.sino_shape, "out"), _view_weight(plan, view_weight),
        _pixel_weight(plan, pixel_weight), RAMPS[ramp], int(bool(transpose)),
        _stream_ptr(stream)), "ctp_ramp_filter")
    return out


def ctp_weighted_backproject(plan: Plan, sino, vol, stream=None):
    """vol <- voxel-driven weighted gather of (filtered) sino (vol overwritten)."""
    _check(load_library().ctp_weighted_backproject(
        plan.handle, _device_f32(sino, plan.sino_shape, "sino"),
        _device_f32(vol, plan.vol_shape, "vol"), _stream_ptr(stream)),
        "ctp_weighted_backproject")
    return vol


def ctp_weighted_backproject_transpose(plan: Plan, vol, sino, stream=None):
    """sino <- transpose of the weighted gather applied to vol (sino overwritten)."""
    _check(load_library().ctp_weighted_backproject_transpose(
        plan.handle, _device_f32(vol, plan.vol_shape, "vol"),
        _device_f32(sino, plan.sino_shape, "sino"), _stream_ptr(stream)),
        "ctp_weighted_backproject_transpose")
    return sino


def ctp_fdk(plan: Plan, sino, work, vol, view_weight=None, ramp: str = "ramlak", stream=None,
            pixel_weight=None):
    """vol <- FBP / FDK of sino: ramp filter into ``work`` (may be ``sino``), then the
    weighted gather."""
    _check(load_library().ctp_fdk(
        plan.handle, _device_f32(sino, plan.sino_shape, "sino"),
        _device_f32(work, plan.sino_shape, "work"), _device_f32(vol, plan.vol_shape, "vol"),
        _view_weight(plan, view_weight), _pixel_weight(plan, pixel_weight), RAMPS[ramp],
        _stream_ptr(stream)), "ctp_fdk")
    return vol


def ctp_parker_weights(plan: Plan, out=None, stream=None):
    """Parker short-scan weights (n_views, n_u) as a float32 CUDA tensor; use with
    view weights equal to the angular step."""
    import torch
    shape = (plan.sino_shape[0], plan.sino_shape[2])
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=torch.device("cuda", plan.device))
    _check(load_library().ctp_parker_weights(plan.handle, _device_f32(out, shape, "out"),
                                             _stream_ptr(stream)), "ctp_parker_weights")
    return out


def full_scan_view_weights(n_views: int):
    """View weights of a full 2 pi scan with equally spaced views: pi / n_views
    (the angular step, halved because every line is measured twice)."""
    return np.full(int(n_views), np.pi / max(int(n_views), 1), dtype=np.float32)


# ------------------------------------------------------------ geometry gradients
def ctp_geometry_vjp(plan: Plan, vol, weight, grad=None, stream=None):
    """grad[s] = sum over view s's rays of weight[ray] * d (A vol)[ray] / d frame[s],
    as a float64 CUDA tensor (n_views, 4, 3): src, det_centre, det_u, det_v."""
    import torch
    n_views = plan.sino_shape[0]
    if grad is None:
        grad = torch.empty((n_views, 4, 3), dtype=torch.float64, device=vol.device)
    if not (isinstance(grad, torch.Tensor) and grad.is_cuda and grad.dtype == torch.float64
            and grad.is_contiguous() and grad.numel() == 12 * n_views):
        raise TypeError("grad must be a contiguous float64 CUDA tensor of n_views * 12 elements")
    _check(load_library().ctp_geometry_vjp(
        plan.handle, _device_f32(vol, plan.vol_shape, "vol"),
        _device_f32(weight, plan.sino_shape, "weight"), grad.data_ptr(), _stream_ptr(stream)),
        "ctp_geometry_vjp")
    return grad


def ctp_surface_vjp(plan: Plan, vol, weight, grad=None, stream=None):
    """grad[iv, iu, m] = sum over views of weight[view, iv, iu] * d (A vol)[ray] / d
    offset_m of pixel (iu, iv), offsets (t, s, e) along det_u, det_v and the unit
    normal: a float64 CUDA tensor (n_v, n_u, 3); with one offset table per view
    (n_views, n_v, n_u, 3), each view's pixel its own gradient."""
    import torch
    per_view = plan.geometry.pixel_offsets is not None and plan.geometry.pixel_offsets.ndim == 4
    shape = ((plan.sino_shape[0],) if per_view else ()) + (plan.sino_shape[1],
                                                           plan.sino_shape[2], 3)
    if grad is None:
        grad = torch.empty(shape, dtype=torch.float64, device=vol.device)
    if not (isinstance(grad, torch.Tensor) and grad.is_cuda and grad.dtype == torch.float64
            and grad.is_contiguous() and grad.numel() == int(np.prod(shape))):
        raise TypeError(f"grad must be a contiguous float64 CUDA tensor of {shape} elements")
    _check(load_library().ctp_surface_vjp(
        plan.handle, _device_f32(vol, plan.vol_shape, "vol"),
        _device_f32(weight, plan.sino_shape, "weight"), grad.data_ptr(), _stream_ptr(stream)),
        "ctp_surface_vjp")
    return grad
