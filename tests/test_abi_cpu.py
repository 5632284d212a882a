"""CPU-side checks of the C ABI library: it builds, loads, exports every symbol
that include/ctp.h declares, and rejects invalid scans on the host (validation
runs before any CUDA call, so no GPU is needed for these)."""

import ctypes
import os
import re

import numpy as np
import pytest

import back_projection_ctp_b300 as ctp
from back_projection_ctp_b300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "ctp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ctp_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = ctp.load_library()
    declared = _declared()
    assert "ctp_plan" in declared and "ctp_forward" in declared and "ctp_backward" in declared
    for name in declared:
        assert hasattr(lib, name), name
    # the binding covers every entry point the header declares, and nothing else
    assert sorted(B.EXPORTS) == declared


def test_status_strings():
    assert ctp.ctp_status_string(0) == "ok"
    assert "finite" in ctp.ctp_status_string(3)
    assert "must differ" in ctp.ctp_status_string(4)
    assert "1e6" in ctp.ctp_status_string(5)
    assert "1e15" in ctp.ctp_status_string(6)
    assert ctp.ctp_status_string(999) == "unknown status"


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(OSError):
        ctypes.CDLL(str(tmp_path / "libctp.so"))


def _cone(n_views=3):
    b = np.linspace(0, 2 * np.pi, n_views, endpoint=False)
    c, s, z = np.cos(b), np.sin(b), np.zeros_like(b)
    f = dict(src=np.stack([600 * c, 600 * s, z], 1), det_centre=np.stack([-400 * c, -400 * s, z], 1),
             det_u=np.stack([-s, c, z], 1), det_v=np.stack([z, z, z + 1], 1))
    return {k: v.astype(np.float32) for k, v in f.items()}


def _plan_status(frames=None, ndim=3, beam="divergent", shape=(8, 8, 8), spacing=(1.0, 1.0, 1.0),
                 n_u=8, n_v=8, pitch=(1.0, 1.0), path="auto"):
    frames = frames or _cone()
    g = ctp.Geometry(ndim=ndim, beam=beam, n_u=n_u, n_v=n_v, pitch_u=pitch[0], pitch_v=pitch[1],
                     **frames)
    D, H, W = shape
    origin = (-0.5 * W * spacing[2], -0.5 * H * spacing[1], -0.5 * D * spacing[0])
    try:
        ctp.ctp_plan(g, ctp.Volume(shape, spacing, origin), path)
    except ctp.CtpError as e:
        return e.status
    return 0


@pytest.mark.parametrize("failure,status,message", [
    ("nonfinite", 3, "finite"), ("coincident", 4, "must differ"),
    ("near", 5, "1e6"), ("far", 6, "1e15"),
])
def test_validation_error_set(failure, status, message):
    f = _cone()
    if failure == "nonfinite":
        f["src"][1, 0] = np.nan
    elif failure == "coincident":
        f["det_centre"][2] = f["src"][2]
    elif failure == "near":
        f["src"][0] *= 1e5
    elif failure == "far":
        f["src"][0] *= 1e13
    assert _plan_status(f) == status
    assert message in ctp.ctp_status_string(status)


@pytest.mark.parametrize("spacing,ok", [
    ((1.0, 1.0, 1.0), True), ((1e-6, 1e-6, 1e-6), True), ((1e-7, 1.0, 1.0), False),
    ((2e6, 1.0, 1.0), False), ((1.0, 1.0, 1e4), True), ((1.0, 1.0, 1.01e4), False),
])
def test_spacing_bounds(spacing, ok):
    st = _plan_status(spacing=spacing)
    if ok:
        assert st != 7
    else:
        assert st == 7


def test_shape_and_option_errors():
    assert _plan_status(shape=(0, 8, 8)) == 2
    assert _plan_status(n_u=0) == 2
    assert _plan_status(ndim=4) == 11
    assert _plan_status(ndim=2, n_v=2, shape=(1, 8, 8)) == 2
    f = _cone()
    f["det_v"][0] = f["det_u"][0]
    assert _plan_status(f) == 8
    f = _cone()
    f["det_u"][1] = 0
    assert _plan_status(f) == 8
    with pytest.raises(KeyError):
        _plan_status(path="sideways")


@pytest.mark.parametrize("options", [
    {"rows_forward": 5}, {"rows_backward": -1}, {"backward_rows_adjacent": 2},
    {"plane_backward": 3}, {"host_chunks": 65}, {"geometry_walk": 2}, {"forward_ahead": 3},
    {"forward_views_first": -1},
])
def test_plan_options_out_of_range_are_rejected_on_the_host(options):
    """ctp_plan_ex checks its work-layout options before any CUDA call."""
    f = _cone()
    g = ctp.Geometry(ndim=3, beam="divergent", n_u=8, n_v=8, pitch_u=1.0, pitch_v=1.0, **f)
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_plan(g, ctp.Volume((8, 8, 8), (1.0, 1.0, 1.0), (-4.0, -4.0, -4.0)),
                     options=options)
    assert e.value.status == 11
    with pytest.raises(ValueError):
        ctp.ctp_plan(g, ctp.Volume((8, 8, 8), (1.0, 1.0, 1.0), (-4.0, -4.0, -4.0)),
                     options={"colour": 1})


def test_library_reads_no_environment():
    """Work layouts are plan options, not process-wide variables: the library's
    sources call no getenv."""
    csrc = os.path.join(ROOT, "back_projection_ctp_b300", "csrc")
    for name in os.listdir(csrc):
        with open(os.path.join(csrc, name)) as fh:
            assert "getenv" not in fh.read(), name


def test_curved_detector_offsets_are_validated_on_the_host():
    f = _cone()
    off = np.zeros((8, 8, 3), np.float32)
    off[3, 4, 2] = np.inf
    g = ctp.Geometry(ndim=3, beam="divergent", n_u=8, n_v=8, pitch_u=1.0, pitch_v=1.0,
                     pixel_offsets=off, **f)
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_plan(g, ctp.Volume((8, 8, 8), (1.0, 1.0, 1.0), (-4.0, -4.0, -4.0)))
    assert e.value.status == 3
    with pytest.raises(ValueError):
        ctp.ctp_plan(ctp.Geometry(ndim=3, beam="divergent", n_u=8, n_v=8, pitch_u=1.0,
                                  pitch_v=1.0, pixel_offsets=np.zeros((7, 8, 3), np.float32),
                                  **f), ctp.Volume((8, 8, 8), (1.0, 1.0, 1.0), (-4.0, -4.0, -4.0)))


def test_parallel_direction_along_detector_is_rejected():
    f = _cone()
    f["src"] = f["det_u"].copy()  # ray direction lying in the detector plane
    assert _plan_status(f, beam="parallel") == 4


def test_normal_build_has_no_access_counters():
    """ctp_check_violations answers CTP_E_OPTION (outputs zeroed) unless the
    library was compiled with CTP_CHECK; no device is needed for the answer."""
    if os.environ.get("CTP_LIBRARY_VARIANT") == "check":
        pytest.skip("running against the checked library")
    lib = B.load_library()
    c, i, e, s = ctypes.c_ulonglong(7), ctypes.c_longlong(7), ctypes.c_longlong(7), ctypes.c_int(7)
    st = lib.ctp_check_violations(ctypes.byref(c), ctypes.byref(i), ctypes.byref(e), ctypes.byref(s))
    assert st == 11 and (c.value, i.value, e.value, s.value) == (0, 0, 0, 0)
    assert lib.ctp_check_violations(None, ctypes.byref(i), ctypes.byref(e), ctypes.byref(s)) == 1
    with pytest.raises(ctp.CtpError):
        ctp.ctp_check_violations()
