"""Curved detectors (per-pixel offsets) on the GPU against the float64 oracle:
the projector pair on a cylindrical detector, the pitch grid written as offsets,
and the calls that refuse curved detectors."""

import numpy as np
import pytest

from cases import TOL_BACKWARD, TOL_FORWARD, ci, rel_l2
from test_oracle_curved_pins import _cylinder_offsets, _flat_offsets

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as _torch
    assert _torch.cuda.is_available(), "CUDA device required"
    return _torch


@pytest.fixture(scope="module")
def ctp():
    import back_projection_ctp_b300 as _ctp
    _ctp.load_library()
    return _ctp


def _cone_scan(oracle_mod, ctp, off, n_u, n_v, pu=1.0, pv=1.0, ou=0.0, ov=0.0, K=24):
    w = ci.small_cases()[3]
    f = ci.frames(ci.scaled(w, 1.0, views=K, ragged=0))
    shape, spacing, origin = w.shape, w.spacing, w.origin
    scan = oracle_mod.Scan("divergent", f["src"], f["det_centre"], f["det_u"], f["det_v"], n_u,
                           n_v, pu, pv, shape, spacing, origin, ou, ov, 3, off)
    g = ctp.Geometry(ndim=3, beam="divergent", n_u=n_u, n_v=n_v, pitch_u=pu, pitch_v=pv,
                     offset_u=ou, offset_v=ov, pixel_offsets=off, **f)
    return w, scan, g, ctp.Volume(shape, spacing, origin)


def _pair(torch, ctp, plan, vol, y):
    d_s = torch.empty(plan.sino_shape, device="cuda")
    ctp.ctp_forward(plan, torch.from_numpy(vol).cuda(), d_s)
    d_g = torch.empty(plan.vol_shape, device="cuda")
    ctp.ctp_backward(plan, torch.from_numpy(y).cuda(), d_g)
    torch.cuda.synchronize()
    return d_s.cpu().numpy(), d_g.cpu().numpy()


@pytest.mark.parametrize("path", ["auto", "ray"])
def test_cylindrical_detector_matches_oracle(torch, ctp, oracle_mod, path):
    """A cylindrical detector (columns straight and vertical, rows evenly spaced)
    takes the column path under AUTO; both paths match the oracle."""
    off = _cylinder_offsets(53, 41, 1000.0, 0.0094, 9.4)
    w, scan, g, v = _cone_scan(oracle_mod, ctp, off, 53, 41)
    plan = ctp.ctp_plan(g, v, path)
    assert plan.path == ("column" if path == "auto" else "ray")
    vol = ci.phantom(w)
    amb = oracle_mod.ambiguous(scan)
    y = np.where(amb, np.float32(0),
                 np.random.default_rng(7).standard_normal(scan.sino_shape).astype(np.float32))
    p, gg = _pair(torch, ctp, plan, vol, y)
    p_ref = oracle_mod.forward(scan, vol).reshape(scan.sino_shape)
    assert rel_l2(p[~amb], p_ref[~amb]) <= TOL_FORWARD
    assert rel_l2(gg, oracle_mod.backward(scan, y.ravel())) <= TOL_BACKWARD
    assert abs(ctp.ctp_segment_count(plan) - oracle_mod.segment_count(scan)) <= \
        1e-6 * oracle_mod.segment_count(scan)


def test_irregular_curved_detector_takes_the_ray_path(torch, ctp, oracle_mod):
    """Tangent offsets that vary down a column: no column structure, so AUTO takes
    the ray path and an explicit column request is refused; the ray path matches
    the oracle."""
    off = _cylinder_offsets(31, 25, 1000.0, 0.015, 12.0)
    off[:, :, 0] += np.linspace(-3.0, 3.0, 25, dtype=np.float32)[:, None]
    w, scan, g, v = _cone_scan(oracle_mod, ctp, off, 31, 25)
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_plan(g, v, "column")
    assert e.value.status == 11
    plan = ctp.ctp_plan(g, v)
    assert plan.path == "ray"
    vol = ci.phantom(w)
    amb = oracle_mod.ambiguous(scan)
    y = np.where(amb, np.float32(0),
                 np.random.default_rng(9).standard_normal(scan.sino_shape).astype(np.float32))
    p, gg = _pair(torch, ctp, plan, vol, y)
    p_ref = oracle_mod.forward(scan, vol).reshape(scan.sino_shape)
    assert rel_l2(p[~amb], p_ref[~amb]) <= TOL_FORWARD
    assert rel_l2(gg, oracle_mod.backward(scan, y.ravel())) <= TOL_BACKWARD


def test_flat_offsets_equal_the_flat_plan(torch, ctp, oracle_mod):
    off = _flat_offsets(49, 49, 9.5, 9.25, 0.5, -0.25)
    w, scan, g, v = _cone_scan(oracle_mod, ctp, off, 49, 49)
    flat = ctp.Geometry(ndim=3, beam="divergent", src=g.src, det_centre=g.det_centre,
                        det_u=g.det_u, det_v=g.det_v, n_u=49, n_v=49, pitch_u=9.5,
                        pitch_v=9.25, offset_u=0.5, offset_v=-0.25)
    vol = ci.phantom(w)
    y = np.random.default_rng(8).standard_normal(scan.sino_shape).astype(np.float32)
    p_c, g_c = _pair(torch, ctp, ctp.ctp_plan(g, v), vol, y)
    p_f, g_f = _pair(torch, ctp, ctp.ctp_plan(flat, v, "ray"), vol, y)
    assert rel_l2(p_c, p_f) <= 1e-6
    assert rel_l2(g_c, g_f) <= 1e-6


def test_calls_that_refuse_curved_detectors(torch, ctp, oracle_mod):
    off = _cylinder_offsets(9, 7, 1000.0, 0.0094, 9.4)
    w, scan, g, v = _cone_scan(oracle_mod, ctp, off, 9, 7, K=3)
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_plan(g, v, "plane")
    assert e.value.status == 11
    plan = ctp.ctp_plan(g, v)
    vol = torch.zeros(plan.vol_shape, device="cuda")
    sino = torch.zeros(plan.sino_shape, device="cuda")
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_weighted_backproject(plan, sino, vol)
    assert e.value.status == 13
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_geometry_vjp(plan, vol, sino)
    assert e.value.status == 11
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_forward_static(g, v, vol, sino)
    assert e.value.status == 11
    bad = np.array(off)
    bad[0, 0, 2] = np.nan
    import dataclasses
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_plan(dataclasses.replace(g, pixel_offsets=bad), v)
    assert e.value.status == 3
