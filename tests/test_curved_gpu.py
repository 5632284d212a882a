"""Curved detectors (per-pixel offsets) on the GPU against the float64 oracle:
the projector pair on a cylindrical detector, the pitch grid written as offsets,
the geometry and surface gradients, and the calls that refuse curved
detectors."""

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
        ctp.ctp_forward_static(g, v, vol, sino)
    assert e.value.status == 11
    bad = np.array(off)
    bad[0, 0, 2] = np.nan
    import dataclasses
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_plan(dataclasses.replace(g, pixel_offsets=bad), v)
    assert e.value.status == 3


# ------------------------------------------------------------- gradients
TOL_GEOMETRY = 1e-4   # as for flat detectors (float32 per-ray sums, float64 totals)


def _grad_weights(oracle_mod, scan, seed):
    w = np.random.default_rng(seed).standard_normal(scan.n_rays).astype(np.float32)
    skip = oracle_mod.ambiguous(scan).ravel() | oracle_mod.kinks(scan).ravel()
    return np.where(skip, np.float32(0), w)


def _curved_cases():
    cyl = _cylinder_offsets(41, 33, 1000.0, 0.0094, 9.4)
    irregular = _cylinder_offsets(31, 25, 1000.0, 0.015, 12.0)
    irregular[:, :, 0] += np.linspace(-3.0, 3.0, 25, dtype=np.float32)[:, None]
    irregular[:, :, 2] += np.linspace(-5.0, 5.0, 31, dtype=np.float32)[None, :]
    return {"cylinder": (cyl, 41, 33), "irregular": (irregular, 31, 25)}


@pytest.mark.parametrize("case", ["cylinder", "irregular"])
def test_curved_geometry_vjp_matches_oracle(torch, ctp, oracle_mod, case):
    """Frame gradients on curved detectors (the u / v gradients carry the
    normal's derivative), on the ray walk whatever the plan's path."""
    off, n_u, n_v = _curved_cases()[case]
    w, scan, g, v = _cone_scan(oracle_mod, ctp, off, n_u, n_v, K=12)
    plan = ctp.ctp_plan(g, v)
    vol = ci.phantom(w)
    wt = _grad_weights(oracle_mod, scan, 91)
    grad = ctp.ctp_geometry_vjp(plan, torch.from_numpy(vol).cuda(),
                                torch.from_numpy(wt.reshape(plan.sino_shape)).cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.geometry_vjp(scan, vol, wt)
    assert rel_l2(grad.cpu().numpy(), ref) <= TOL_GEOMETRY
    # every part of the frame has a gradient (the u / v rows are not the flat chain)
    assert np.abs(ref[:, 2:]).max() > 0


@pytest.mark.parametrize("case", ["cylinder", "irregular", "flat"])
def test_surface_vjp_matches_oracle(torch, ctp, oracle_mod, case):
    """Gradients with respect to every pixel's offsets along u, v and the normal,
    summed over views; flat detectors take their pitch grid."""
    if case == "flat":
        w = ci.small_cases()[3]
        from cases import geometry_of, volume_of
        f = ci.frames(w)
        scan = oracle_mod.Scan.from_workload(w, f)
        g, v = geometry_of(w, f), volume_of(w)
    else:
        off, n_u, n_v = _curved_cases()[case]
        w, scan, g, v = _cone_scan(oracle_mod, ctp, off, n_u, n_v, K=12)
    plan = ctp.ctp_plan(g, v)
    vol = ci.phantom(w)
    wt = _grad_weights(oracle_mod, scan, 92)
    grad = ctp.ctp_surface_vjp(plan, torch.from_numpy(vol).cuda(),
                               torch.from_numpy(wt.reshape(plan.sino_shape)).cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.surface_vjp(scan, vol, wt)
    assert grad.shape == ref.shape == (scan.n_v, scan.n_u, 3)
    assert rel_l2(grad.cpu().numpy(), ref) <= TOL_GEOMETRY


# ------------------------------------------------------ one offset table per view
def _per_view_tables(K, n_u, n_v, columnar):
    """K tables: cylinders whose radius changes from view to view (columns stay
    straight: the column path), or the same with a per-view tangent shear down
    the columns (the ray path)."""
    tabs = []
    for k in range(K):
        t = _cylinder_offsets(n_u, n_v, 800.0 + 40.0 * k, 0.0118, 11.8)
        if not columnar:
            t[:, :, 0] += np.linspace(-1.0, 1.0, n_v, dtype=np.float32)[:, None] * (1 + k % 3)
        tabs.append(t)
    return np.stack(tabs).astype(np.float32)


@pytest.mark.parametrize("columnar", [True, False])
def test_per_view_offsets_match_oracle(torch, ctp, oracle_mod, columnar):
    K, n_u, n_v = 12, 37, 29
    off = _per_view_tables(K, n_u, n_v, columnar)
    w, scan, g, v = _cone_scan(oracle_mod, ctp, off, n_u, n_v, K=K)
    assert scan.offsets_per_view
    plan = ctp.ctp_plan(g, v)
    assert plan.path == ("column" if columnar else "ray")
    vol = ci.phantom(w)
    amb = oracle_mod.ambiguous(scan)
    y = np.where(amb, np.float32(0),
                 np.random.default_rng(13).standard_normal(scan.sino_shape).astype(np.float32))
    p, gg = _pair(torch, ctp, plan, vol, y)
    p_ref = oracle_mod.forward(scan, vol).reshape(scan.sino_shape)
    assert rel_l2(p[~amb], p_ref[~amb]) <= TOL_FORWARD
    assert rel_l2(gg, oracle_mod.backward(scan, y.ravel())) <= TOL_BACKWARD
    n_ref = oracle_mod.segment_count(scan)
    assert abs(ctp.ctp_segment_count(plan) - n_ref) <= max(1e-6 * n_ref, 4)
    # each view's rays are those of a one-view plan with that view's table
    k = K // 2
    import dataclasses
    one = dataclasses.replace(g, src=g.src[k:k + 1], det_centre=g.det_centre[k:k + 1],
                              det_u=g.det_u[k:k + 1], det_v=g.det_v[k:k + 1],
                              pixel_offsets=off[k])
    p1, _ = _pair(torch, ctp, ctp.ctp_plan(one, v), vol, y[k:k + 1])
    assert rel_l2(p1[0], p[k]) <= 1e-6


def test_per_view_gradients_match_oracle(torch, ctp, oracle_mod):
    K, n_u, n_v = 8, 29, 23
    off = _per_view_tables(K, n_u, n_v, False)
    w, scan, g, v = _cone_scan(oracle_mod, ctp, off, n_u, n_v, K=K)
    plan = ctp.ctp_plan(g, v)
    vol = ci.phantom(w)
    wt = _grad_weights(oracle_mod, scan, 93)
    d_vol = torch.from_numpy(vol).cuda()
    d_w = torch.from_numpy(wt.reshape(plan.sino_shape)).cuda()
    s_grad = ctp.ctp_surface_vjp(plan, d_vol, d_w)
    g_grad = ctp.ctp_geometry_vjp(plan, d_vol, d_w)
    torch.cuda.synchronize()
    s_ref = oracle_mod.surface_vjp(scan, vol, wt)
    assert s_grad.shape == s_ref.shape == (K, n_v, n_u, 3)
    assert rel_l2(s_grad.cpu().numpy(), s_ref) <= TOL_GEOMETRY
    assert rel_l2(g_grad.cpu().numpy(), oracle_mod.geometry_vjp(scan, vol, wt)) <= TOL_GEOMETRY
