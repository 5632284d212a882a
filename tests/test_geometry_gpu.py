"""GPU parity of the geometry gradients (``ctp_geometry_vjp``, through the C ABI)
against the float64 oracle's ``geometry_vjp``.

Bar: relative L2 over every view's twelve components <= 1e-4 (float32 values
and per-ray sums, float64 per-view sums).  Rays lying in a cell-face plane
(ambiguous path sums) and rays through a cell edge or corner (kinks of the path
sum, where the value jump may go to either coincident crossing) get weight 0 on
both sides; the symmetric synthetic scans hit such rays systematically (about
2 % of the rays of the reduced 256^3 cone scan).
"""

import numpy as np
import pytest

from cases import ci, geometry_of, rel_l2, volume_of

pytestmark = pytest.mark.gpu

TOL_GEOMETRY = 1e-4
SMALL = ci.small_cases()


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


def _weights(oracle_mod, scan, seed):
    w = np.random.default_rng(seed).standard_normal(scan.n_rays).astype(np.float32)
    skip = oracle_mod.ambiguous(scan).ravel() | oracle_mod.kinks(scan).ravel()
    return np.where(skip, np.float32(0), w)


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("walk", ["auto", "ray"])
def test_small_cases_match_oracle(torch, ctp, oracle_mod, idx, walk):
    """AUTO runs the column walk on the 3-D circular / helical scans and the ray
    walk elsewhere; the plan option geometry_walk = "ray" forces the ray walk."""
    w = SMALL[idx]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), options={"geometry_walk": walk})
    vol = ci.phantom(w)
    wt = _weights(oracle_mod, scan, 50 + idx)
    g = ctp.ctp_geometry_vjp(plan, torch.from_numpy(vol).cuda(),
                             torch.from_numpy(wt.reshape(plan.sino_shape)).cuda())
    torch.cuda.synchronize()
    ref = oracle_mod.geometry_vjp(scan, vol, wt)
    assert rel_l2(g.cpu().numpy(), ref) <= TOL_GEOMETRY


@pytest.mark.parametrize("beam", ["divergent", "parallel"])
def test_tilted_frames_and_random_volume(torch, ctp, oracle_mod, beam):
    import geom_helpers
    rng = np.random.default_rng(60 if beam == "divergent" else 61)
    frames = geom_helpers.random_frames(rng, 5, beam, radius=30.0, det_dist=25.0, tilt=0.4)
    shape, spacing = (9, 11, 10), (1.1, 0.9, 1.3)
    origin = (-0.5 * 10 * 1.3, -0.5 * 11 * 0.9, -0.5 * 9 * 1.1)
    scan = oracle_mod.Scan(beam, *frames, 23, 19, 1.4, 1.2, shape, spacing, origin, 0.4, -0.3)
    g_ = ctp.Geometry(ndim=3, beam=beam, src=frames[0], det_centre=frames[1], det_u=frames[2],
                      det_v=frames[3], n_u=23, n_v=19, pitch_u=1.4, pitch_v=1.2, offset_u=0.4,
                      offset_v=-0.3)
    plan = ctp.ctp_plan(g_, ctp.Volume(shape, spacing, origin))
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    wt = _weights(oracle_mod, scan, 62)
    g = ctp.ctp_geometry_vjp(plan, torch.from_numpy(vol).cuda(),
                             torch.from_numpy(wt.reshape(plan.sino_shape)).cuda())
    torch.cuda.synchronize()
    assert rel_l2(g.cpu().numpy(), oracle_mod.geometry_vjp(scan, vol, wt)) <= TOL_GEOMETRY


def test_source_inside_the_volume(torch, ctp, oracle_mod):
    """Rays that start inside the grid: their start is not a plane crossing."""
    K = 8
    b = np.arange(K) * 2 * np.pi / K
    c, s, z, o = np.cos(b), np.sin(b), np.zeros(K), np.ones(K)
    fr = [np.stack(x, 1).astype(np.float32) for x in ((3 * c, 3 * s, z + 0.3),
                                                     (-20 * c, -20 * s, z),
                                                     (-s, c, z), (z, z, o))]
    shape, spacing = (7, 12, 13), (1.0, 1.0, 1.0)
    origin = (-6.5, -6.0, -3.5)
    scan = oracle_mod.Scan("divergent", *fr, 17, 9, 1.3, 1.1, shape, spacing, origin, 0.2, 0.1)
    g_ = ctp.Geometry(ndim=3, beam="divergent", src=fr[0], det_centre=fr[1], det_u=fr[2],
                      det_v=fr[3], n_u=17, n_v=9, pitch_u=1.3, pitch_v=1.1, offset_u=0.2,
                      offset_v=0.1)
    plan = ctp.ctp_plan(g_, ctp.Volume(shape, spacing, origin), "ray")
    vol = np.random.default_rng(63).uniform(0, 1, shape).astype(np.float32)
    wt = _weights(oracle_mod, scan, 64)
    g = ctp.ctp_geometry_vjp(plan, torch.from_numpy(vol).cuda(),
                             torch.from_numpy(wt.reshape(plan.sino_shape)).cuda())
    torch.cuda.synchronize()
    assert rel_l2(g.cpu().numpy(), oracle_mod.geometry_vjp(scan, vol, wt)) <= TOL_GEOMETRY


@pytest.mark.parametrize("idx", [3, 4])
def test_full_size_sampled_views(torch, ctp, oracle_mod, idx):
    """Full-size scans: weights on two views only; those views' gradients against
    the oracle, every other view exactly zero."""
    w = ci.WORKLOADS[idx]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w))
    rng = np.random.default_rng(80 + idx)
    views = np.sort(rng.choice(w.n_views, 2, replace=False))
    per = w.n_u * w.n_v
    wt = np.zeros(scan.n_rays, np.float32)
    for v in views:
        wt[v * per:(v + 1) * per] = rng.standard_normal(per).astype(np.float32)
    sub = oracle_mod.Scan(w.beam, *(a[views] for a in scan.arrays), w.n_u, w.n_v, w.pitch_u,
                          w.pitch_v, w.shape, w.spacing, w.origin, w.offset_u, w.offset_v, w.ndim)
    sub_w = np.concatenate([wt[v * per:(v + 1) * per] for v in views])
    skip = oracle_mod.ambiguous(sub).ravel() | oracle_mod.kinks(sub).ravel()
    sub_w = np.where(skip, np.float32(0), sub_w)
    for q, v in enumerate(views):
        wt[v * per:(v + 1) * per] = sub_w[q * per:(q + 1) * per]
    vol = ci.phantom(w)
    g = ctp.ctp_geometry_vjp(plan, torch.from_numpy(vol).cuda(),
                             torch.from_numpy(wt.reshape(plan.sino_shape)).cuda())
    torch.cuda.synchronize()
    g = g.cpu().numpy()
    ref = oracle_mod.geometry_vjp(sub, vol, sub_w)
    assert rel_l2(g[views], ref) <= TOL_GEOMETRY
    others = np.setdiff1d(np.arange(w.n_views), views)
    assert np.abs(g[others]).max() == 0.0


def test_empty_scan(torch, ctp):
    z = np.zeros((0, 3), np.float32)
    g_ = ctp.Geometry(ndim=3, beam="divergent", src=z, det_centre=z, det_u=z, det_v=z, n_u=4,
                      n_v=4, pitch_u=1.0, pitch_v=1.0)
    plan = ctp.ctp_plan(g_, ctp.Volume((3, 4, 5), (1.0, 1.0, 1.0), (-2.5, -2.0, -1.5)))
    out = torch.empty((0, 4, 3), dtype=torch.float64, device="cuda")
    ctp.ctp_geometry_vjp(plan, torch.zeros((3, 4, 5), device="cuda"),
                         torch.zeros((0, 4, 4), device="cuda"), out)
