"""GPU parity of the analytical FBP / FDK operators (through the C ABI) against the
float64 oracle ``oracle/fdk.py``.

Bars: ramp filter, weighted gather and the whole FDK within relative L2 1e-5
(float32 data and accumulation, coordinates exact to ~1e-7 pixel); the gather's
transpose within 1e-4 (float32 atomics, order-dependent); the GPU pair's own
adjoint identity within 1e-5 (Cauchy-Schwarz normalised).
"""

import math

import numpy as np
import pytest

from cases import TOL_ADJOINT, adjoint_mismatch, ci, geometry_of, rel_l2, volume_of

pytestmark = pytest.mark.gpu

TOL_GATHER = 1e-5
TOL_FILTER = 1e-5
TOL_SCATTER = 1e-4
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


@pytest.fixture(scope="module")
def ofdk(oracle_mod):
    from oracle import fdk as _fdk
    return _fdk


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _case(idx):
    w = SMALL[idx]
    f = ci.frames(w)
    return w, f


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_small_cases_match_oracle(torch, ctp, oracle_mod, ofdk, idx):
    w, f = _case(idx)
    scan = oracle_mod.Scan.from_workload(w, f)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w))
    p = oracle_mod.forward(scan, ci.phantom(w)).reshape(scan.sino_shape).astype(np.float32)
    vw = ctp.full_scan_view_weights(w.n_views)
    d_p, d_vw = _dev(torch, p), _dev(torch, vw)
    for ramp, kind in (("ramlak", ofdk.RAMLAK), ("shepp_logan", ofdk.SHEPP_LOGAN),
                       ("cosine", ofdk.COSINE), ("hamming", ofdk.HAMMING), ("hann", ofdk.HANN)):
        for transpose in (False, True):
            out = torch.full(plan.sino_shape, float("nan"), device="cuda")
            ctp.ctp_ramp_filter(plan, d_p, out, d_vw, ramp, transpose)
            ref = (ofdk.filter_sinogram_transpose if transpose else ofdk.filter_sinogram)(
                scan, p, vw, kind)
            torch.cuda.synchronize()
            assert rel_l2(out.cpu().numpy(), ref) <= TOL_FILTER, (ramp, transpose)
    # gather of the oracle's filtered sinogram (as float32)
    q = ofdk.filter_sinogram(scan, p, vw).astype(np.float32)
    g = torch.full(plan.vol_shape, float("nan"), device="cuda")
    ctp.ctp_weighted_backproject(plan, _dev(torch, q), g)
    g_ref = ofdk.weighted_backproject(scan, q)
    torch.cuda.synchronize()
    assert rel_l2(g.cpu().numpy(), g_ref) <= TOL_GATHER
    # the whole FDK, in place on a copy of the sinogram
    work = d_p.clone()
    vol = torch.full(plan.vol_shape, float("nan"), device="cuda")
    ctp.ctp_fdk(plan, work, work, vol, d_vw)
    torch.cuda.synchronize()
    assert rel_l2(vol.cpu().numpy(), ofdk.fdk(scan, p, vw)) <= TOL_GATHER
    # transpose of the gather
    x = np.random.default_rng(idx).standard_normal(plan.vol_shape).astype(np.float32)
    t = torch.full(plan.sino_shape, float("nan"), device="cuda")
    ctp.ctp_weighted_backproject_transpose(plan, _dev(torch, x), t)
    torch.cuda.synchronize()
    assert rel_l2(t.cpu().numpy(), ofdk.weighted_backproject_transpose(scan, x)) <= TOL_SCATTER


@pytest.mark.parametrize("idx", [2, 3, 5])
def test_gpu_gather_and_scatter_are_adjoint(torch, ctp, idx):
    w, f = _case(idx)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w))
    rng = np.random.default_rng(40 + idx)
    q = _dev(torch, rng.standard_normal(plan.sino_shape))
    x = _dev(torch, rng.standard_normal(plan.vol_shape))
    Bq = torch.empty(plan.vol_shape, device="cuda")
    Btx = torch.empty(plan.sino_shape, device="cuda")
    ctp.ctp_weighted_backproject(plan, q, Bq)
    ctp.ctp_weighted_backproject_transpose(plan, x, Btx)
    torch.cuda.synchronize()
    cs, _ = adjoint_mismatch(Bq.cpu().numpy(), x.cpu().numpy(), q.cpu().numpy(),
                             Btx.cpu().numpy())
    assert cs <= TOL_ADJOINT


def _ball_sinogram(scan, centre, radius):
    """Closed-form line integrals of a unit ball, one view at a time (float32)."""
    import geom_helpers
    out = np.empty(scan.sino_shape, np.float32)
    m = np.asarray(centre, np.float64)[None, :]
    for k in range(scan.n_views):
        X0, r, _, _ = geom_helpers.pixel_rays(scan.beam, *(a[k:k + 1] for a in scan.arrays),
                                              scan.n_u, scan.n_v, scan.pitch_u, scan.pitch_v,
                                              scan.offset_u, scan.offset_v)
        rh = r / np.linalg.norm(r, axis=1, keepdims=True)
        wv = m - X0
        d2 = np.sum(wv * wv, 1) - np.sum(wv * rh, 1) ** 2
        out[k] = (2 * np.sqrt(np.maximum(radius ** 2 - d2, 0.0))).reshape(scan.n_v, scan.n_u)
    return out


def test_fdk_of_a_ball_at_full_c3_size(torch, ctp, oracle_mod, ofdk):
    """At the full 256^3 / 360-view cone scan: FDK of the closed-form line integrals
    of a unit ball gives 1 inside it (mid-plane band), and the sampled voxels
    equal the oracle's gather of the GPU-filtered sinogram."""
    w = ci.WORKLOADS[3]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w))
    centre, radius = (10.0, -6.0, 0.0), 50.0
    p = _ball_sinogram(scan, centre, radius)
    vw = _dev(torch, ctp.full_scan_view_weights(w.n_views))
    work = _dev(torch, p)
    vol = torch.empty(plan.vol_shape, device="cuda")
    ctp.ctp_fdk(plan, work, work, vol, vw)
    torch.cuda.synchronize()
    g = vol.cpu().numpy()
    X = ofdk.voxel_centres(scan)
    rel = X - np.asarray(centre)
    r = np.linalg.norm(rel, axis=1)
    inner = (r < 0.75 * radius) & (np.abs(rel[:, 2]) <= 2.0)
    assert abs(g.ravel()[inner].mean() - 1.0) < 2e-3
    assert np.abs(g.ravel()[inner] - 1.0).max() < 2e-2
    # sampled parity of the gather on the filtered sinogram the GPU produced
    q = work.cpu().numpy()
    rng = np.random.default_rng(7)
    D, H, W = w.shape
    vox = np.stack([rng.integers(0, D, 400), rng.integers(0, H, 400), rng.integers(0, W, 400)], 1)
    ref = ofdk.weighted_backproject(scan, q, voxels=vox)
    got = g[vox[:, 0], vox[:, 1], vox[:, 2]]
    assert rel_l2(got, ref) <= TOL_GATHER


@pytest.mark.parametrize("idx", [4, 5])
def test_full_size_sampled_parity(torch, ctp, oracle_mod, ofdk, idx):
    """Full-size scans: the filter on sampled views (oracle on a scan of just those
    views) and the gather at sampled voxels."""
    w = ci.WORKLOADS[idx]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w))
    rng = np.random.default_rng(70 + idx)
    p = ci.sinogram_noise(w).reshape(plan.sino_shape)
    vw = ctp.full_scan_view_weights(w.n_views)
    q = torch.empty(plan.sino_shape, device="cuda")
    ctp.ctp_ramp_filter(plan, _dev(torch, p), q, _dev(torch, vw))
    vol = torch.empty(plan.vol_shape, device="cuda")
    ctp.ctp_weighted_backproject(plan, q, vol)
    torch.cuda.synchronize()
    qh = q.cpu().numpy()
    views = np.sort(rng.choice(w.n_views, 3, replace=False))
    sub = oracle_mod.Scan(w.beam, *(a[views] for a in scan.arrays), w.n_u, w.n_v, w.pitch_u,
                          w.pitch_v, w.shape, w.spacing, w.origin, w.offset_u, w.offset_v,
                          w.ndim)
    ref = ofdk.filter_sinogram(sub, p[views], vw[views])
    assert rel_l2(qh[views], ref) <= TOL_FILTER
    D, H, W = w.shape
    vox = np.stack([rng.integers(0, D, 200), rng.integers(0, H, 200), rng.integers(0, W, 200)], 1)
    ref = ofdk.weighted_backproject(scan, qh, voxels=vox)
    g = vol.cpu().numpy()
    assert rel_l2(g[vox[:, 0], vox[:, 1], vox[:, 2]], ref) <= TOL_GATHER


# ------------------------------------------------------------------ edge cases
def test_outside_the_class_reports_geometry_error(torch, ctp):
    import geom_helpers
    rng = np.random.default_rng(3)
    src, cen, U, V = geom_helpers.random_frames(rng, 3, "divergent", 40.0, 30.0, tilt=0.4)
    g = ctp.Geometry(ndim=3, beam="divergent", src=src, det_centre=cen, det_u=U, det_v=V,
                     n_u=16, n_v=12, pitch_u=1.0, pitch_v=1.0)
    plan = ctp.ctp_plan(g, ctp.Volume((6, 7, 8), (1.0, 1.0, 1.0), (-4.0, -3.5, -3.0)))
    sino = torch.zeros(plan.sino_shape, device="cuda")
    vol = torch.zeros(plan.vol_shape, device="cuda")
    with pytest.raises(ctp.CtpError) as e:
        ctp.ctp_weighted_backproject(plan, sino, vol)
    assert e.value.status == 13
    ctp.ctp_forward(plan, vol, sino)   # the projector pair still serves this plan


def test_empty_scan_zeroes_the_volume(torch, ctp):
    z = np.zeros((0, 3), np.float32)
    g = ctp.Geometry(ndim=3, beam="divergent", src=z, det_centre=z, det_u=z, det_v=z, n_u=4,
                     n_v=4, pitch_u=1.0, pitch_v=1.0)
    plan = ctp.ctp_plan(g, ctp.Volume((3, 4, 5), (1.0, 1.0, 1.0), (-2.5, -2.0, -1.5)))
    sino = torch.empty((0, 4, 4), device="cuda")
    vol = torch.full((3, 4, 5), 7.0, device="cuda")
    ctp.ctp_fdk(plan, sino, sino, vol)
    assert float(vol.abs().max()) == 0.0


def test_source_inside_the_volume_and_truncated_detector(torch, ctp, oracle_mod, ofdk):
    """Voxels behind or beside the source get nothing from that view; the detector
    covers only part of the volume (zero padding outside)."""
    K = 12
    b = np.arange(K) * 2 * math.pi / K
    c, s, zero, one = np.cos(b), np.sin(b), np.zeros(K), np.ones(K)
    frames = {"src": np.stack([6 * c, 6 * s, zero], 1), "det_centre": np.stack([-20 * c, -20 * s, zero], 1),
              "det_u": np.stack([-s, c, zero], 1), "det_v": np.stack([zero, zero, one], 1)}
    frames = {k: v.astype(np.float32) for k, v in frames.items()}
    shape, spacing = (9, 20, 22), (1.1, 1.0, 0.9)
    origin = (-0.5 * 22 * 0.9, -0.5 * 20 * 1.0, -0.5 * 9 * 1.1)
    n_u, n_v, pu, pv = 21, 11, 1.3, 1.2
    scan = oracle_mod.Scan("divergent", frames["src"], frames["det_centre"], frames["det_u"],
                           frames["det_v"], n_u, n_v, pu, pv, shape, spacing, origin, 0.3, -0.4, 3)
    g = ctp.Geometry(ndim=3, beam="divergent", n_u=n_u, n_v=n_v, pitch_u=pu, pitch_v=pv,
                     offset_u=0.3, offset_v=-0.4, **frames)
    plan = ctp.ctp_plan(g, ctp.Volume(shape, spacing, origin))
    q = np.random.default_rng(9).standard_normal(plan.sino_shape).astype(np.float32)
    vol = torch.empty(plan.vol_shape, device="cuda")
    ctp.ctp_weighted_backproject(plan, _dev(torch, q), vol)
    torch.cuda.synchronize()
    assert rel_l2(vol.cpu().numpy(), ofdk.weighted_backproject(scan, q)) <= TOL_GATHER


@pytest.mark.parametrize("pitch_v", [8.0, 1.2, 0.4])
@pytest.mark.parametrize("v_sign", [1.0, -1.0])
def test_row_steps_of_every_size_and_a_flipped_v_axis(torch, ctp, oracle_mod, ofdk, pitch_v,
                                                      v_sign):
    """Along a voxel column the stencil rows advance by dv = magnification x dz /
    pitch_v per z step: under one row (consecutive steps share both rows), between
    one and two (they share one), over two (none), and with the v axis along -z
    (rows decrease).  The transpose's register row sums and the gather's and
    transpose's skip of off-detector columns must match the oracle in each case;
    40 z voxels make two whole 16-voxel chunks and a ragged one."""
    K = 10
    b = np.arange(K) * 2 * math.pi / K + 0.1
    c, s, zero, one = np.cos(b), np.sin(b), np.zeros(K), np.ones(K)
    frames = {"src": np.stack([40 * c, 40 * s, zero], 1),
              "det_centre": np.stack([-30 * c, -30 * s, zero], 1),
              "det_u": np.stack([-s, c, zero], 1), "det_v": np.stack([zero, zero, v_sign * one], 1)}
    frames = {k: v.astype(np.float32) for k, v in frames.items()}
    shape, spacing = (40, 12, 12), (1.0, 1.0, 1.0)
    origin = (-6.0, -6.0, -20.0)
    n_u, n_v, pu = 26, 24, 1.5
    scan = oracle_mod.Scan("divergent", frames["src"], frames["det_centre"], frames["det_u"],
                           frames["det_v"], n_u, n_v, pu, pitch_v, shape, spacing, origin, 0.2,
                           0.3, 3)
    g = ctp.Geometry(ndim=3, beam="divergent", n_u=n_u, n_v=n_v, pitch_u=pu, pitch_v=pitch_v,
                     offset_u=0.2, offset_v=0.3, **frames)
    plan = ctp.ctp_plan(g, ctp.Volume(shape, spacing, origin))
    rng = np.random.default_rng(int(10 * pitch_v) + (v_sign > 0))
    q = rng.standard_normal(plan.sino_shape).astype(np.float32)
    x = rng.standard_normal(plan.vol_shape).astype(np.float32)
    d_q, d_x = _dev(torch, q), _dev(torch, x)
    vol = torch.full(plan.vol_shape, float("nan"), device="cuda")
    t = torch.full(plan.sino_shape, float("nan"), device="cuda")
    ctp.ctp_weighted_backproject(plan, d_q, vol)
    ctp.ctp_weighted_backproject_transpose(plan, d_x, t)
    torch.cuda.synchronize()
    got_b, got_t = vol.cpu().numpy(), t.cpu().numpy()
    assert rel_l2(got_b, ofdk.weighted_backproject(scan, q)) <= TOL_GATHER
    ref_t = ofdk.weighted_backproject_transpose(scan, x)
    assert np.abs(ref_t).max() > 0.0
    assert rel_l2(got_t, ref_t) <= TOL_SCATTER
    cs, _ = adjoint_mismatch(got_b, x, q, got_t)
    assert cs <= TOL_ADJOINT


@pytest.mark.parametrize("n_u", [5000, 16385])
def test_wide_detector_rows(torch, ctp, oracle_mod, ofdk, n_u):
    """Rows wider than 4096 pixels take the one-row-per-block filter with more than
    48 KB of shared memory; beyond 16384 the filter reports CTP_E_LIMIT."""
    frames = {"src": np.array([[300.0, 0, 0]], np.float32),
              "det_centre": np.array([[-200.0, 0, 0]], np.float32),
              "det_u": np.array([[0, 1.0, 0]], np.float32),
              "det_v": np.array([[0, 0, 1.0]], np.float32)}
    g = ctp.Geometry(ndim=3, beam="divergent", n_u=n_u, n_v=2, pitch_u=0.05, pitch_v=1.0,
                     **frames)
    vol = ctp.Volume((2, 2, 2), (1.0, 1.0, 1.0), (-1.0, -1.0, -1.0))
    plan = ctp.ctp_plan(g, vol)
    p = np.random.default_rng(1).standard_normal(plan.sino_shape).astype(np.float32)
    out = torch.empty(plan.sino_shape, device="cuda")
    if n_u > 16384:
        with pytest.raises(ctp.CtpError) as e:
            ctp.ctp_ramp_filter(plan, _dev(torch, p), out)
        assert e.value.status == 12
        return
    ctp.ctp_ramp_filter(plan, _dev(torch, p), out)
    scan = oracle_mod.Scan("divergent", frames["src"], frames["det_centre"], frames["det_u"],
                           frames["det_v"], n_u, 2, 0.05, 1.0, (2, 2, 2), (1.0, 1.0, 1.0),
                           (-1.0, -1.0, -1.0), 0.0, 0.0, 3)
    torch.cuda.synchronize()
    assert rel_l2(out.cpu().numpy(), ofdk.filter_sinogram(scan, p)) <= TOL_FILTER


def test_pixel_weights_and_parker_short_scan(torch, ctp, oracle_mod, ofdk):
    """Parker weights from the library equal the oracle's; the filter with pixel
    weights (forward and transpose) matches the oracle; the short-scan fan FBP
    reconstructs the disc and matches the oracle."""
    import test_oracle_fdk_pins as pins
    scan, centre, radius, w = pins._short_fan_case(oracle_mod, ofdk)
    g = ctp.Geometry(ndim=2, beam="divergent", src=scan.arrays[0], det_centre=scan.arrays[1],
                     det_u=scan.arrays[2], det_v=scan.arrays[3], n_u=scan.n_u, n_v=1,
                     pitch_u=scan.pitch_u, pitch_v=1.0)
    plan = ctp.ctp_plan(g, ctp.Volume(scan.shape, scan.spacing, scan.origin))
    pw = ctp.ctp_parker_weights(plan)
    pw_ref = ofdk.parker_weights(scan)
    torch.cuda.synchronize()
    assert np.abs(pw.cpu().numpy() - pw_ref).max() <= 1e-6
    p = pins._ball_sinogram(scan, centre, radius).astype(np.float32)
    d_p, d_w = _dev(torch, p), _dev(torch, w)
    for transpose in (False, True):
        out = torch.empty(plan.sino_shape, device="cuda")
        ctp.ctp_ramp_filter(plan, d_p, out, d_w, "hann", transpose, pixel_weight=pw)
        if transpose:
            ref = ofdk.filter_sinogram_transpose(scan, p, w, ofdk.HANN) * pw_ref[:, None, :]
        else:
            ref = ofdk.filter_sinogram_pw(scan, p, w, pw_ref, ofdk.HANN)
        torch.cuda.synchronize()
        assert rel_l2(out.cpu().numpy(), ref) <= TOL_FILTER, transpose
    vol = torch.empty(plan.vol_shape, device="cuda")
    ctp.ctp_fdk(plan, d_p, torch.empty_like(d_p), vol, d_w, pixel_weight=pw)
    torch.cuda.synchronize()
    got = vol.cpu().numpy()
    ref = ofdk.weighted_backproject(scan, ofdk.filter_sinogram_pw(scan, p, w, pw_ref))
    assert rel_l2(got, ref) <= TOL_GATHER
    assert pins._check_reconstruction(ofdk, scan, got, centre, radius, 1e-3, 5e-3, None)
