"""GPU parity: the CUDA pair (through the C ABI) against the float64 oracle.

Bars: forward relative L2 <= 1e-5, backward relative L2 <= 1e-4 (float32
atomics, order-dependent), the GPU pair's own adjoint identity <= 1e-5
(Cauchy-Schwarz normalised).  Rays that lie in a cell-face plane (where the
+ side rule decides and any finite-precision traversal may legitimately pick
the other side) are excluded: their pixels from the forward comparison, their
values from the backward input.
"""

import dataclasses
import json
import os

import numpy as np
import pytest

import strata
from cases import (TOL_ADJOINT, TOL_BACKWARD, TOL_BACKWARD_MAX, TOL_FORWARD, TOL_FORWARD_MAX,
                   adjoint_mismatch, ci, geometry_of, max_rel_err, rel_l2, volume_of)

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


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


def _run_pair(torch, ctp, plan, vol, y):
    d_vol = torch.from_numpy(np.ascontiguousarray(vol)).cuda()
    d_sino = torch.empty(plan.sino_shape, dtype=torch.float32, device="cuda")
    ctp.ctp_forward(plan, d_vol, d_sino)
    d_y = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    d_g = torch.full(plan.vol_shape, float("nan"), dtype=torch.float32, device="cuda")
    ctp.ctp_backward(plan, d_y, d_g)
    torch.cuda.synchronize()
    return d_sino.cpu().numpy(), d_g.cpu().numpy()


SMALL = ci.small_cases()


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("path", ["auto", "ray"])
def test_small_cases_match_oracle(torch, ctp, oracle_mod, idx, path):
    w = SMALL[idx]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    vol = ci.phantom(w)
    y = ci.sinogram_noise(w)
    amb = oracle_mod.ambiguous(scan)
    y_clean = np.where(amb, np.float32(0), y)
    p_ref = oracle_mod.forward(scan, vol)
    g_ref = oracle_mod.backward(scan, y_clean.ravel())

    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), path)
    expected = {"auto": "column" if w.ndim == 3 else "plane", "ray": "ray"}[path]
    assert plan.path == expected
    p, g = _run_pair(torch, ctp, plan, vol, y_clean)
    assert rel_l2(p[~amb], p_ref[~amb]) <= TOL_FORWARD
    assert rel_l2(g, g_ref) <= TOL_BACKWARD
    assert max_rel_err(p[~amb], p_ref[~amb]) <= TOL_FORWARD_MAX
    assert max_rel_err(g, g_ref) <= TOL_BACKWARD_MAX

    # the GPU pair's own adjoint identity, random x and y, every ray included
    rng = np.random.default_rng(idx)
    x = rng.standard_normal(w.shape).astype(np.float32)
    Ax, Aty = _run_pair(torch, ctp, plan, x, y)
    cs, raw = adjoint_mismatch(Ax, y, x, Aty)
    assert cs <= TOL_ADJOINT, (cs, raw)

    n_ref = oracle_mod.segment_count(scan)
    n_gpu = ctp.ctp_segment_count(plan)
    assert abs(n_gpu - n_ref) <= max(1e-6 * n_ref, 4), (n_gpu, n_ref)


@pytest.mark.parametrize("idx", [3, 4, 5])
def test_ray_and_column_paths_agree(torch, ctp, idx):
    w = SMALL[idx]
    f = ci.frames(w)
    vol = ci.phantom(w)
    y = ci.sinogram_noise(w)
    out = {}
    for path in ("ray", "column"):
        plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), path)
        out[path] = _run_pair(torch, ctp, plan, vol, y)
    assert rel_l2(out["column"][0], out["ray"][0]) <= TOL_FORWARD
    assert rel_l2(out["column"][1], out["ray"][1]) <= TOL_BACKWARD


@pytest.mark.parametrize("idx", [1, 2])
def test_ray_and_plane_paths_agree(torch, ctp, idx):
    w = SMALL[idx]
    f = ci.frames(w)
    vol = ci.phantom(w)
    y = ci.sinogram_noise(w)
    out = {}
    for path in ("ray", "plane"):
        plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), path)
        assert plan.path == path
        out[path] = _run_pair(torch, ctp, plan, vol, y)
    assert rel_l2(out["plane"][0], out["ray"][0]) <= TOL_FORWARD
    assert rel_l2(out["plane"][1], out["ray"][1]) <= TOL_BACKWARD


@pytest.mark.parametrize("mode", ["tiled", "privatised"])
def test_plane_backward_variants_match_oracle(torch, ctp, oracle_mod, mode):
    """The plane backward's two work layouts (shared-memory tiles for small
    scans, privatised global accumulators for larger ones) on the same scan."""
    w = SMALL[2]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    y = ci.sinogram_noise(w)
    g_ref = oracle_mod.backward(scan, y.ravel())
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), "plane",
                        options={"plane_backward": mode})
    _, g = _run_pair(torch, ctp, plan, ci.phantom(w), y)
    assert rel_l2(g, g_ref) <= TOL_BACKWARD


@pytest.mark.parametrize("idx,keep", [(2, 17), (2, 97), (1, 29)])
def test_plane_backward_sparse_sinogram(torch, ctp, oracle_mod, idx, keep):
    """A sinogram that is zero but on every keep-th ray leaves most lanes of a
    lockstep warp idle, so the warp's union of slab ranges has gaps that whole
    chunks fall into: both plane backwards still equal the oracle."""
    w = SMALL[idx]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    amb = oracle_mod.ambiguous(scan)
    y = ci.sinogram_noise(w)
    mask = (np.arange(y.size).reshape(y.shape) % keep) == 0
    y = np.where(mask & ~amb, y, np.float32(0))
    g_ref = oracle_mod.backward(scan, y.ravel())
    for mode in ("privatised", "tiled"):
        plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), "plane",
                            options={"plane_backward": mode})
        _, g = _run_pair(torch, ctp, plan, ci.phantom(w), y)
        assert rel_l2(g, g_ref) <= TOL_BACKWARD, mode
        assert max_rel_err(g, g_ref) <= TOL_BACKWARD_MAX, mode


def test_plane_privatised_copies_start_every_call_at_zero(torch, ctp, oracle_mod):
    """The privatised backward's accumulator copies carry nothing from one call
    to the next: calls in a row on one plan (device and host-buffer, sinograms
    of growing scale) each match the oracle, and a zero sinogram after nonzero
    ones backprojects to exactly zero."""
    w = SMALL[2]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), "plane",
                        options={"plane_backward": "privatised", "host_chunks": 3})
    rng = np.random.default_rng(77)
    d_g = torch.empty(plan.vol_shape, dtype=torch.float32, device="cuda")
    for k in range(3):
        y = (rng.standard_normal(plan.sino_shape) * 10.0 ** k).astype(np.float32)
        g_ref = oracle_mod.backward(scan, y.ravel())
        if k == 1:
            g = np.full(plan.vol_shape, np.nan, np.float32)
            ctp.ctp_backward_host(plan, y, g)
        else:
            d_g.fill_(float("nan"))
            ctp.ctp_backward(plan, torch.from_numpy(y).cuda(), d_g)
            g = d_g.cpu().numpy()
        assert rel_l2(g, g_ref) <= TOL_BACKWARD, k
        assert max_rel_err(g, g_ref) <= TOL_BACKWARD_MAX, k
    d_g.fill_(float("nan"))
    ctp.ctp_backward(plan, torch.zeros(plan.sino_shape, device="cuda"), d_g)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d_g).item() == 0


@pytest.mark.parametrize("rows", [1, 2, 3, 4])
@pytest.mark.parametrize("adjacent", [0, 1])
@pytest.mark.parametrize("ahead", ["off", "on"])
def test_column_work_layouts_match_oracle(torch, ctp, oracle_mod, rows, adjacent, ahead):
    """Every rows-per-thread choice of the column walks (forward and backward),
    both row orders of the 2-row backward and the forward with and without its
    gathers loaded a slab ahead compute the same operator."""
    w = SMALL[3]
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    vol = ci.phantom(w)
    y = ci.sinogram_noise(w)
    amb = oracle_mod.ambiguous(scan)
    y_clean = np.where(amb, np.float32(0), y)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), "column",
                        options={"rows_forward": rows, "rows_backward": rows,
                                 "backward_rows_adjacent": adjacent, "forward_ahead": ahead})
    p, g = _run_pair(torch, ctp, plan, vol, y_clean)
    p_ref = oracle_mod.forward(scan, vol)
    g_ref = oracle_mod.backward(scan, y_clean.ravel())
    assert rel_l2(p[~amb], p_ref[~amb]) <= TOL_FORWARD
    assert rel_l2(g, g_ref) <= TOL_BACKWARD
    assert max_rel_err(p[~amb], p_ref[~amb]) <= TOL_FORWARD_MAX
    assert max_rel_err(g, g_ref) <= TOL_BACKWARD_MAX
    n_ref = oracle_mod.segment_count(scan)
    assert abs(ctp.ctp_segment_count(plan) - n_ref) <= max(1e-6 * n_ref, 4)


@pytest.mark.parametrize("idx", [3, 4, 5])
def test_forward_ahead_and_order_are_bit_identical(torch, ctp, idx):
    """Loading the gathers a slab ahead and running the blocks views first change
    when values arrive and which blocks run together, not the sums: the column
    forward agrees bit for bit in all four combinations."""
    w = SMALL[idx]
    f = ci.frames(w)
    vol = torch.from_numpy(ci.phantom(w)).cuda()
    out = []
    for ahead in ("off", "on"):
        for first in ("off", "on"):
            plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), "column",
                                options={"forward_ahead": ahead, "forward_views_first": first})
            p = torch.empty(plan.sino_shape, device="cuda")
            ctp.ctp_forward(plan, vol, p)
            out.append(p.cpu().numpy())
    for o in out[1:]:
        assert np.array_equal(out[0], o)


def test_tilted_2d_frames_fall_back_to_ray_path(torch, ctp, oracle_mod):
    # a 2-D scan whose rays leave the slice plane is not a plane-path scan
    w = SMALL[2]
    f = {k: v.copy() for k, v in ci.frames(w).items()}
    f["src"][:, 2] = 0.3
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w))
    assert plan.path == "ray"
    with pytest.raises(ctp.CtpError):
        ctp.ctp_plan(geometry_of(w, f), volume_of(w), "plane")
    scan = oracle_mod.Scan.from_workload(w, f)
    vol = ci.phantom(w)
    p_ref = oracle_mod.forward(scan, vol)
    p, _ = _run_pair(torch, ctp, plan, vol, ci.sinogram_noise(w))
    assert rel_l2(p, p_ref) <= TOL_FORWARD


@pytest.mark.parametrize("idx,path,backward", [(3, "auto", None), (3, "ray", None),
                                               (2, "auto", "privatised"), (2, "auto", "tiled"),
                                               (5, "auto", None)])
@pytest.mark.parametrize("chunks", [0, 1, 3, 7])
@pytest.mark.parametrize("pinned", [False, True])
def test_host_entry_points_match_device(torch, ctp, idx, path, backward, chunks, pinned):
    """The host-buffer calls (view-chunked, copies overlapped with the walk)
    give the device calls' results: the forward bit for bit, the backward up to
    the order of its float atomics."""
    options = {"host_chunks": chunks, "plane_backward": backward or "auto"}
    w = SMALL[idx]
    f = ci.frames(w)
    plan = ctp.ctp_plan(geometry_of(w, f), volume_of(w), path, options=options)
    vol = ci.phantom(w)
    y = ci.sinogram_noise(w)
    p_dev, g_dev = _run_pair(torch, ctp, plan, vol, y)

    def buf(shape, fill=None):
        t = torch.empty(shape, dtype=torch.float32, pin_memory=pinned)
        a = t.numpy()
        a[...] = np.nan if fill is None else fill
        return t, a

    _, vol_h = buf(plan.vol_shape, vol)
    _, y_h = buf(plan.sino_shape, y)
    _, p_host = buf(plan.sino_shape)
    _, g_host = buf(plan.vol_shape)
    for _ in range(2):   # the second call reuses the staging buffers, stream and events
        ctp.ctp_forward_host(plan, vol_h, p_host)
        ctp.ctp_backward_host(plan, y_h, g_host)
        assert np.array_equal(p_host, p_dev)
        assert rel_l2(g_host, g_dev) <= 1e-6


# ------------------------------------------------------------------ edge cases
def _custom(oracle_mod, beam, frames, shape, spacing, n_u, n_v, pu, pv, ou=0.0, ov=0.0):
    D, H, W = shape
    origin = (-0.5 * W * spacing[2], -0.5 * H * spacing[1], -0.5 * D * spacing[0])
    frames = {k: np.ascontiguousarray(v, np.float32) for k, v in frames.items()}
    scan = oracle_mod.Scan(beam, frames["src"], frames["det_centre"], frames["det_u"],
                           frames["det_v"], n_u, n_v, pu, pv, shape, spacing, origin, ou, ov)
    import back_projection_ctp_b300 as ctp
    g = ctp.Geometry(ndim=3, beam=beam, n_u=n_u, n_v=n_v, pitch_u=pu, pitch_v=pv, offset_u=ou,
                     offset_v=ov, **frames)
    return scan, g, ctp.Volume(shape, spacing, origin)


def _check_case(torch, ctp, oracle_mod, scan, g, v, paths=("ray",), seed=0):
    rng = np.random.default_rng(seed)
    vol = rng.uniform(0, 1, v.shape).astype(np.float32)
    y = rng.standard_normal(scan.sino_shape).astype(np.float32)
    amb = oracle_mod.ambiguous(scan)
    y = np.where(amb, np.float32(0), y)
    p_ref = oracle_mod.forward(scan, vol)
    g_ref = oracle_mod.backward(scan, y.ravel())
    for path in paths:
        plan = ctp.ctp_plan(g, v, path)
        p, gg = _run_pair(torch, ctp, plan, vol, y)
        assert rel_l2(p[~amb], p_ref[~amb]) <= TOL_FORWARD, path
        assert rel_l2(gg, g_ref) <= TOL_BACKWARD, path
        assert max_rel_err(p[~amb], p_ref[~amb]) <= TOL_FORWARD_MAX, path
        assert max_rel_err(gg, g_ref) <= TOL_BACKWARD_MAX, path


def test_empty_scan_zeroes_backprojection(torch, ctp):
    z = np.zeros((0, 3), np.float32)
    g = ctp.Geometry(ndim=3, beam="divergent", src=z, det_centre=z, det_u=z, det_v=z, n_u=4,
                     n_v=4, pitch_u=1.0, pitch_v=1.0)
    plan = ctp.ctp_plan(g, ctp.Volume((3, 4, 5), (1.0, 1.0, 1.0), (-2.5, -2.0, -1.5)))
    assert plan.n_rays == 0
    sino = torch.empty((0, 4, 4), dtype=torch.float32, device="cuda")
    vol = torch.full((3, 4, 5), 7.0, dtype=torch.float32, device="cuda")
    ctp.ctp_forward(plan, vol, sino)
    ctp.ctp_backward(plan, sino, vol)
    assert float(vol.abs().max()) == 0.0
    assert ctp.ctp_segment_count(plan) == 0


def test_single_cell_and_single_pixel(torch, ctp, oracle_mod):
    frames = dict(src=[[5.0, 0.3, 0.2]], det_centre=[[-5.0, -0.1, 0.05]], det_u=[[0, 1, 0]],
                  det_v=[[0, 0, 1]])
    scan, g, v = _custom(oracle_mod, "divergent", frames, (1, 1, 1), (0.7, 1.3, 0.9), 1, 1, 1.0, 1.0)
    _check_case(torch, ctp, oracle_mod, scan, g, v, paths=("ray", "column"))


def test_source_and_detector_inside_volume(torch, ctp, oracle_mod):
    # rays start and end inside the grid: partial first / last slabs
    rng = np.random.default_rng(3)
    n = 6
    src = rng.uniform(-3, 3, (n, 3))
    cen = rng.uniform(-3, 3, (n, 3))
    u = np.tile([0.0, 1.0, 0.0], (n, 1))
    vv = np.tile([0.0, 0.0, 1.0], (n, 1))
    cen[:, 0] = src[:, 0] - rng.uniform(2, 5, n)
    cen[:, 2] = src[:, 2]  # rows stay shallow (at most one z plane per slab)
    frames = dict(src=src, det_centre=cen, det_u=u, det_v=vv)
    scan, g, v = _custom(oracle_mod, "divergent", frames, (9, 10, 11), (1.0, 0.9, 0.8), 7, 5, 0.4, 0.5)
    _check_case(torch, ctp, oracle_mod, scan, g, v, paths=("ray", "column"))


def test_tilted_detectors_and_parallel_3d(torch, ctp, oracle_mod):
    from geom_helpers import random_frames
    rng = np.random.default_rng(4)
    for beam in ("divergent", "parallel"):
        fr = random_frames(rng, 7, beam, radius=50.0, det_dist=30.0)
        frames = dict(src=fr[0], det_centre=fr[1], det_u=fr[2], det_v=fr[3])
        scan, g, v = _custom(oracle_mod, beam, frames, (13, 17, 15), (1.1, 0.9, 1.0), 19, 23, 1.3, 1.1,
                             0.25, -0.5)
        _check_case(torch, ctp, oracle_mod, scan, g, v, paths=("ray",), seed=5)


def test_parallel_3d_vertical_detector_uses_column_path(torch, ctp, oracle_mod):
    b = np.linspace(0, np.pi, 10, endpoint=False)
    c, s, z = np.cos(b), np.sin(b), np.zeros_like(b)
    frames = dict(src=np.stack([c, s, 0.1 + z], 1) / np.sqrt(1.01), det_centre=np.stack([z, z, z], 1),
                  det_u=np.stack([-s, c, z], 1), det_v=np.stack([z, z, 1 + z], 1))
    scan, g, v = _custom(oracle_mod, "parallel", frames, (12, 14, 16), (1.0, 1.0, 1.0), 25, 40, 0.8, 0.45)
    assert ctp.ctp_plan(g, v).path == "column"
    _check_case(torch, ctp, oracle_mod, scan, g, v, paths=("column", "ray"), seed=6)


def test_axis_aligned_rays(torch, ctp, oracle_mod):
    frames = dict(src=[[1, 0, 0], [0, 1, 0], [0, 0, 1], [0, -1, 0]],
                  det_centre=[[0, 0.31, 0.17], [0.23, 0, 0.41], [0.13, 0.29, 0], [0.37, 0, 0.11]],
                  det_u=[[0, 1, 0], [0, 0, 1], [1, 0, 0], [1, 0, 0]],
                  det_v=[[0, 0, 1], [1, 0, 0], [0, 1, 0], [0, 0, 1]])
    scan, g, v = _custom(oracle_mod, "parallel", frames, (6, 7, 8), (1.0, 0.8, 1.2), 9, 8, 0.77, 0.61)
    _check_case(torch, ctp, oracle_mod, scan, g, v, paths=("ray",), seed=7)


def test_steep_cone_falls_back_to_ray_path(torch, ctp, oracle_mod):
    # cone half-angle above 45 degrees in cell units: some rows cross several
    # z planes per slab, which the column walk does not cover
    frames = dict(src=[[30, 0, 0], [0, 30, 0]], det_centre=[[-10, 0, 0], [0, -10, 0]],
                  det_u=[[0, 1, 0], [-1, 0, 0]], det_v=[[0, 0, 1], [0, 0, 1]])
    scan, g, v = _custom(oracle_mod, "divergent", frames, (20, 8, 8), (1.0, 1.0, 1.0), 12, 101, 1.0, 1.0)
    assert ctp.ctp_plan(g, v).path == "ray"
    with pytest.raises(ctp.CtpError):
        ctp.ctp_plan(g, v, "column")
    _check_case(torch, ctp, oracle_mod, scan, g, v, paths=("auto",), seed=8)


# ------------------------------------------------------------- full-size runs
def _full_counts():
    with open(os.path.join(HERE, "golden", "segment_counts.json")) as fh:
        return json.load(fh)["full"]


@pytest.fixture(scope="module", params=[1, 2, 3, 4, 5])
def full_case(request, oracle_mod):
    """A workload at full size with its stratified ray and voxel samples and
    the float64 oracle's values there (computed once for both paths)."""
    idx = request.param
    w = ci.get(idx)
    f = ci.frames(w)
    scan = oracle_mod.Scan.from_workload(w, f)
    vol = ci.phantom(w)
    y = ci.sinogram_noise(w)
    amb = oracle_mod.ambiguous(scan)
    y_clean = np.where(amb, np.float32(0), y)
    rng = np.random.default_rng(100 + idx)
    amb_flat = amb.ravel()
    rays = {k: v[~amb_flat[v]] for k, v in strata.ray_strata(w, rng).items()}
    voxels = strata.voxel_strata(w, rng)
    if w.ndim == 2:
        p_all = oracle_mod.forward(scan, vol).ravel()
        g_all = oracle_mod.backward(scan, y_clean.ravel()).ravel()
        p_ref = {k: p_all[v] for k, v in rays.items()}
        g_ref = {k: g_all[v] for k, v in voxels.items()}
    else:
        p_ref = {k: oracle_mod.forward_rays(scan, vol, v) for k, v in rays.items()}
        g_ref = {k: oracle_mod.backward_voxels(scan, y_clean, v) for k, v in voxels.items()}
    return dict(idx=idx, w=w, f=f, vol=vol, y=y_clean, rays=rays, voxels=voxels, p_ref=p_ref,
                g_ref=g_ref)


@pytest.mark.parametrize("path", ["auto", "ray"])
def test_full_size_stratified_parity(torch, ctp, full_case, path):
    """The workloads at full size in the benchmark's launch configuration (AUTO
    path, default stream) and on the ray path: stratified rays and voxels
    against the oracle, per stratum by relative L2 and element by element, the
    GPU pair's adjoint identity and the segment count over the whole scan."""
    c = full_case
    w = c["w"]
    plan = ctp.ctp_plan(geometry_of(w, c["f"]), volume_of(w), path)
    p, g = _run_pair(torch, ctp, plan, c["vol"], c["y"])
    p, g = p.ravel(), g.ravel()
    got_p = {k: p[v] for k, v in c["rays"].items()}
    got_g = {k: g[v] for k, v in c["voxels"].items()}
    strata.check_strata(got_p, c["p_ref"], TOL_FORWARD, TOL_FORWARD_MAX, f"{w.name} forward")
    strata.check_strata(got_g, c["g_ref"], TOL_BACKWARD, TOL_BACKWARD_MAX, f"{w.name} backward")
    # no output element is left unwritten (the backward's output was NaN-filled)
    assert np.all(np.isfinite(p)) and np.all(np.isfinite(g))

    cs, raw = adjoint_mismatch(p, c["y"], c["vol"], g)
    assert cs <= TOL_ADJOINT, (cs, raw)

    n_gpu = ctp.ctp_segment_count(plan)
    n_ref = _full_counts()[str(c["idx"])]["segments"]
    assert abs(n_gpu - n_ref) <= 1e-6 * n_ref, (n_gpu, n_ref)
    plan.destroy()
