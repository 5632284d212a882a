"""Pins of the float64 oracle against things other than itself.

Each test fixes one part of the oracle with a value the mathematics or a
hand derivation fixes: hand-worked path sums, chord lengths of boxes and balls,
brute force over every cell, a supersampled line integral with its error
bound, textbook axis-aligned cases, invariances, and the adjoint identity
(diffct 2.1.0 -> 2.2.1, README "Matched operators": the forward / backward pair
is an exact adjoint pair for the cell-constant Siddon model; diffct 2.2.1 ->
2.4.0, README quickstart: an adjoint mismatch of about 1e-8 per beam).
"""

import json
import math
import os

import numpy as np
import pytest

from geom_helpers import chord, pixel_rays, random_frames

HERE = os.path.dirname(os.path.abspath(__file__))


def _scan(oracle, beam, frames, n_u, n_v, pu, pv, shape, spacing, ou=0.0, ov=0.0):
    D, H, W = shape
    dz, dy, dx = spacing
    origin = (-0.5 * W * dx, -0.5 * H * dy, -0.5 * D * dz)
    return oracle.Scan(beam, *frames, n_u, n_v, pu, pv, shape, spacing, origin, ou, ov)


def _rays_of(scan):
    return pixel_rays(scan.beam, *scan.arrays, scan.n_u, scan.n_v, scan._ctx.pitch_u,
                      scan._ctx.pitch_v, scan._ctx.offset_u, scan._ctx.offset_v)


# --------------------------------------------------------------------------- golden
def test_hand_cases(oracle_mod):
    with open(os.path.join(HERE, "golden", "hand_cases.json")) as fh:
        cases = json.load(fh)["cases"]
    for case in cases:
        shape = tuple(case["shape"])
        frames = [np.array(case[k], dtype=np.float32)
                  for k in ("src", "det_centre", "det_u", "det_v")]
        scan = _scan(oracle_mod, case["beam"], frames, case["n_u"], case["n_v"],
                     case["pitch_u"], case["pitch_v"], shape, tuple(case["spacing"]),
                     case["offset_u"], case["offset_v"])
        vol = (1 + np.arange(np.prod(shape))).reshape(shape).astype(np.float32)
        got = oracle_mod.forward(scan, vol).ravel()
        want = np.array([eval(e, {"math": math}) for e in case["expected"]])
        np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13, err_msg=case["name"])
        if "backward_input" in case:
            g = oracle_mod.backward(scan, np.array(case["backward_input"], np.float32))
            np.testing.assert_allclose(g, np.array(case["backward_expected"], float),
                                       rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ closed forms
@pytest.mark.parametrize("beam", ["divergent", "parallel"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_uniform_subbox_equals_chord(oracle_mod, beam, seed):
    rng = np.random.default_rng(100 + seed)
    shape = (7, 9, 11)
    spacing = (1.3, 0.7, 0.9)
    frames = random_frames(rng, 6, beam, radius=40.0, det_dist=30.0)
    scan = _scan(oracle_mod, beam, frames, 13, 11, 0.83, 0.91, shape, spacing, 0.3, -0.2)
    D, H, W = shape
    dz, dy, dx = spacing
    origin = np.array(scan.origin)
    d = np.array([dx, dy, dz])
    X0, r, tlo, thi = _rays_of(scan)
    for trial in range(4):
        lo_c = np.array([rng.integers(0, W - 1), rng.integers(0, H - 1), rng.integers(0, D - 1)])
        hi_c = np.array([rng.integers(lo_c[0] + 1, W + 1), rng.integers(lo_c[1] + 1, H + 1),
                         rng.integers(lo_c[2] + 1, D + 1)])
        vol = np.zeros(shape, np.float32)
        vol[lo_c[2]:hi_c[2], lo_c[1]:hi_c[1], lo_c[0]:hi_c[0]] = 1.0
        got = oracle_mod.forward(scan, vol).ravel()
        want = chord(X0, r, tlo, thi, origin + lo_c * d, origin + hi_c * d)
        assert np.count_nonzero(want) > 10
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-11)


def test_ball_chords_converge_with_grid(oracle_mod):
    """Centre-voxelised ball of radius R: projections approach the analytic
    chord 2 sqrt(R^2 - dist^2); the relative L2 error shrinks as the grid refines."""
    R = 9.0
    c = np.array([1.3, -0.7, 0.4])
    rng = np.random.default_rng(7)
    frames = random_frames(rng, 5, "divergent", radius=60.0, det_dist=40.0)
    errs = []
    for h in (1.0, 0.5, 0.25):
        n = int(round(24 / h))
        shape = (n, n, n)
        scan = _scan(oracle_mod, "divergent", frames, 21, 21, 1.4, 1.4, shape, (h, h, h))
        xs = scan.origin[0] + (np.arange(n) + 0.5) * h
        Z, Y, X = np.meshgrid(xs, xs, xs, indexing="ij")
        vol = (((X - c[0]) ** 2 + (Y - c[1]) ** 2 + (Z - c[2]) ** 2) <= R * R).astype(np.float32)
        X0, r, tlo, thi = _rays_of(scan)
        rn = r / np.linalg.norm(r, axis=1, keepdims=True)
        w = X0 - c
        dist2 = (w * w).sum(1) - (w * rn).sum(1) ** 2
        want = 2 * np.sqrt(np.clip(R * R - dist2, 0, None))
        got = oracle_mod.forward(scan, vol).ravel()
        errs.append(np.linalg.norm(got - want) / np.linalg.norm(want))
    assert errs[2] < 0.6 * errs[0], errs
    assert errs[2] < 0.02, errs


# ------------------------------------------------------------------- brute force
@pytest.mark.parametrize("case", range(6))
def test_traversal_equals_brute_force(oracle_mod, case):
    rng = np.random.default_rng(300 + case)
    shapes = [(3, 4, 5), (1, 7, 6), (5, 3, 4), (4, 4, 4), (2, 6, 3), (6, 5, 1)]
    spacings = [(1.0, 1.0, 1.0), (1.0, 0.5, 1.5), (2.0, 0.7, 0.3), (1.0, 1.0, 1.0),
                (0.9, 1.1, 1.3), (1.2, 0.8, 2.0)]
    shape, spacing = shapes[case], spacings[case]
    beam = "divergent" if case % 2 == 0 else "parallel"
    frames = random_frames(rng, 4, beam, radius=20.0, det_dist=15.0)
    if case == 3:
        # axis-aligned rays: directions along x, y and z, through non-face points
        frames[0][:] = np.array([[1, 0, 0], [0, 1, 0], [0, 0, 1], [0, 0, -1]], np.float32)
        frames[1][:] = np.array([[0, 0.31, 0.17]] * 4, np.float32)
        frames[2][:] = np.array([[0, 1, 0], [0, 0, 1], [1, 0, 0], [1, 0, 0]], np.float32)
        frames[3][:] = np.array([[0, 0, 1], [1, 0, 0], [0, 1, 0], [0, 1, 0]], np.float32)
    scan = _scan(oracle_mod, beam, frames, 9, 8, 0.61, 0.57, shape, spacing, 0.13, 0.07)
    vol = rng.uniform(-1, 1, shape).astype(np.float32)
    got = oracle_mod.forward(scan, vol)
    want = oracle_mod.brute_forward(scan, vol)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.count_nonzero(want) > 20
    assert oracle_mod.segment_count(scan) == oracle_mod.brute_count(scan)


def test_supersampled_integral_within_midpoint_bound(oracle_mod):
    """Midpoint rule with M samples of a piecewise-constant integrand errs only
    on the sub-intervals that hold a jump: |S_M - p| <= (jumps + 2) * h * max|f|;
    the error falls ~10x per decade of M."""
    import ctp_inputs as ci
    w = ci.small_cases()[3]
    scan = oracle_mod.Scan.from_workload(w, ci.frames(w))
    vol = ci.phantom(w)
    rng = np.random.default_rng(11)
    rays = rng.choice(scan.n_rays, 40, replace=False)
    p = oracle_mod.forward_rays(scan, vol, rays)
    X0, r, tlo, thi = _rays_of(scan)
    D, H, W = w.shape
    full = chord(X0[rays], r[rays], tlo[rays], thi[rays], np.array(scan.origin),
                 np.array(scan.origin) + np.array([W, H, D]) * np.array(w.spacing[::-1]))
    fmax = float(np.abs(vol).max())
    errs = []
    for M in (1000, 10000, 100000):
        s = oracle_mod.supersampled(scan, vol, rays, M)
        h = full / M
        bound = (W + H + D + 2) * h * fmax
        assert np.all(np.abs(s - p) <= bound + 1e-12)
        errs.append(np.abs(s - p).sum())
    assert errs[1] < errs[0] / 4 and errs[2] < errs[1] / 4, errs


# ----------------------------------------------------------- textbook / invariance
def test_axis_aligned_rows_and_columns(oracle_mod):
    """Parallel rays along x through cell-centre rows sum dx * row; along y, dy * column."""
    rng = np.random.default_rng(5)
    H, W = 10, 12
    dy, dx = 0.7, 1.3
    img = rng.uniform(0, 1, (1, H, W)).astype(np.float32)
    frames = [np.array([[1, 0, 0], [0, 1, 0]], np.float32), np.zeros((2, 3), np.float32),
              np.array([[0, 1, 0], [-1, 0, 0]], np.float32),
              np.array([[0, 0, 1], [0, 0, 1]], np.float32)]
    # view 0: rays along x, u = +y, pitch dy: one ray per row centre
    scan0 = _scan(oracle_mod, "parallel", [f[:1] for f in frames], H, 1, dy, 1.0,
                  (1, H, W), (1.0, dy, dx))
    got0 = oracle_mod.forward(scan0, img).ravel()
    np.testing.assert_allclose(got0, dx * img[0].astype(np.float64).sum(1), rtol=1e-13)
    # view 1: rays along y, u = -x, pitch dx: pixel iu sits at x = -(iu - (W-1)/2) dx
    scan1 = _scan(oracle_mod, "parallel", [f[1:] for f in frames], W, 1, dx, 1.0,
                  (1, H, W), (1.0, dy, dx))
    got1 = oracle_mod.forward(scan1, img).ravel()
    np.testing.assert_allclose(got1, dy * img[0].astype(np.float64).sum(0)[::-1], rtol=1e-13)


def test_isotropic_diagonal_pieces(oracle_mod):
    """A ray along the diagonal of a cubic grid through a generic point: every
    piece has length sqrt(3) d once the corner-aligned ray splits no cell."""
    n, d = 6, 0.5
    frames = [np.array([[1, 1, 1]], np.float32) / np.float32(np.sqrt(3)),
              np.zeros((1, 3), np.float32), np.array([[1, -1, 0]], np.float32) / np.float32(np.sqrt(2)),
              np.array([[1, 1, -2]], np.float32) / np.float32(np.sqrt(6))]
    scan = _scan(oracle_mod, "parallel", frames, 1, 1, 1.0, 1.0, (n, n, n), (d, d, d))
    vol = np.ones((n, n, n), np.float32)
    assert oracle_mod.segment_count(scan) == n
    np.testing.assert_allclose(oracle_mod.forward(scan, vol).ravel(), [n * d * math.sqrt(3)],
                               rtol=1e-6)  # float32 direction: |r| = 1 to ~1e-7


def test_spacing_and_geometry_scale_together(oracle_mod):
    rng = np.random.default_rng(9)
    frames = random_frames(rng, 3, "divergent", 30.0, 20.0)
    vol = rng.uniform(0, 1, (5, 6, 7)).astype(np.float32)
    s = 2.0  # power of two: float32 frames scale exactly
    a = _scan(oracle_mod, "divergent", frames, 7, 6, 0.9, 0.8, (5, 6, 7), (1.1, 0.9, 0.7))
    b = _scan(oracle_mod, "divergent", [frames[0] * s, frames[1] * s, frames[2], frames[3]],
              7, 6, 0.9 * s, 0.8 * s, (5, 6, 7), (1.1 * s, 0.9 * s, 0.7 * s))
    np.testing.assert_allclose(oracle_mod.forward(b, vol), s * oracle_mod.forward(a, vol),
                               rtol=1e-12, atol=1e-12)


def test_offset_shifts_pixels(oracle_mod):
    rng = np.random.default_rng(10)
    frames = random_frames(rng, 2, "divergent", 30.0, 20.0)
    vol = rng.uniform(0, 1, (5, 6, 7)).astype(np.float32)
    a = _scan(oracle_mod, "divergent", frames, 9, 8, 0.9, 0.8, (5, 6, 7), (1, 1, 1), 0.0, 0.0)
    b = _scan(oracle_mod, "divergent", frames, 9, 8, 0.9, 0.8, (5, 6, 7), (1, 1, 1), 2.0, -1.0)
    pa, pb = oracle_mod.forward(a, vol), oracle_mod.forward(b, vol)
    # offset +2 in u moves pixel iu to where iu+2 sat; offset -1 in v: iv to iv-1
    np.testing.assert_allclose(pb[:, 1:, :-2], pa[:, :-1, 2:], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------- transpose
@pytest.mark.parametrize("idx", [1, 2, 3, 5])
def test_adjoint_identity_float64(oracle_mod, idx):
    import ctp_inputs as ci
    w = ci.small_cases()[idx]
    scan = oracle_mod.Scan.from_workload(w, ci.frames(w))
    rng = np.random.default_rng(idx)
    x = rng.standard_normal(w.shape).astype(np.float32)
    y = rng.standard_normal(w.sino_shape).astype(np.float32)
    Ax = oracle_mod.forward(scan, x)
    Aty = oracle_mod.backward(scan, y.ravel())
    lhs = float((Ax * y.astype(np.float64)).sum())
    rhs = float((x.astype(np.float64) * Aty).sum())
    scale = np.linalg.norm(Ax) * np.linalg.norm(y)
    assert abs(lhs - rhs) / scale < 1e-13
    assert abs(lhs - rhs) / abs(lhs) < 1e-8  # the pages' quickstart mismatch, beaten


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_backward_equals_voxel_driven(oracle_mod, idx):
    import ctp_inputs as ci
    w = ci.small_cases()[idx]
    scan = oracle_mod.Scan.from_workload(w, ci.frames(w))
    y = ci.sinogram_noise(w)
    g = oracle_mod.backward(scan, y.ravel())
    rng = np.random.default_rng(idx)
    vox = rng.choice(w.n_voxels, min(w.n_voxels, 400), replace=False)
    gv = oracle_mod.backward_voxels(scan, y, vox)
    np.testing.assert_allclose(gv, g.ravel()[vox], rtol=1e-11, atol=1e-11 * np.abs(g).max())


def test_backward_deterministic_over_threads(oracle_mod):
    import ctp_inputs as ci
    w = ci.small_cases()[3]
    scan = oracle_mod.Scan.from_workload(w, ci.frames(w))
    y = ci.sinogram_noise(w).ravel()
    g1 = oracle_mod.backward(scan, y, threads=1)
    g3 = oracle_mod.backward(scan, y, threads=3)
    g3b = oracle_mod.backward(scan, y, threads=3)
    g8 = oracle_mod.backward(scan, y, threads=8)
    # Bitwise repeatable at a fixed thread count (owned bands, no atomics).
    assert np.array_equal(g3, g3b)
    # Across band layouts only pieces shorter than ~1e-12 at a band face can
    # land on the other side of it (their midpoint rounds onto the plane).
    scale = np.abs(g1).max()
    np.testing.assert_allclose(g3, g1, rtol=0, atol=1e-11 * scale)
    np.testing.assert_allclose(g8, g1, rtol=0, atol=1e-11 * scale)


def test_partial_ray_ranges_compose(oracle_mod):
    import ctp_inputs as ci
    w = ci.small_cases()[2]
    scan = oracle_mod.Scan.from_workload(w, ci.frames(w))
    vol = ci.phantom(w)
    y = ci.sinogram_noise(w).ravel()
    full = oracle_mod.forward(scan, vol).ravel()
    cut = scan.n_rays // 3
    np.testing.assert_array_equal(oracle_mod.forward(scan, vol, 0, cut), full[:cut])
    g = oracle_mod.backward(scan, y)
    g2 = oracle_mod.backward(scan, y[:cut], 0, cut) + oracle_mod.backward(scan, y[cut:], cut)
    np.testing.assert_allclose(g, g2, rtol=1e-12, atol=1e-12)
    n = oracle_mod.segment_count(scan)
    assert n == oracle_mod.segment_count(scan, 0, cut) + oracle_mod.segment_count(scan, cut)


# ------------------------------------------------------------------- ambiguity
def test_ambiguity_flags(oracle_mod):
    frames = [np.array([[10, 0, 0], [10, 0.0, 0.0]], np.float32),
              np.array([[-10, 0, 0], [-10, 0.3, 0.0]], np.float32),
              np.array([[0, 1, 0]] * 2, np.float32), np.array([[0, 0, 1]] * 2, np.float32)]
    # 4x4 grid, spacing 1: y = 0 is a cell face.  Pixel offsets 0 and 0.5 (pitch 1).
    scan = _scan(oracle_mod, "divergent", frames, 2, 1, 1.0, 1.0, (1, 4, 4), (1, 1, 1), 0.5)
    flags = oracle_mod.ambiguous(scan).reshape(2, 2)
    # view 0: pixel 0 at y=0 -> ray in the face y = 0; pixel 1 at y=1 -> slanted
    # view 1: pixel 0 at y=0.3 (slanted), pixel 1 at y=1.3 (slanted)
    assert flags.tolist() == [[True, False], [False, False]]


def test_workload_c4_central_column_is_flagged(oracle_mod):
    """With the 3.5 px u-offset the u = 0 detector column of the first view lies
    in the face plane y = 0 of the 512-cell grid; the flag marks exactly it."""
    import dataclasses
    import ctp_inputs as ci
    # two rows at v = -0.5 and +0.5 (as on the 512-row detector); an odd row
    # count would put a whole row in the face plane z = 0
    w = dataclasses.replace(ci.get(4), n_views=1, n_v=2)
    scan = oracle_mod.Scan.from_workload(w, ci.frames(w))
    flags = oracle_mod.ambiguous(scan)[0]
    assert flags[:, 380].all() and flags.sum() == 2
