"""Pins of the float64 FBP / FDK oracle (``oracle/fdk.py``) against things other
than itself.

* the ramp kernels' frequency responses (the Ram-Lak kernel is the band-limited
  ramp |omega|; Shepp-Logan is |omega| times a sinc window), from their discrete
  Fourier sums;
* the gather reproduces sinograms that are linear in the pixel indices exactly,
  with the detector hit point, depth and normal of every voxel computed by an
  independent 3 x 3 linear solve and an SVD null space;
* the gather and the separately written scatter are transposes (float64);
* filtered backprojection of closed-form line integrals of discs (parallel and
  fan beam) and of a ball (cone beam, mid-plane) gives back the unit density;
* planted mistakes (no cosine weight, no distance weight, no 1/2 of the full
  scan, no 2 pi) make those reconstructions fail -- the pins can see them.

The pages fix the structure and the constants (diffct 2.1.0 -> 2.2.1,
``diffct/analytical.py``: voxel-driven gathers with the analytical constant
1/(2 pi) or SDD/(2 pi SID) and their dedicated transposes; README "Analytical
helpers": ramp filters including Ram-Lak and Shepp-Logan; diffct 2.4.3 ->
2.4.4, ``diffct/analytical.py``: the per-view SDD/(2 pi SID)).
"""

import math

import numpy as np
import pytest

from geom_helpers import pixel_rays, random_frames


@pytest.fixture(scope="module")
def fdk(oracle_mod):
    from oracle import fdk as _fdk
    return _fdk


def _scan(oracle, beam, frames, n_u, n_v, pu, pv, shape, spacing, ou=0.0, ov=0.0, ndim=3,
          centre=(0.0, 0.0, 0.0)):
    D, H, W = shape
    dz, dy, dx = spacing
    origin = (centre[0] - 0.5 * W * dx, centre[1] - 0.5 * H * dy, centre[2] - 0.5 * D * dz)
    return oracle.Scan(beam, *frames, n_u, n_v, pu, pv, shape, spacing, origin, ou, ov, ndim)


def _circular(n_views, beam, sid, sdd, arc=2 * math.pi, z=0.0):
    b = np.arange(n_views) * arc / n_views
    c, s, zero, one = np.cos(b), np.sin(b), np.zeros(n_views), np.ones(n_views)
    U = np.stack([-s, c, zero], 1)
    V = np.stack([zero, zero, one], 1)
    if beam == "parallel":
        src = np.stack([c, s, zero], 1)
        cen = np.zeros((n_views, 3))
    else:
        src = np.stack([sid * c, sid * s, zero + z], 1)
        cen = np.stack([-(sdd - sid) * c, -(sdd - sid) * s, zero + z], 1)
    return [x.astype(np.float32) for x in (src, cen, U, V)]


# ----------------------------------------------------------------- ramp kernels
@pytest.mark.parametrize("tau", [1.0, 0.7])
def test_ramp_kernel_frequency_responses(fdk, tau):
    n = 4097
    m = np.arange(-(n - 1), n)
    for kind, target in ((fdk.RAMLAK, lambda w: np.abs(w)),
                         (fdk.SHEPP_LOGAN, lambda w: (2 / tau) * np.abs(np.sin(w * tau / 2))),
                         (fdk.COSINE, lambda w: np.abs(w) * np.cos(w * tau / 2)),
                         (fdk.HAMMING, lambda w: np.abs(w) * (0.54 + 0.46 * np.cos(w * tau))),
                         (fdk.HANN, lambda w: np.abs(w) * 0.5 * (1 + np.cos(w * tau)))):
        h = fdk.ramp_kernel(n, tau, kind)
        for frac in (0.05, 0.2, 0.5, 0.8, 0.95):
            w = frac * math.pi / tau
            H = tau * np.sum(h * np.cos(w * m * tau))
            assert abs(H - target(w)) < 2e-3 / tau, (kind, frac, H, target(w))
        # zero frequency: the ramp removes the mean
        assert abs(tau * h.sum()) < 2e-3 / tau, kind


# ------------------------------------------------------- geometry, independent solve
def _independent_projection(scan, X, view):
    """Pixel (u, v), weight W and scale s of points X in one view, from a 3x3 solve
    and an SVD normal -- no cross products, no dual basis."""
    a, c, U, V = (arr[view].astype(np.float64) for arr in scan.arrays)
    basis = np.stack([U, V])
    n = np.linalg.svd(basis)[2][-1]          # null space of [U; V]
    u_out, v_out, W = [], [], []
    iso = np.array(scan.origin) + 0.5 * np.array(scan.shape[::-1]) * np.array(scan.spacing[::-1])
    if scan.beam == "divergent":
        if np.dot(c - a, n) < 0:
            n = -n
        sdd, sid = np.dot(c - a, n), np.dot(iso - a, n)
        s = sdd / (2 * math.pi * sid)
    else:
        s = 1 / (2 * math.pi)
    for x in X:
        if scan.beam == "divergent":
            M = np.stack([x - a, -U, -V], 1)
            t, al, be = np.linalg.solve(M, c - a)
            W.append((sid / np.dot(x - a, n)) ** 2)
        else:
            M = np.stack([a, -U, -V], 1)
            t, al, be = np.linalg.solve(M, c - x)
            W.append(1.0)
        u_out.append(al / scan.pitch_u + 0.5 * (scan.n_u - 1) - scan.offset_u)
        v_out.append(be / scan.pitch_v + 0.5 * (scan.n_v - 1) - scan.offset_v)
    return np.array(u_out), np.array(v_out), np.array(W), s


@pytest.mark.parametrize("beam", ["divergent", "parallel"])
def test_gather_reproduces_linear_sinograms(oracle_mod, fdk, beam):
    rng = np.random.default_rng(11 if beam == "divergent" else 12)
    frames = random_frames(rng, 3, beam, radius=40.0, det_dist=30.0, tilt=0.4)
    scan = _scan(oracle_mod, beam, frames, 61, 47, 1.3, 1.1, (5, 6, 7), (1.1, 0.9, 1.4),
                 ou=0.8, ov=-1.7)
    X = fdk.voxel_centres(scan)
    for view in range(scan.n_views):
        al, be, ga = rng.standard_normal(3)
        q = np.zeros(scan.sino_shape)
        iu, iv = np.meshgrid(np.arange(scan.n_u), np.arange(scan.n_v))
        q[view] = al + be * iu + ga * iv
        g = fdk.weighted_backproject(scan, q).ravel()
        u, v, W, s = _independent_projection(scan, X, view)
        inside = (u >= 0) & (u <= scan.n_u - 1.001) & (v >= 0) & (v <= scan.n_v - 1.001)
        assert inside.sum() > 0.8 * len(X)
        expect = s * W * (al + be * u + ga * v)
        np.testing.assert_allclose(g[inside], expect[inside], rtol=1e-11, atol=1e-11)


def test_gather_2d_interpolates_along_u_only(oracle_mod, fdk):
    frames = _circular(4, "divergent", 80.0, 130.0)
    scan = _scan(oracle_mod, "divergent", frames, 41, 1, 1.7, 1.0, (1, 9, 8), (1.0, 1.2, 1.1),
                 ou=0.4, ndim=2)
    X = fdk.voxel_centres(scan)
    for view in range(scan.n_views):
        q = np.zeros(scan.sino_shape)
        q[view, 0] = 2.0 - 0.3 * np.arange(scan.n_u)
        g = fdk.weighted_backproject(scan, q).ravel()
        u, _, W, s = _independent_projection(scan, X, view)
        np.testing.assert_allclose(g, s * W * (2.0 - 0.3 * u), rtol=1e-11, atol=1e-11)


# --------------------------------------------------------------- adjoint identity
@pytest.mark.parametrize("beam,ndim", [("divergent", 3), ("parallel", 3), ("divergent", 2),
                                       ("parallel", 2)])
def test_gather_and_scatter_are_transposes(oracle_mod, fdk, beam, ndim):
    rng = np.random.default_rng(21)
    if ndim == 3:
        frames = random_frames(rng, 4, beam, radius=25.0, det_dist=20.0, tilt=0.3)
        scan = _scan(oracle_mod, beam, frames, 23, 19, 1.2, 1.4, (6, 7, 8), (1.3, 1.0, 0.8),
                     ou=0.3, ov=0.6)
    else:
        frames = _circular(7, beam, 30.0, 55.0)
        scan = _scan(oracle_mod, beam, frames, 29, 1, 1.1, 1.0, (1, 12, 13), (1.0, 1.1, 0.9),
                     ou=-0.7, ndim=2)
    q = rng.standard_normal(scan.sino_shape)
    x = rng.standard_normal(scan.shape)
    lhs = np.vdot(fdk.weighted_backproject(scan, q), x)
    rhs = np.vdot(q, fdk.weighted_backproject_transpose(scan, x))
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), 1.0) * 10
    # the filter pair as well
    w = rng.uniform(0.5, 1.5, scan.n_views)
    for kind in (fdk.RAMLAK, fdk.SHEPP_LOGAN, fdk.COSINE, fdk.HAMMING, fdk.HANN):
        p = rng.standard_normal(scan.sino_shape)
        y = rng.standard_normal(scan.sino_shape)
        a = np.vdot(fdk.filter_sinogram(scan, p, w, kind), y)
        b = np.vdot(p, fdk.filter_sinogram_transpose(scan, y, w, kind))
        assert abs(a - b) <= 1e-11 * max(abs(a), 1.0)


# ------------------------------------------------------ closed-form reconstructions
def _ball_sinogram(scan, centre, radius):
    """Line integrals of a unit ball (disc in 2-D: the ball's mid-plane) along every
    pixel ray: 2 sqrt(R^2 - d^2), d the line's distance from the centre."""
    X0, r, _, _ = pixel_rays(scan.beam, *scan.arrays, scan.n_u, scan.n_v, scan.pitch_u,
                             scan.pitch_v, scan.offset_u, scan.offset_v)
    rh = r / np.linalg.norm(r, axis=1, keepdims=True)
    m = np.asarray(centre, np.float64)
    w = m[None, :] - X0
    d2 = np.sum(w * w, 1) - np.sum(w * rh, 1) ** 2
    return (2 * np.sqrt(np.maximum(radius ** 2 - d2, 0.0))).reshape(scan.sino_shape)


def _check_reconstruction(fdk, scan, g, centre, radius, mean_tol, max_tol, zband=None):
    X = fdk.voxel_centres(scan)
    rel = X - np.asarray(centre)[None, :]
    if zband is not None:
        keep = np.abs(rel[:, 2]) <= zband
    else:
        keep = np.ones(len(X), bool)
    r = np.linalg.norm(rel, axis=1)
    inner = keep & (r < 0.75 * radius)
    outer = keep & (r > 1.3 * radius) & (r < 1.8 * radius)
    gv = g.ravel()
    assert inner.sum() > 20 and outer.sum() > 20
    return (abs(gv[inner].mean() - 1.0) < mean_tol and np.abs(gv[inner] - 1.0).max() < max_tol
            and abs(gv[outer].mean()) < 1e-2)


def _parallel_case(oracle_mod):
    K = 360
    frames = _circular(K, "parallel", 0, 0)
    scan = _scan(oracle_mod, "parallel", frames, 192, 1, 1.0, 1.0, (1, 128, 128),
                 (1.0, 1.0, 1.0), ndim=2)
    return scan, (8.0, -5.0, 0.0), 30.0, np.full(K, math.pi / K)


def _fan_case(oracle_mod):
    K = 360
    frames = _circular(K, "divergent", 150.0, 300.0)
    scan = _scan(oracle_mod, "divergent", frames, 256, 1, 1.0, 1.0, (1, 96, 96),
                 (1.0, 1.0, 1.0), ndim=2)
    return scan, (25.0, -15.0, 0.0), 22.0, np.full(K, math.pi / K)


def _cone_case(oracle_mod):
    K = 180
    frames = _circular(K, "divergent", 250.0, 400.0)
    scan = _scan(oracle_mod, "divergent", frames, 96, 64, 1.0, 1.0, (40, 40, 40),
                 (1.0, 1.0, 1.0), ndim=3)
    return scan, (3.0, -2.0, 0.0), 12.0, np.full(K, math.pi / K)


# interior mean / max error bounds: the float64 reconstructions of these cases
# err by < 3e-5 (mean) and < 3e-3 (max); a dropped weight errs by > 8e-3 (mean)
CASES = {"parallel": (_parallel_case, 1e-3, 5e-3, None),
         "fan": (_fan_case, 1e-3, 5e-3, None),
         "cone": (_cone_case, 1e-3, 1e-2, 1.0)}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("kind", ["ramlak", "shepp_logan"])
def test_fbp_reconstructs_unit_density(oracle_mod, fdk, name, kind):
    make, mean_tol, max_tol, zband = CASES[name]
    scan, centre, radius, w = make(oracle_mod)
    p = _ball_sinogram(scan, centre, radius)
    k = fdk.RAMLAK if kind == "ramlak" else fdk.SHEPP_LOGAN
    g = fdk.fdk(scan, p, w, k)
    assert _check_reconstruction(fdk, scan, g, centre, radius, mean_tol, max_tol, zband)


@pytest.mark.parametrize("name,mistake", [("fan", "no_cosine"), ("fan", "no_distance"),
                                          ("cone", "no_distance"), ("parallel", "full_weight"),
                                          ("fan", "no_2pi"), ("cone", "no_magnification")])
def test_planted_mistakes_fail_the_reconstruction_pins(oracle_mod, fdk, monkeypatch, name,
                                                       mistake):
    make, mean_tol, max_tol, zband = CASES[name]
    scan, centre, radius, w = make(oracle_mod)
    p = _ball_sinogram(scan, centre, radius)
    if mistake == "no_cosine":
        monkeypatch.setattr(fdk, "cosine_weights", lambda s: np.ones(s.sino_shape))
    elif mistake == "no_distance":
        real = fdk.project

        def project(scan_, G, view, X):
            u, v, W = real(scan_, G, view, X)
            return u, v, np.where(W > 0, 1.0, 0.0)
        monkeypatch.setattr(fdk, "project", project)
    elif mistake == "full_weight":
        w = 2 * w
    elif mistake in ("no_2pi", "no_magnification"):
        real_geom = fdk.view_geometry

        def geometry(scan_):
            G = real_geom(scan_)
            if mistake == "no_2pi":
                G["s"] = G["s"] * 2 * math.pi
            else:
                G["s"] = 1 / (2 * math.pi) + 0 * G["s"]
            return G
        monkeypatch.setattr(fdk, "view_geometry", geometry)
    g = fdk.fdk(scan, p, w, fdk.RAMLAK)
    assert not _check_reconstruction(fdk, scan, g, centre, radius, mean_tol, max_tol, zband)


# ------------------------------------------------------------ short scans (Parker)
def test_parker_conjugate_rays_sum_to_one(fdk):
    """The conjugate of the ray (beta, gamma) is found here from the circle
    geometry (the other end of the chord through the source at beta with
    direction angle beta + pi + gamma); the two weights sum to one."""
    rng = np.random.default_rng(91)
    big = 0.35
    for _ in range(200):
        gamma = rng.uniform(-big, big)
        beta = rng.uniform(0, math.pi + 2 * big)
        S = np.array([math.cos(beta), math.sin(beta)])
        th = beta + math.pi + gamma
        d = np.array([math.cos(th), math.sin(th)])
        # other intersection of S + t d with the unit circle: t = -2 S.d
        Q = S - 2 * np.dot(S, d) * d
        beta2 = math.atan2(Q[1], Q[0])
        while beta2 < beta:
            beta2 += 2 * math.pi
        c = -Q
        gamma2 = math.atan2(c[0] * (-d[1]) - c[1] * (-d[0]), np.dot(c, -d))
        if beta2 > math.pi + 2 * big:
            continue   # conjugate outside the scan: weight must be 1 or the pair is partial
        total = fdk.parker(beta, gamma, big) + fdk.parker(beta2, gamma2, big)
        assert abs(total - 1.0) < 1e-12, (beta, gamma, beta2, gamma2)


def _short_fan_case(oracle_mod, fdk):
    """Fan beam over pi + 2 Gamma, equally spaced views, Parker weights, view
    weights = the angular step."""
    n_u, pu, sid, sdd = 256, 1.0, 150.0, 300.0
    big = math.atan(0.5 * n_u * pu / sdd)
    arc = math.pi + 2 * big
    K = 240
    b = np.arange(K) * arc / (K - 1)
    c, s, zero = np.cos(b), np.sin(b), np.zeros(K)
    frames = [np.stack(x, 1).astype(np.float32) for x in
              ((sid * c, sid * s, zero), (-(sdd - sid) * c, -(sdd - sid) * s, zero),
               (-s, c, zero), (zero, zero, zero + 1))]
    scan = _scan(oracle_mod, "divergent", frames, n_u, 1, pu, 1.0, (1, 96, 96), (1.0, 1.0, 1.0),
                 ndim=2)
    return scan, (25.0, -15.0, 0.0), 22.0, np.full(K, arc / (K - 1))


def test_short_scan_fbp_with_parker_weights(oracle_mod, fdk):
    scan, centre, radius, w = _short_fan_case(oracle_mod, fdk)
    p = _ball_sinogram(scan, centre, radius)
    pw = fdk.parker_weights(scan)
    g = fdk.weighted_backproject(scan, fdk.filter_sinogram_pw(scan, p, w, pw))
    # float64: mean error ~2e-5, max ~3e-4 inside the disc
    assert _check_reconstruction(fdk, scan, g, centre, radius, 1e-3, 5e-3, None)
    # without Parker weights the short scan counts some lines twice: it fails
    g_bad = fdk.weighted_backproject(scan, fdk.filter_sinogram(scan, p, 0.5 * w))
    assert not _check_reconstruction(fdk, scan, g_bad, centre, radius, 1e-3, 5e-3, None)
