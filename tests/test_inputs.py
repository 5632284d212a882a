"""Checks of the seeded input generators (workload frames and phantoms)."""

import math

import numpy as np
import pytest

import ctp_inputs as ci


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_frames_geometry(idx):
    w = ci.get(idx)
    f = ci.frames(w)
    for key in ("src", "det_centre", "det_u", "det_v"):
        assert f[key].dtype == np.float32 and f[key].shape == (w.n_views, 3)
    np.testing.assert_allclose(np.linalg.norm(f["det_u"], axis=1), 1, rtol=1e-6)
    np.testing.assert_allclose(np.linalg.norm(f["det_v"], axis=1), 1, rtol=1e-6)
    if w.beam == "parallel":
        np.testing.assert_allclose(np.linalg.norm(f["src"], axis=1), 1, rtol=1e-6)
        ang = np.arctan2(f["src"][:, 1], f["src"][:, 0]) % math.pi
        np.testing.assert_allclose(np.sort(ang), np.arange(w.n_views) * math.pi / w.n_views,
                                   atol=1e-6)
    else:
        src, cen = f["src"].astype(float), f["det_centre"].astype(float)
        np.testing.assert_allclose(np.linalg.norm(src[:, :2], axis=1), w.sid, rtol=1e-6)
        np.testing.assert_allclose(np.linalg.norm(src - cen, axis=1), w.sdd, rtol=1e-6)
        # detector u axis is perpendicular to the central ray
        cr = (cen - src) / w.sdd
        assert np.abs((cr * f["det_u"]).sum(1)).max() < 1e-6
    if w.trajectory == "helical":
        z = f["src"][:, 2].astype(float)
        np.testing.assert_allclose(np.diff(z), w.table_per_turn * (w.arc / w.n_views) / (2 * math.pi),
                                   rtol=1e-4)
        assert abs(z[0] - w.z_start) < 1e-6
        assert abs(z[-1] - (w.z_start + 4 * w.table_per_turn * (w.n_views - 1) / w.n_views)) < 1e-3


def test_phantom_2d_matches_definition():
    w = ci.small_cases()[1]
    vol = ci.phantom(w)
    from ctp_inputs.phantom import shapes
    centres, semi, R, inten = shapes(w)
    D, H, W = w.shape
    dz, dy, dx = w.spacing
    ox, oy, _ = w.origin
    rng = np.random.default_rng(0)
    for _ in range(300):
        j, i = rng.integers(0, H), rng.integers(0, W)
        p = np.array([ox + (i + 0.5) * dx, oy + (j + 0.5) * dy])
        val = 0.0
        for n in range(w.n_shapes):
            q = R[n].T @ (p - centres[n])
            if (q[0] / semi[n][0]) ** 2 + (q[1] / semi[n][1]) ** 2 <= 1.0:
                val += inten[n]
        assert abs(vol[0, j, i] - val) < 1e-6


def test_phantom_3d_matches_definition():
    w = ci.small_cases()[3]
    vol = ci.phantom(w)
    from ctp_inputs.phantom import shapes
    centres, semi, R, inten = shapes(w)
    dz, dy, dx = w.spacing
    ox, oy, oz = w.origin
    rng = np.random.default_rng(1)
    hits = 0
    for _ in range(300):
        k, j, i = (rng.integers(0, s) for s in w.shape)
        p = np.array([ox + (i + 0.5) * dx, oy + (j + 0.5) * dy, oz + (k + 0.5) * dz])
        val = sum(inten[n] for n in range(w.n_shapes)
                  if (((R[n].T @ (p - centres[n])) / semi[n]) ** 2).sum() <= 1.0)
        hits += val > 0
        assert abs(vol[k, j, i] - val) < 1e-6
    assert hits > 30
    # rotations are orthonormal
    for n in range(w.n_shapes):
        np.testing.assert_allclose(R[n] @ R[n].T, np.eye(3), atol=1e-12)


def test_generators_are_seeded():
    w = ci.small_cases()[4]
    assert np.array_equal(ci.phantom(w), ci.phantom(w))
    assert np.array_equal(ci.sinogram_noise(w), ci.sinogram_noise(w))
    assert ci.sinogram_noise(w).dtype == np.float32
    assert ci.phantom(w).max() > 0.0


def test_scaled_keeps_physical_extent():
    for idx, w in ci.WORKLOADS.items():
        s = ci.small_cases()[idx]
        for a in range(3):
            ext_full = w.shape[a] * w.spacing[a]
            ext_small = s.shape[a] * s.spacing[a]
            if w.ndim == 3 or a > 0:
                assert abs(ext_full - ext_small) < 1e-9 * ext_full
        assert abs(w.n_u * w.pitch_u - s.n_u * s.pitch_u) < 1e-9 * w.n_u * w.pitch_u
        assert abs(w.offset_u * w.pitch_u - s.offset_u * s.pitch_u) < 1e-9
