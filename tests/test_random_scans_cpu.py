"""The oracle on the random small scans of the GPU parity sweep, pinned to the
brute-force path (every cell's box clipped against every ray, no traversal):
values to 1e-12 and piece counts exactly, rays in a cell-face plane left out of
the values (they are where the two paths may legitimately differ)."""

import numpy as np
import pytest

from random_scans import N_CASES, random_scan


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_scan_traversal_equals_brute_force(oracle_mod, seed):
    beam, ndim, frames, n_u, n_v, pu, pv, ou, ov, shape, spacing = random_scan(seed)
    D, H, W = shape
    origin = (-0.5 * W * spacing[2], -0.5 * H * spacing[1], -0.5 * D * spacing[0])
    scan = oracle_mod.Scan(beam, *frames, n_u, n_v, pu, pv, shape, spacing, origin, ou, ov, ndim)
    vol = np.random.default_rng(9000 + seed).uniform(-1, 1, shape).astype(np.float32)
    amb = oracle_mod.ambiguous(scan)
    got = oracle_mod.forward(scan, vol)
    want = oracle_mod.brute_forward(scan, vol)
    scale = max(float(np.abs(want).max()), 1e-300)
    np.testing.assert_allclose(got[~amb], want[~amb], rtol=1e-12, atol=1e-12 * scale)
    assert oracle_mod.segment_count(scan) == oracle_mod.brute_count(scan)
