"""The stratified samples of the full-size parity tests (no GPU): every index
lies in its array, the strata cover the regimes they are named for, and the
per-stratum check catches an error confined to a few elements that a
whole-sample relative L2 lets through."""

import numpy as np
import pytest

import strata
from cases import TOL_FORWARD, TOL_FORWARD_MAX, ci


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_strata_indices_lie_in_their_arrays(idx):
    w = ci.get(idx)
    rng = np.random.default_rng(idx)
    rays = strata.ray_strata(w, rng)
    voxels = strata.voxel_strata(w, rng)
    for name, v in rays.items():
        assert v.size and v.min() >= 0 and v.max() < w.n_rays, name
    for name, v in voxels.items():
        assert v.size and v.min() >= 0 and v.max() < w.n_voxels, name
    if w.ndim == 3:
        D, H, W = w.shape
        k = voxels["z_extreme"] // (H * W)
        assert set(np.unique(k)) == {0, 1, D - 2, D - 1}
        i = voxels["xy_edge"] % W
        j = (voxels["xy_edge"] // W) % H
        assert np.all((i <= 1) | (i >= W - 2) | (j <= 1) | (j >= H - 2))
        rows = (rays["edge_rows"] // w.n_u) % w.n_v
        assert set(np.unique(rows)) == set(range(4)) | set(range(w.n_v - 4, w.n_v))
        rows = (rays["centre_rows"] // w.n_u) % w.n_v
        assert ((w.n_v - 1) // 2) in set(np.unique(rows))
        per = w.n_u * w.n_v
        assert rays["whole_views"].size == 3 * per


def test_check_strata_sees_a_localised_error():
    rng = np.random.default_rng(0)
    want = {"bulk": rng.uniform(1, 2, 100000), "edge": rng.uniform(1, 2, 50)}
    got = {k: v * (1 + 1e-7 * rng.standard_normal(v.size)) for k, v in want.items()}
    strata.check_strata(got, want, TOL_FORWARD, TOL_FORWARD_MAX, "clean")
    # one wrong element at the edge: invisible to a norm over everything ...
    bad = dict(got)
    bad["edge"] = got["edge"].copy()
    bad["edge"][7] *= 1.001
    all_got = np.concatenate([bad["bulk"], bad["edge"]])
    all_want = np.concatenate([want["bulk"], want["edge"]])
    assert np.linalg.norm(all_got - all_want) / np.linalg.norm(all_want) < TOL_FORWARD
    # ... but not to the per-element bound
    with pytest.raises(AssertionError, match="edge"):
        strata.check_strata(bad, want, TOL_FORWARD, TOL_FORWARD_MAX, "planted")
