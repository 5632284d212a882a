"""The allocation-free forward entry point (ctp_forward_static).

Some callers may not allocate device memory while they run -- applications whose
device memory belongs to their own pool allocator, or loops that must not take
cudaMalloc's implicit synchronisation.  For them ctp_forward_static keeps its
only scratch, the per-view frame table, in a fixed device array.  This file is
collected last so that a run stopping at its first failure has run every other
test already; it also passes on its own in a fresh process.
"""

import numpy as np
import pytest

from cases import TOL_FORWARD, ci, geometry_of, rel_l2, volume_of

pytestmark = pytest.mark.gpu


def test_forward_static_matches_planned_forward_and_oracle_on_consecutive_calls(oracle_mod):
    import torch
    import back_projection_ctp_b300 as ctp

    assert torch.cuda.is_available()
    results = []
    # two calls in a row on different scans: the second reuses (and fully
    # rewrites) the shared frame array that the first one filled
    for idx in (3, 1):
        w = ci.small_cases()[idx]
        f = ci.frames(w)
        geom, volg = geometry_of(w, f), volume_of(w)
        vol_h = ci.phantom(w)
        vol = torch.from_numpy(vol_h).cuda()
        plan = ctp.ctp_plan(geom, volg, "ray")
        ref = torch.empty(plan.sino_shape, dtype=torch.float32, device="cuda")
        ctp.ctp_forward(plan, vol, ref)
        out = torch.full(plan.sino_shape, float("nan"), dtype=torch.float32, device="cuda")
        ctp.ctp_forward_static(geom, volg, vol, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        err = rel_l2(got, ref.cpu().numpy())
        assert err <= TOL_FORWARD, (w.name, err)
        # and directly against the float64 oracle (rays in a cell-face plane,
        # where the + side rule decides, left out as in the parity tests)
        scan = oracle_mod.Scan.from_workload(w, f)
        amb = oracle_mod.ambiguous(scan)
        p_ref = oracle_mod.forward(scan, vol_h)
        err_ref = rel_l2(got[~amb], p_ref[~amb])
        assert err_ref <= TOL_FORWARD, (w.name, err_ref)
        results.append(err)
        plan.destroy()
    assert len(results) == 2


def test_forward_static_rejects_more_views_than_its_array():
    import torch
    import back_projection_ctp_b300 as ctp

    w = ci.small_cases()[1]
    f = ci.frames(w)
    many = {k: np.repeat(v, 4097 // v.shape[0] + 1, axis=0)[:4097] for k, v in f.items()}
    geom = geometry_of(w, many)
    vol = torch.zeros(w.shape, dtype=torch.float32, device="cuda")
    sino = torch.zeros((4097, w.n_v, w.n_u), dtype=torch.float32, device="cuda")
    with pytest.raises(ctp.CtpError) as exc:
        ctp.ctp_forward_static(geom, volume_of(w), vol, sino)
    assert exc.value.status == 12
