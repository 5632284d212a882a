"""Seeded random scans: the CUDA pair against the float64 oracle across the
space of small geometries -- beam type, arbitrary or vertical detector axes
(column path), circular arcs with the source inside or outside the grid, 2-D
slices (plane path), grid sizes from one cell upwards, anisotropic spacing,
detector sizes, pitches and offsets -- each on every path AUTO takes and on the
ray path.  Rays in a cell-face plane are left out as in the other parity tests.
"""

import numpy as np
import pytest

from cases import (TOL_ADJOINT, TOL_BACKWARD, TOL_BACKWARD_MAX, TOL_FORWARD, TOL_FORWARD_MAX,
                   adjoint_mismatch, max_rel_err, rel_l2)
from random_scans import N_CASES, random_scan

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_scan_matches_oracle(oracle_mod, seed):
    import torch
    import back_projection_ctp_b300 as ctp

    beam, ndim, frames, n_u, n_v, pu, pv, ou, ov, shape, spacing = random_scan(seed)
    D, H, W = shape
    origin = (-0.5 * W * spacing[2], -0.5 * H * spacing[1], -0.5 * D * spacing[0])
    scan = oracle_mod.Scan(beam, *frames, n_u, n_v, pu, pv, shape, spacing, origin, ou, ov, ndim)
    geom = ctp.Geometry(ndim=ndim, beam=beam, src=frames[0], det_centre=frames[1],
                        det_u=frames[2], det_v=frames[3], n_u=n_u, n_v=n_v, pitch_u=pu,
                        pitch_v=pv, offset_u=ou, offset_v=ov)
    vol_g = ctp.Volume(shape, spacing, origin)
    rng = np.random.default_rng(8000 + seed)
    vol = rng.uniform(0.0, 1.0, shape).astype(np.float32)
    amb = oracle_mod.ambiguous(scan)
    y = np.where(amb, np.float32(0), rng.standard_normal(scan.sino_shape).astype(np.float32))
    p_ref = oracle_mod.forward(scan, vol)
    g_ref = oracle_mod.backward(scan, y.ravel())
    n_ref = oracle_mod.segment_count(scan)
    paths = {"auto", "ray"}
    for path in sorted(paths):
        plan = ctp.ctp_plan(geom, vol_g, path)
        d_p = torch.empty(plan.sino_shape, device="cuda")
        d_g = torch.full(plan.vol_shape, float("nan"), device="cuda")
        ctp.ctp_forward(plan, torch.from_numpy(vol).cuda(), d_p)
        ctp.ctp_backward(plan, torch.from_numpy(y).cuda(), d_g)
        torch.cuda.synchronize()
        p, g = d_p.cpu().numpy(), d_g.cpu().numpy()
        tag = (seed, plan.path, beam, shape, n_u, n_v)
        if np.abs(p_ref[~amb]).max(initial=0.0) > 0:
            assert rel_l2(p[~amb], p_ref[~amb]) <= TOL_FORWARD, tag
            assert max_rel_err(p[~amb], p_ref[~amb]) <= TOL_FORWARD_MAX, tag
        else:
            assert np.abs(p[~amb]).max(initial=0.0) == 0.0, tag
        if np.abs(g_ref).max() > 0:
            assert rel_l2(g, g_ref) <= TOL_BACKWARD, tag
            assert max_rel_err(g, g_ref) <= TOL_BACKWARD_MAX, tag
        else:
            assert np.abs(g).max() == 0.0, tag
        x = rng.standard_normal(shape).astype(np.float32)
        yy = rng.standard_normal(scan.sino_shape).astype(np.float32)
        d_p2 = torch.empty(plan.sino_shape, device="cuda")
        d_g2 = torch.empty(plan.vol_shape, device="cuda")
        ctp.ctp_forward(plan, torch.from_numpy(x).cuda(), d_p2)
        ctp.ctp_backward(plan, torch.from_numpy(yy).cuda(), d_g2)
        torch.cuda.synchronize()
        Ax, Aty = d_p2.cpu().numpy(), d_g2.cpu().numpy()
        if np.linalg.norm(Ax) > 0:
            cs, raw = adjoint_mismatch(Ax, yy, x, Aty)
            assert cs <= TOL_ADJOINT, (tag, cs, raw)
        assert abs(ctp.ctp_segment_count(plan) - n_ref) <= max(1e-6 * n_ref, 4), tag
        plan.destroy()
