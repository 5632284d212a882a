"""Stratified samples of rays and voxels for the full-size parity tests.

A whole-array norm over a few hundred random samples cannot see an error
confined to one band of the volume or one group of detector rows, so the
samples deliberately include the places where the GPU walks change regime:

rays (flat indices into the (n_views, n_v, n_u) sinogram)
  whole_views  every pixel of a few whole views (every detector column, every
               row -- the edges of the volume's shadow included)
  centre_rows  the detector rows around the source's height in many views:
               their rays straddle the source's z, so one warp of the column
               walk holds rows stepping up and rows stepping down in z
  edge_rows    the first and last detector rows in many views: the rays that
               leave the grid through its top or bottom, where the column walk
               switches between its z-checked and check-free slab ranges
  random       uniformly drawn rays

voxels (flat indices into the (D, H, W) volume)
  z_extreme    the two first and two last z slabs
  xy_edge      cells in the two outermost x columns and y rows on each side,
               next to the walks' zero halo
  z_centre     the two z slabs around the volume centre (the source plane of
               the circular scans)
  lines        one whole line of cells along each axis through the volume centre
  random       uniformly drawn voxels

2-D scans are small enough to compare whole: one stratum "all" each.
"""

import numpy as np


def ray_strata(w, rng, n_views_whole=3, n_views_rows=32, n_random=8000):
    V, NV, NU = w.n_views, w.n_v, w.n_u
    if w.ndim == 2:
        return {"all": np.arange(w.n_rays, dtype=np.int64)}
    per = NV * NU
    out = {}
    views = np.unique(np.linspace(0, V - 1, n_views_whole).round().astype(np.int64))
    out["whole_views"] = (views[:, None] * per + np.arange(per)[None, :]).ravel()
    many = np.sort(rng.choice(V, min(V, n_views_rows), replace=False)).astype(np.int64)
    c = (NV - 1) // 2
    centre = np.arange(max(0, c - 2), min(NV, c + 3), dtype=np.int64)
    edge = np.unique(np.concatenate([np.arange(min(4, NV)), np.arange(max(0, NV - 4), NV)]))
    for name, rows in (("centre_rows", centre), ("edge_rows", edge)):
        idx = (many[:, None, None] * per + rows[None, :, None] * NU +
               np.arange(NU)[None, None, :]).ravel()
        out[name] = idx
    out["random"] = np.sort(rng.choice(w.n_rays, min(w.n_rays, n_random), replace=False))
    return out


def voxel_strata(w, rng, n_per=500, n_random=4000):
    D, H, W = w.shape
    if w.ndim == 2:
        return {"all": np.arange(w.n_voxels, dtype=np.int64)}

    def flat(k, j, i):
        return (np.asarray(k, np.int64) * H + np.asarray(j, np.int64)) * W + np.asarray(i, np.int64)

    out = {}
    ks = np.unique([0, min(1, D - 1), max(D - 2, 0), D - 1])
    out["z_extreme"] = np.concatenate([flat(k, rng.integers(0, H, n_per), rng.integers(0, W, n_per))
                                       for k in ks])
    xs = np.unique([0, min(1, W - 1), max(W - 2, 0), W - 1])
    ys = np.unique([0, min(1, H - 1), max(H - 2, 0), H - 1])
    parts = [flat(rng.integers(0, D, n_per), rng.integers(0, H, n_per), i) for i in xs]
    parts += [flat(rng.integers(0, D, n_per), j, rng.integers(0, W, n_per)) for j in ys]
    out["xy_edge"] = np.concatenate(parts)
    kc = np.unique([max(D // 2 - 1, 0), D // 2])
    out["z_centre"] = np.concatenate([flat(k, rng.integers(0, H, n_per), rng.integers(0, W, n_per))
                                      for k in kc])
    out["lines"] = np.concatenate([flat(np.arange(D), H // 2, W // 2), flat(D // 2, np.arange(H), W // 2),
                                   flat(D // 2, H // 2, np.arange(W))])
    out["random"] = rng.choice(w.n_voxels, min(w.n_voxels, n_random), replace=False).astype(np.int64)
    return {k: np.unique(v) for k, v in out.items()}


def check_strata(got, want, tol_l2, tol_max, what):
    """got, want: {stratum: values}.  Per stratum: relative L2 <= tol_l2 (strata
    whose reference is not all zero) and, element by element, |got - want| <=
    tol_max * max|want| with the scale taken over every stratum.  Returns
    {stratum: (relative L2, max |error| / scale)}."""
    scale = max((float(np.max(np.abs(r))) for r in want.values() if np.size(r)), default=0.0)
    report = {}
    for name, r in want.items():
        g = np.asarray(got[name], np.float64)
        r = np.asarray(r, np.float64)
        assert g.shape == r.shape, (what, name, g.shape, r.shape)
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite values"
        err = np.abs(g - r)
        worst = float(err.max()) if err.size else 0.0
        den = float(np.linalg.norm(r))
        l2 = float(np.linalg.norm(g - r) / den) if den > 0 else float(np.linalg.norm(g))
        report[name] = (l2, worst / scale if scale > 0 else worst)
        if den > 0:
            assert l2 <= tol_l2, f"{what} {name}: relative L2 {l2:.3e} > {tol_l2:.0e}"
        assert worst <= tol_max * scale, (
            f"{what} {name}: max |error| {worst:.3e} > {tol_max:.0e} x max|ref| {scale:.3e} "
            f"(element {int(np.argmax(err))} of the stratum)")
    return report
