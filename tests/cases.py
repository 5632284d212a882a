"""Test-side glue: workload -> C-ABI geometry / volume, error metrics."""

import numpy as np

import ctp_inputs as ci


def geometry_of(w, frames):
    from back_projection_ctp_b300 import Geometry
    return Geometry(ndim=w.ndim, beam=w.beam, src=frames["src"], det_centre=frames["det_centre"],
                    det_u=frames["det_u"], det_v=frames["det_v"], n_u=w.n_u, n_v=w.n_v,
                    pitch_u=w.pitch_u, pitch_v=w.pitch_v, offset_u=w.offset_u,
                    offset_v=w.offset_v)


def volume_of(w):
    from back_projection_ctp_b300 import Volume
    return Volume(shape=w.shape, spacing=w.spacing, origin=w.origin)


def rel_l2(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / den) if den > 0 else float(np.linalg.norm(got))


def max_rel_err(got, want):
    """max |got - want| / max |want| (element by element, float64)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    scale = float(np.max(np.abs(want))) if want.size else 0.0
    err = float(np.max(np.abs(got - want))) if want.size else 0.0
    return err / scale if scale > 0 else err


def adjoint_mismatch(Ax, y, x, Aty):
    """|<Ax, y> - <x, A^T y>| / (||Ax|| ||y||) and the raw relative value."""
    lhs = float(np.dot(np.asarray(Ax, np.float64).ravel(), np.asarray(y, np.float64).ravel()))
    rhs = float(np.dot(np.asarray(x, np.float64).ravel(), np.asarray(Aty, np.float64).ravel()))
    cs = float(np.linalg.norm(np.asarray(Ax, np.float64)) * np.linalg.norm(np.asarray(y, np.float64)))
    return abs(lhs - rhs) / cs, abs(lhs - rhs) / max(abs(lhs), 1e-300)


# Tolerances of the pair against the float64 oracle (forward and the
# atomics-ordered backward) and of the GPU pair's own adjoint identity.
TOL_FORWARD = 1e-5
TOL_BACKWARD = 1e-4
TOL_ADJOINT = 1e-5
# Element by element (the per-pixel / per-voxel reading of the same bars):
# |gpu - oracle| <= tol * max|oracle| over the compared sample.  Float32
# accumulation of a path sum of ~1e3 pieces errs by ~1e-7 of the largest
# values; the backward's atomics add order-dependent rounding of the same size.
TOL_FORWARD_MAX = 1e-5
TOL_BACKWARD_MAX = 1e-4

__all__ = ["ci", "geometry_of", "volume_of", "rel_l2", "max_rel_err", "adjoint_mismatch", "TOL_FORWARD",
           "TOL_BACKWARD", "TOL_ADJOINT", "TOL_FORWARD_MAX", "TOL_BACKWARD_MAX"]
