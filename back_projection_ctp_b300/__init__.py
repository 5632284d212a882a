"""B300-native ray-driven Siddon projector pair (forward projection and its
matched backprojection) behind the C ABI of ``include/ctp.h``.

The entry points carry the C names: :func:`ctp_plan`, :func:`ctp_forward`,
:func:`ctp_backward`, :func:`ctp_segment_count`, :func:`ctp_forward_host`,
:func:`ctp_backward_host`, :func:`ctp_destroy`, :func:`ctp_status_string`, the
allocation-free :func:`ctp_forward_static`, and the analytical FBP / FDK operators
:func:`ctp_ramp_filter`, :func:`ctp_weighted_backproject`,
:func:`ctp_weighted_backproject_transpose`, :func:`ctp_fdk` and
:func:`ctp_parker_weights`, and the geometry gradients :func:`ctp_geometry_vjp` and
:func:`ctp_surface_vjp`.
:class:`ViewShardedProjector` runs the pair view-sharded over a
``torch.distributed`` group (one GPU per rank, one all-reduce per backward).
"""

from ._binding import (EXPORTS, CtpError, Geometry, Plan, Volume, ctp_backward,
                       ctp_backward_host, ctp_check_violations, ctp_destroy, ctp_fdk,
                       ctp_forward, ctp_forward_host, ctp_forward_static, ctp_geometry_vjp,
                       ctp_parker_weights, ctp_plan, ctp_ramp_filter, ctp_segment_count,
                       ctp_status_string, ctp_surface_vjp, ctp_weighted_backproject,
                       ctp_weighted_backproject_transpose, full_scan_view_weights,
                       load_library)
from .partition import ViewShardedProjector, shard_geometry, view_shard

__all__ = ["EXPORTS", "CtpError", "Geometry", "Plan", "Volume", "ctp_backward",
           "ctp_backward_host", "ctp_check_violations", "ctp_destroy", "ctp_fdk",
           "ctp_forward", "ctp_forward_host", "ctp_forward_static", "ctp_geometry_vjp",
           "ctp_parker_weights", "ctp_plan", "ctp_ramp_filter", "ctp_segment_count",
           "ctp_status_string", "ctp_surface_vjp", "ctp_weighted_backproject",
           "ctp_weighted_backproject_transpose", "full_scan_view_weights", "load_library",
           "ViewShardedProjector", "shard_geometry", "view_shard"]
