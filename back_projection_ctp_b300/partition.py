"""View-partitioned projector pair over several processes, one GPU each.

The pages' default multi-GPU mode shards the projections and replicates the
volume (diffct 2.1.0 -> 2.2.1, README "Multi-GPU and multi-node":
``partition="views"``), and sums the ranks' partial results on the devices
before anything is downloaded (CHANGELOG 2.2.0, "Changed": local GPU and NCCL
reductions occur before completed-result downloads).  Here:

* every rank holds the whole volume and plans only its contiguous shard of
  views ``[v0, v1)`` (the per-view frames of those views; the operator's rays
  are independent, so a shard's plan walks exactly the rays of those views);
* forward: each rank writes its own sinogram rows; no exchange;
* backward: each rank backprojects its rows into a full-volume partial and one
  all-reduce (sum) over the group turns the partials into ``A^T y`` on every
  rank.

The collective is ``torch.distributed.all_reduce`` on the volume tensor (NCCL
for CUDA tensors, gloo for host tensors); the projector calls are the C ABI's.
The operator a rank runs on its shard can be injected (``make_operator``), so
the sharding and the reduction are testable on the CPU.
"""

from __future__ import annotations

import dataclasses

import numpy as np


def view_shard(n_views: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, balanced view range [v0, v1) of ``rank`` among ``world``
    ranks: sizes differ by at most one, the ranges tile [0, n_views) in rank
    order, and ranks beyond the views get empty ranges."""
    if world < 1 or not 0 <= rank < world or n_views < 0:
        raise ValueError(f"bad shard request: n_views={n_views}, world={world}, rank={rank}")
    return n_views * rank // world, n_views * (rank + 1) // world


def shard_geometry(geometry, v0: int, v1: int):
    """The scan restricted to views [v0, v1) (frames sliced; detector unchanged)."""
    return dataclasses.replace(
        geometry, src=np.asarray(geometry.src)[v0:v1], det_centre=np.asarray(geometry.det_centre)[v0:v1],
        det_u=np.asarray(geometry.det_u)[v0:v1], det_v=np.asarray(geometry.det_v)[v0:v1])


class _CudaShardOperator:
    """The C-ABI pair on one rank's shard: a plan of the shard's views."""

    def __init__(self, geometry, volume, path="auto", options=None):
        from . import _binding as b
        self._b = b
        self.plan = b.ctp_plan(geometry, volume, path, options=options)

    def forward(self, vol, sino):
        return self._b.ctp_forward(self.plan, vol, sino)

    def backward(self, sino, vol):
        return self._b.ctp_backward(self.plan, sino, vol)

    def destroy(self):
        self.plan.destroy()


class ViewShardedProjector:
    """A = the stacked rows of every rank's shard; A^T = the sum of their
    transposes.  ``group``: a torch.distributed process group (default: the
    world group when initialised, else a single rank).  ``make_operator(geometry,
    volume)`` builds the shard's operator (default: a CUDA plan on the current
    device)."""

    def __init__(self, geometry, volume, path="auto", options=None, group=None,
                 make_operator=None):
        import torch.distributed as dist
        self.group = group
        if dist.is_available() and dist.is_initialized():
            self.world = dist.get_world_size(group)
            self.rank = dist.get_rank(group)
        else:
            self.world, self.rank = 1, 0
        self.n_views = int(np.asarray(geometry.src).reshape(-1, 3).shape[0])
        self.v0, self.v1 = view_shard(self.n_views, self.world, self.rank)
        self.geometry = geometry
        self.volume = volume
        self.local_geometry = shard_geometry(geometry, self.v0, self.v1)
        if make_operator is None:
            self.op = _CudaShardOperator(self.local_geometry, volume, path, options)
        else:
            self.op = make_operator(self.local_geometry, volume)
        self.local_sino_shape = (self.v1 - self.v0, int(geometry.n_v), int(geometry.n_u))

    def forward(self, vol, sino_local):
        """This rank's rows of A vol into ``sino_local`` (v1 - v0, n_v, n_u)."""
        return self.op.forward(vol, sino_local)

    def backward(self, sino_local, vol):
        """vol <- sum over ranks of A_rank^T sino_rank, on every rank."""
        self.op.backward(sino_local, vol)
        self.all_reduce(vol)
        return vol

    def all_reduce(self, t):
        if self.world > 1:
            import torch.distributed as dist
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=self.group)
        return t

    def gather_sinogram(self, sino_local):
        """The whole (n_views, n_v, n_u) sinogram on every rank (the shards are
        padded to the largest one for the collective and trimmed after)."""
        if self.world == 1:
            return sino_local
        import torch
        import torch.distributed as dist
        per = -(-self.n_views // self.world)
        pad = torch.zeros((per,) + self.local_sino_shape[1:], dtype=sino_local.dtype,
                          device=sino_local.device)
        pad[:sino_local.shape[0]] = sino_local
        parts = [torch.empty_like(pad) for _ in range(self.world)]
        dist.all_gather(parts, pad, group=self.group)
        rows = [view_shard(self.n_views, self.world, r) for r in range(self.world)]
        return torch.cat([p[:v1 - v0] for p, (v0, v1) in zip(parts, rows)], 0)

    def destroy(self):
        if hasattr(self.op, "destroy"):
            self.op.destroy()
