"""The view-partitioned projector's host logic on the CPU: shard arithmetic, and
a 2- and 3-rank gloo run in which every rank's shard operator is the float64
oracle (injected), checked against the oracle on the whole scan -- the stacked
forward rows and the all-reduced backward."""

import json
import os
import socket
import subprocess
import sys

import pytest

from back_projection_ctp_b300.partition import view_shard

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("n_views", [0, 1, 5, 24, 720, 1441])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_view_shards_tile_the_views_in_rank_order(n_views, world):
    ranges = [view_shard(n_views, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n_views
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [v1 - v0 for v0, v1 in ranges]
    assert min(sizes) >= 0 and max(sizes) - min(sizes) <= 1


def test_bad_shard_requests_are_rejected():
    for args in ((10, 0, 0), (10, 2, 2), (10, 2, -1), (-1, 2, 0)):
        with pytest.raises(ValueError):
            view_shard(*args)


_WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r})
sys.path.insert(0, os.path.join({root!r}, "tests"))
import numpy as np
import torch
import torch.distributed as dist
import ctp_inputs as ci
import oracle
from back_projection_ctp_b300.partition import ViewShardedProjector
from cases import geometry_of, volume_of

dist.init_process_group("gloo")
w = ci.small_cases()[{idx}]
f = ci.frames(w)
geom, volg = geometry_of(w, f), volume_of(w)


def scan_of(g, v):
    return oracle.Scan(w.beam, g.src, g.det_centre, g.det_u, g.det_v, g.n_u, g.n_v, g.pitch_u,
                       g.pitch_v, v.shape, v.spacing, v.origin, g.offset_u, g.offset_v, w.ndim)


class OracleShard:
    # the float64 oracle on one rank's views (host tensors, float64 results)
    def __init__(self, g, v):
        self.scan = scan_of(g, v)

    def forward(self, vol, sino):
        if self.scan.n_rays:
            sino.copy_(torch.from_numpy(oracle.forward(self.scan, vol.numpy())))
        return sino

    def backward(self, sino, vol):
        vol.zero_()
        if self.scan.n_rays:
            vol.copy_(torch.from_numpy(oracle.backward(self.scan, sino.numpy().ravel())))
        return vol


proj = ViewShardedProjector(geom, volg, make_operator=OracleShard)
vol = torch.from_numpy(ci.phantom(w))
y = ci.sinogram_noise(w)
sino_local = torch.zeros(proj.local_sino_shape, dtype=torch.float64)
proj.forward(vol, sino_local)
full = proj.gather_sinogram(sino_local).numpy()
g = torch.full(w.shape, float("nan"), dtype=torch.float64)
proj.backward(torch.from_numpy(np.ascontiguousarray(y[proj.v0:proj.v1])), g)

scan = scan_of(geom, volg)
p_ref = oracle.forward(scan, ci.phantom(w))
g_ref = oracle.backward(scan, y.ravel())
rec = dict(rank=proj.rank, world=proj.world, v0=proj.v0, v1=proj.v1,
           fwd=float(np.max(np.abs(full - p_ref)) / np.max(np.abs(p_ref))),
           bwd=float(np.max(np.abs(g.numpy() - g_ref)) / np.max(np.abs(g_ref))),
           shape=list(full.shape))
with open(os.path.join({out!r}, f"rank{{proj.rank}}.json"), "w") as fh:
    fh.write(json.dumps(rec))
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("idx,world", [(3, 2), (2, 3)])
def test_view_sharded_pair_over_gloo_ranks(tmp_path, idx, world):
    script = tmp_path / "worker.py"
    script.write_text(_WORKER.format(root=ROOT, out=str(tmp_path), idx=idx))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={world}", "--master-addr", "127.0.0.1", "--master-port",
           str(_free_port()), str(script)]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-3000:]
    recs = sorted((json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(world)),
                  key=lambda r: r["rank"])
    import ctp_inputs as ci
    w = ci.small_cases()[idx]
    assert [(r["v0"], r["v1"]) for r in recs] == [view_shard(w.n_views, world, r)
                                                   for r in range(world)]
    for r in recs:
        assert r["world"] == world and r["shape"] == [w.n_views, w.n_v, w.n_u]
        # each ray is computed by exactly one rank: the stacked rows are the whole
        # scan's forward, and the summed partials its backward (up to the order
        # of the float64 sums)
        assert r["fwd"] <= 1e-14, r
        assert r["bwd"] <= 1e-12, r
