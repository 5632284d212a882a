"""The view-partitioned pair on the GPU.

One B300 per run, so two things are checked here: (1) shard plans -- the
scan's views split in 2 and 3 contiguous ranges, each planned on its own as a
rank would -- give, stacked, the whole plan's forward and, summed, its
backward; (2) ViewShardedProjector in a one-rank NCCL group (the collective
path itself: all-reduce of the volume on the device) equals the plain calls.
The 2- and 3-rank exchange runs on the CPU over gloo (test_partition_cpu.py).
"""

import os
import socket
import subprocess
import sys


import pytest

from cases import ci, geometry_of, rel_l2, volume_of

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("idx", [1, 2, 3, 5])
@pytest.mark.parametrize("world", [2, 3])
def test_shard_plans_stack_to_the_whole_scan(idx, world):
    import torch
    import back_projection_ctp_b300 as ctp

    w = ci.small_cases()[idx]
    geom, volg = geometry_of(w, ci.frames(w)), volume_of(w)
    vol = torch.from_numpy(ci.phantom(w)).cuda()
    y = torch.from_numpy(ci.sinogram_noise(w)).cuda()
    full = ctp.ctp_plan(geom, volg)
    p_ref = torch.empty(full.sino_shape, dtype=torch.float32, device="cuda")
    g_ref = torch.empty(full.vol_shape, dtype=torch.float32, device="cuda")
    ctp.ctp_forward(full, vol, p_ref)
    ctp.ctp_backward(full, y, g_ref)

    p = torch.full(full.sino_shape, float("nan"), dtype=torch.float32, device="cuda")
    g = torch.zeros(full.vol_shape, dtype=torch.float32, device="cuda")
    part = torch.empty_like(g)
    for r in range(world):
        v0, v1 = ctp.view_shard(w.n_views, world, r)
        plan = ctp.ctp_plan(ctp.shard_geometry(geom, v0, v1), volg)
        assert plan.path == full.path
        ctp.ctp_forward(plan, vol, p[v0:v1])
        ctp.ctp_backward(plan, y[v0:v1].contiguous(), part)
        g += part
        plan.destroy()
    torch.cuda.synchronize()
    # the same rays in the same kernels: the stacked rows equal the whole
    # plan's (the 2-D forward splits long rays into a number of chunks that
    # depends on the plan's ray count, hence the tolerance)
    assert rel_l2(p.cpu().numpy(), p_ref.cpu().numpy()) <= 1e-6
    assert rel_l2(g.cpu().numpy(), g_ref.cpu().numpy()) <= 1e-6
    full.destroy()


_WORKER = r"""
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})

import torch
import torch.distributed as dist
import back_projection_ctp_b300 as ctp
import ctp_inputs as ci
from cases import geometry_of, rel_l2, volume_of

torch.cuda.set_device(0)
dist.init_process_group("nccl", init_method="tcp://127.0.0.1:{port}", rank=0, world_size=1)
w = ci.small_cases()[3]
geom, volg = geometry_of(w, ci.frames(w)), volume_of(w)
vol = torch.from_numpy(ci.phantom(w)).cuda()
y = torch.from_numpy(ci.sinogram_noise(w)).cuda()
proj = ctp.ViewShardedProjector(geom, volg)
assert (proj.world, proj.rank, proj.v0, proj.v1) == (1, 0, 0, w.n_views)
p = torch.empty(proj.local_sino_shape, dtype=torch.float32, device="cuda")
g = torch.empty(w.shape, dtype=torch.float32, device="cuda")
proj.forward(vol, p)
proj.backward(y, g)
plan = ctp.ctp_plan(geom, volg)
p_ref = torch.empty_like(p)
g_ref = torch.empty_like(g)
ctp.ctp_forward(plan, vol, p_ref)
ctp.ctp_backward(plan, y, g_ref)
# a one-rank all-reduce through NCCL on the device
t = torch.arange(8, dtype=torch.float32, device="cuda")
proj.all_reduce(t)
torch.cuda.synchronize()
assert torch.equal(t, torch.arange(8, dtype=torch.float32, device="cuda"))
assert torch.equal(p, p_ref)
assert rel_l2(g.cpu().numpy(), g_ref.cpu().numpy()) <= 1e-6
proj.destroy()
plan.destroy()
dist.destroy_process_group()
print("ONE_RANK_OK")
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_projector_in_a_one_rank_nccl_group(tmp_path):
    script = tmp_path / "one_rank.py"
    script.write_text(_WORKER.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                                     port=_free_port()))
    env = dict(os.environ, NCCL_NVLS_ENABLE="0")
    out = subprocess.run([sys.executable, str(script)], capture_output=True, text=True,
                         timeout=300, env=env)
    assert out.returncode == 0 and "ONE_RANK_OK" in out.stdout, out.stderr[-3000:]


def test_bench_partitioned_mode_prints_one_strong_scaling_line():
    import json
    out = subprocess.run([sys.executable, "bench.py", "--partition", "views", "--config", "3",
                          "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["scaling"] == "strong" and rec["config"]["parallelism"] == "views1"
    assert rec["value"] > 0 and rec["e2e"]["value"] > 0
    assert rec["config"]["views_per_rank"] == [[0, 360]]
