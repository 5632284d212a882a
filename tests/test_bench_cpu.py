"""CPU checks of bench.py's host logic: the reference (oracle) arm, argument
rules, and the multi-rank reduction over a 2-rank gloo group."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "1",
                          "--steps", "1", "--warmup", "3", "--ref-budget", "0.2"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "Gseg/s" and rec["value"] > 0
    cpu = rec["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1
    # the step's rate is the harmonic combination of the forward and backward rates
    f, b = cpu["forward_gseg_per_s"], cpu["backward_gseg_per_s"]
    assert abs(2.0 / (1.0 / f + 1.0 / b) - cpu["value"]) <= 1e-9 * cpu["value"]
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["value"] == rec["value"]
    assert rec["config"]["workload"] == "c1_parallel2d_64"


def test_warmup_below_three_is_rejected():
    out = subprocess.run([sys.executable, "bench.py", "--warmup", "2"], cwd=ROOT,
                         capture_output=True, text=True, timeout=120)
    assert out.returncode != 0 and "warmup" in out.stderr


_WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
world, rank, local = bench.dist_setup(2)
bench.barrier(world)
v = bench.max_over_ranks(float(rank + 1) * 1.5, world)
# one file per rank: lines printed by two processes to one pipe can interleave
with open(os.path.join({out!r}, f"rank{{rank}}.json"), "w") as fh:
    fh.write(json.dumps({{"rank": rank, "max": v}}))
dist.destroy_process_group()
"""


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    script = tmp_path / "worker.py"
    script.write_text(_WORKER.format(root=ROOT, out=str(tmp_path)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(script)]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    recs = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in (0, 1)]
    assert sorted(r["rank"] for r in recs) == [0, 1]
    assert all(r["max"] == 3.0 for r in recs)


def test_reference_arm_under_two_ranks_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--config", "1", "--steps", "1", "--warmup", "3",
           "--ref-budget", "0.2"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["impl"] == "reference"


def test_stored_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """roofline.traffic comes from profiles/traffic.json only while the profiled
    kernel's own sources (comments and blank space aside) match the capture."""
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    for name in os.listdir(bench.CSRC):
        (csrc / name).write_text(open(os.path.join(bench.CSRC, name)).read())
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    kernel = "column_forward_kernel"
    h = bench.source_hash(kernel)
    record = tmp_path / "traffic.json"
    record.write_text(json.dumps({kernel: {"c4_cone_512_aniso": {
        "dram_bytes_per_launch": 123.0, "source_hash": h, "ncu": {"l1tex_pct": 50.0}}}}))
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(record))
    assert bench.stored_traffic(kernel, "c4_cone_512_aniso") == 123.0
    assert bench.stored_ncu(kernel, "c4_cone_512_aniso") == {"l1tex_pct": 50.0}
    f = csrc / "ctp_column.cuh"
    text = f.read_text()
    f.write_text(text.replace("namespace ctp {", "namespace ctp {\n// a new comment\n\n", 1))
    assert bench.source_hash(kernel) == h  # comments and blank lines do not count
    assert bench.stored_traffic(kernel, "c4_cone_512_aniso") == 123.0
    f.write_text(text.replace("constexpr int kHalo = 2;", "constexpr int kHalo = 3;", 1))
    assert bench.source_hash(kernel) != h
    assert bench.stored_traffic(kernel, "c4_cone_512_aniso") is None
    assert bench.stored_ncu(kernel, "c4_cone_512_aniso") is None
    (csrc / "ctp_fdk.cuh").write_text("// unrelated file changed\nint x;\n")
    f.write_text(text)
    assert bench.stored_traffic(kernel, "c4_cone_512_aniso") == 123.0


def test_stored_traffic_record_is_well_formed():
    """Every committed ncu record names its capture and the hash it belongs to."""
    sys.path.insert(0, ROOT)
    import bench
    with open(bench.TRAFFIC_JSON) as fh:
        rec = json.load(fh)
    for kernel, by_workload in rec.items():
        for workload, entry in by_workload.items():
            assert entry["dram_bytes_per_launch"] > 0, (kernel, workload)
            assert len(entry["source_hash"]) == 16 and entry["captured_on"], (kernel, workload)
