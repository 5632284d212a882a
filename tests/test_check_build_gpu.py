"""The kernels stay inside their buffers: the GPU suites rerun against the
bounds-checked library (``libctp_check.so``, compiled with CTP_CHECK), where
every load, store and reduction of the ray, column and plane walks, of the
FDK gather and transpose and of the geometry-gradient walks tests its index
first and counts an index outside its buffer (skipping the access).  The suites' own checks must pass there too, and the autouse
fixture in conftest.py requires zero counted accesses after every test --
small ragged cases, every path, host-buffer chunking and the five workloads at
full size in the benchmark's launch configuration, and the seeded random small
scans (sources inside the grid, one-cell grids, single-row detectors)."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_parity_gpu.py", "tests/test_random_scans_gpu.py", "tests/test_curved_gpu.py",
          "tests/test_fdk_gpu.py", "tests/test_geometry_gpu.py", "tests/test_autograd_gpu.py",
          "tests/test_zz_no_alloc.py"]


def test_walks_stay_in_bounds_in_the_checked_build():
    if os.environ.get("CTP_LIBRARY_VARIANT") == "check":
        pytest.skip("already running against the checked library")
    from back_projection_ctp_b300 import build
    build.build(check=True)
    env = dict(os.environ, CTP_LIBRARY_VARIANT="check")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p",
                        "no:cacheprovider", *SUITES], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=2400)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    assert " passed" in tail, tail

