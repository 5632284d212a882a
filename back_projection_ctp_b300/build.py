"""Build the CUDA library ``libctp.so`` in-tree for sm_103a with nvcc."""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libctp.so")
# bounds-checked debug build (-DCTP_CHECK): every walk access tested and counted
CHECK_LIB = os.path.join(HERE, "libctp_check.so")
# bandwidth probes of the benchmark's L2 roofline (measurement only)
PROBE_LIB = os.path.join(HERE, "libctp_probe.so")
PROBE_SOURCE = "ctp_probe.cu"
SOURCES = ["ctp_api.cu"]
DEPS = ["ctp_api.cu", "ctp_ray.cuh", "ctp_column.cuh", "ctp_plane.cuh", "ctp_fdk.cuh",
        "ctp_geometry.cuh", "ctp_internal.h", "ctp_check.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _newest_input():
    paths = [os.path.join(CSRC, d) for d in DEPS] + [os.path.join(ROOT, "include", "ctp.h"),
                                                      os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, check: bool = False) -> str:
    """Build ``libctp.so`` (``check``: the bounds-checked ``libctp_check.so``)."""
    lib = CHECK_LIB if check else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-I", os.path.join(ROOT, "include"), "-o", tmp]
    if check:
        cmd += ["-DCTP_CHECK"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def build_probe(force: bool = False) -> str:
    """Build ``libctp_probe.so``, the benchmark's L2 bandwidth probes."""
    src = os.path.join(CSRC, PROBE_SOURCE)
    if (not force and os.path.exists(PROBE_LIB)
            and os.path.getmtime(PROBE_LIB) >= os.path.getmtime(src)):
        return PROBE_LIB
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = PROBE_LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-shared", "-o", tmp, src], check=True)
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


if __name__ == "__main__":
    if "--probe" in sys.argv:
        print(build_probe(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                    check="--check" in sys.argv))
