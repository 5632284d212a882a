"""Seeded synthetic inputs for the Siddon projector pair: workloads, frames, phantoms.

This package builds INPUTS only: the five scan workloads (volume grid, detector,
per-view source / detector frames), voxelised random-ellipse and random-ellipsoid
phantoms, and N(0,1) sinograms.  It holds none of the projector's arithmetic
(no ray set-up, no traversal, no intersection lengths), so that both the float64
oracle and the CUDA path can be fed from it without sharing any of the method.

The workload shapes follow the diffct release pages (my.diffend.io, diffct
2.1.0 -> 2.2.1, README "Performance": circular cone beam, per-view trajectories;
diffct 2.4.3 -> 2.4.4, CHANGELOG "Added": per-axis spacing in tensor order).
"""

from .workloads import Workload, WORKLOADS, get, scaled, small_cases
from .frames import frames
from .phantom import phantom, sinogram_noise

__all__ = ["Workload", "WORKLOADS", "get", "scaled", "small_cases", "frames",
           "phantom", "sinogram_noise"]
