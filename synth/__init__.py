"""Seeded synthetic inputs for StateKV streaming prefill.

This package holds the workload shapes and the seeded generator of per-frame
Q/K/V.  It contains none of the method's arithmetic (no RoPE, attention,
scoring or selection): both the CUDA library's tests/bench and the CPU oracle
draw their inputs from here, so that the two sides see identical bits.
"""

from .shapes import SHAPES, WorkloadShape, serving_shape
from .frames import FrameSource

__all__ = ["SHAPES", "WorkloadShape", "serving_shape", "FrameSource"]
