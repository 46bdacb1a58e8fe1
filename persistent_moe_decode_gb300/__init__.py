"""GB300-native persistent MoE decode step.

One persistent CUDA kernel (one thread block per SM) runs a whole decode step
of a BF16 parallel-layer MoE transformer from host-built per-SM task lists,
with global-memory counters for dependencies and shared claim queues for the
attention and expert tiles.  The step sits behind the C-ABI library in
``include/mk.h``; :mod:`persistent_moe_decode_gb300.mk` is its thin binding.

Importing the package loads nothing native; ``mk`` loads the library on first
use and raises if it is missing.
"""
from .configs import ModelDims, Workload, WORKLOADS  # noqa: F401

__all__ = ["ModelDims", "Workload", "WORKLOADS"]
