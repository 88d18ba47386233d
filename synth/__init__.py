"""Seeded synthetic inputs for query-aware sparse-page decode attention.

This package only draws random tensors with the shapes, dtypes and value
distributions of the five decode workloads (page tables, sequence lengths,
queries, paged K/V pools, int8 scales, the fixed Gaussian sketch projection
and planted needle keys).  It holds none of the method's arithmetic: no
page scores, no selection, no attention.  Both the fp64 oracle tests and the
CUDA path consume what it produces.
"""

from .workloads import WORKLOADS, Workload, get_workload, scaled
from .gen import DecodeInputs, make_inputs

__all__ = ["WORKLOADS", "Workload", "get_workload", "scaled", "DecodeInputs", "make_inputs"]
