"""Seeded synthetic inputs for the MoE layer (generator + workload shapes).

Shared by the tests, the bench and the oracle's checks.  Holds none of the
layer's arithmetic."""
from . import gen, workloads  # noqa: F401
from .workloads import WORKLOADS, Workload, make_inputs  # noqa: F401
