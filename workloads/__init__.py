"""Seeded synthetic inputs for the MoE permute + grouped-matmul backward.

This package builds inputs only: routing (expert choice per token, the
expanded order, expandedRowIdx, groupList) and value tensors. It holds none
of the method's arithmetic, and both the oracle-based tests and the CUDA
path consume what it produces.
"""

from .moe import (  # noqa: F401
    WORKLOADS,
    Inputs,
    Workload,
    make_inputs,
    make_case,
    forward_input,
    route_experts,
    expanded_order,
)
