"""Seeded synthetic inputs for the dropless MoE layer.

This package only draws random numbers and lays them out in the shapes of the
workloads; it holds none of the layer's arithmetic (no routing, no softmax, no
permutation, no expert FFN).  Both the CUDA path (through its tests and the
benchmark) and the CPU oracle take their inputs from here.
"""
from .workloads import CONFIGS, Workload, make_workload, shrink  # noqa: F401
