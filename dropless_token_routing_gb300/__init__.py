"""Dropless MoE layer hot path for GB300 (sm_103a): route -> permute -> grouped SwiGLU
GEMM -> combine, forward and backward, behind the C ABI of include/moe.h.

``import dropless_token_routing_gb300`` only exposes the build step; the torch-facing
wrappers live in ``dropless_token_routing_gb300.api`` and load the compiled library
(raising ImportError if it has not been built).
"""
from .builder import build, LIB  # noqa: F401
