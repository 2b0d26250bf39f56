"""grouped_gemm_moe_gb300: one MoE layer's single-GPU hot path on GB300 (sm_103a).

The compute lives in libmoe_gb300.so (C ABI, include/moe_gb300.h), built in
tree by ``grouped_gemm_moe_gb300.build.build()``. ``binding`` exposes each C
entry point under its own name for torch tensors; ``layer.MoELayer`` runs a
whole layer's forward and backward as a sequence of those calls;
``workloads`` draws the seeded synthetic inputs.

Importing the package does not load the library; the first binding call
does, and raises if it has not been built.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "binding", "layer", "build"]
