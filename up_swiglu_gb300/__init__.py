"""Fused 4-bit MoE expert gate/up projection with SwiGLU for GB300 (sm_103a).

``up_swiglu_gb300.q4moe`` is the Python binding of the C ABI in
``include/q4moe.h`` (libq4moe.so, built in-tree by ``up_swiglu_gb300.build``);
``up_swiglu_gb300.synthetic`` draws the seeded synthetic workloads.  Nothing
is loaded at import time.
"""
__all__ = ["q4moe", "synthetic", "build"]
