"""GB300 routed Mixture-of-Experts layer: sigmoid+bias top-k routing, a stable
expert permutation, int8 block-quantised SwiGLU experts (Q8_0 or 2-bit) with a
shared expert, and an ordered combine -- all in the CUDA library ``libmoe.so``.

``routed_expert_decode_gb300.moe`` is the Python binding of its C ABI
(``include/moe.h``).
"""
from . import moe  # noqa: F401

__all__ = ["moe"]
