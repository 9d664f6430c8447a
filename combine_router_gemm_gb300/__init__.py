"""GB300-native single-GPU Mixture-of-Experts layer hot path.

Router scoring and top-k selection, dispatch (histogram, scan, permute), the
per-expert SwiGLU FFN as grouped GEMMs, and the gate-weighted combine, each a
CUDA kernel for sm_103a behind the C ABI declared in ``include/moe.h``.  The
Python side (``binding``) only marshals pointers, sizes and streams.
"""
__all__ = ["inputs", "binding"]
