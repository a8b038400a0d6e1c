"""Routed Mixture-of-Experts expert-MLP layer (forward and backward) for one
NVIDIA GB300 (sm_103a): a C-ABI CUDA library (libmoe_gb300.so, include/moe_gb300.h)
with a thin ctypes binding.  Importing the package loads nothing; the library is
loaded on first use and its absence is an error (there is no fallback).
"""

__all__ = ["binding", "layer", "synth", "build"]
