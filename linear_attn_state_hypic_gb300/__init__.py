"""GB300 (sm_103a) library for the linear-attention state path of HYPIC.

The product is the C-ABI shared library ``libhypic.so`` (declared in
``include/hypic.h``); this package holds its CUDA sources (``csrc/``), the
build step (``build_lib``), a thin ctypes binding with the same call names
(``binding``) and the seeded input generators (``synth``).  Nothing here
computes on the CPU: every step of the path runs in the library's kernels,
and the binding raises if the library has not been built.
"""
__all__ = ["binding", "synth", "build_lib"]
