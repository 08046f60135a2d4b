"""Tensor-core GEMM D = A·B + C for one GB300 (sm_103a).

The compute runs in the CUDA library ``libgb300gemm.so`` (built from
``csrc/``) behind the C ABI declared in ``include/gb300gemm.h``; ``gemm``
is a thin ctypes binding with the same entry-point names.  ``synth`` makes
the seeded synthetic inputs.
"""
