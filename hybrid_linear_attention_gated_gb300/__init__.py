"""GB300 (sm_103a) kernels for the hybrid linear-attention (KDA) + routed-MoE decode step.

The compute lives in a C-ABI shared library of hand-written CUDA kernels
(``csrc/``, declared in ``include/hla.h``); ``hla`` is a thin ctypes binding
with the same entry-point names.  ``inputs`` draws seeded synthetic workloads.
"""

__all__ = ["hla", "inputs"]
