"""MoE grouped GEMM for GB300 (sm_103a): contiguous, masked and K-grouped forms.

The compute path is the C-ABI library ``libmoegemm.so`` built from ``csrc/``
(hand-written CUDA for sm_103a).  ``binding`` is a thin ctypes layer over it;
nothing in this package computes the method on the CPU, and every call raises
if the library is missing.  ``workloads`` draws seeded synthetic inputs.
"""

__all__ = ["binding", "workloads", "build"]
