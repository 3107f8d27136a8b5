"""GB300-native tile-centric AllGather->GEMM and GEMM->ReduceScatter overlap.

The hot path is a C-ABI library of hand-written sm_103a kernels
(``csrc/``, declared in ``include/opw.h``); ``api`` is a thin ctypes binding
that only marshals arguments.  Importing this package does not load the
library; the first call into ``api`` does, and fails loudly if it is missing.
"""
__all__ = ["api", "inputs"]
