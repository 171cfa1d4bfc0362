"""Batch-invariant bf16 contractions for GB300 (sm_103a).

The operations (``mm``, ``addmm``, ``bmm``, ``conv2d_patch``,
``softmax_lastdim``) run in hand-written CUDA kernels behind the C ABI
declared in ``include/bi.h``; this package only marshals torch tensors into
that ABI.  The shared library is loaded on first use and an operation raises
if it is missing -- there is no CPU or library fallback.
"""
from . import inputs  # noqa: F401  (seeded input generators; no arithmetic)
