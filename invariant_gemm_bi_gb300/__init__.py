"""Batch-invariant bf16 contractions for GB300 (sm_103a).

The operations run in hand-written CUDA kernels behind the C ABI declared in
``include/bi.h``; ``binding`` only marshals torch tensors into that ABI, with
the same names as the C entry points:

    bi_mm, bi_addmm, bi_bmm, bi_conv2d_patch, bi_softmax_lastdim,
    bi_pack_weight, bi_addmm_packed, bi_device_status

The shared library is loaded on first use; a call raises if it is missing --
there is no CPU or library fallback.
"""
from . import inputs  # noqa: F401  (seeded input generators; no arithmetic)
from .binding import (BiError, PackedWeight, bi_addmm, bi_addmm_packed, bi_bmm,  # noqa: F401
                      bi_conv2d_patch, bi_device_status, bi_mm, bi_pack_weight,
                      bi_softmax_lastdim)
