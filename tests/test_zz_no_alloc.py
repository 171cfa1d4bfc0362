"""bi_attention_noalloc: the split-key-range attention with the library's
static device scratch instead of a caller workspace.  Collected last (file
name) so that the scratch is exercised after every other test has run on the
same device.  Its results must be those of bi_attention_ws bit for bit, and a
problem whose workspace exceeds the static scratch must be refused before any
launch."""
from __future__ import annotations

import ctypes

import pytest
import torch

from invariant_gemm_bi_gb300 import binding, inputs
from tests.gpu_helpers import bits_equal

SCRATCH = 64 << 20
D = 256


def _t(shape, dtype=0, ptr=0x7F0000000000):
    d = binding.BiTensor()
    d.ptr, d.ndim, d.dtype = ptr, len(shape), dtype
    s = 1
    for i in reversed(range(len(shape))):
        d.shape[i], d.stride[i] = shape[i], s
        s *= shape[i]
    return d


def test_noalloc_refuses_a_workspace_larger_than_the_scratch():
    lib = binding.load()
    L, Tq, Tk = 8, 8192, 8192
    assert lib.bi_attention_workspace_bytes(L, Tq, Tk, 256) > SCRATCH
    q, k, v, o = _t([L, Tq, D]), _t([L, Tk, D]), _t([L, Tk, D]), _t([L, Tq, D], dtype=2)
    st = lib.bi_attention_noalloc(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.c_float(0.0625),
                                  ctypes.byref(o), None)
    assert st == binding.BI_ERR_INVALID_ARG
    assert "scratch" in binding.last_error_message()


@pytest.mark.gpu
def test_noalloc_equals_caller_workspace_bit_for_bit():
    binding.load()
    L, Tq, Tk = 4, 300, 5000
    assert 0 < binding.bi_attention_workspace_bytes(L, Tq, Tk) <= SCRATCH
    q = inputs.normal_bf16((L, Tq, D), 1.0, 70).cuda()
    k = inputs.normal_bf16((L, Tk, D), 1.0, 71).cuda()
    v = inputs.normal_bf16((L, Tk, D), 1.0, 72).cuda()
    ref = binding.bi_attention_ws(q, k, v, 1.0 / 16)
    for _ in range(3):
        assert bits_equal(binding.bi_attention_noalloc(q, k, v, 1.0 / 16), ref)
    # bf16 output, and a key range short enough to need no scratch at all
    assert bits_equal(binding.bi_attention_noalloc(q, k, v, 1.0 / 16, out_dtype=torch.bfloat16),
                      binding.bi_attention_ws(q, k, v, 1.0 / 16, out_dtype=torch.bfloat16))
    assert bits_equal(binding.bi_attention_noalloc(q, k[:, :2000], v[:, :2000], 1.0 / 16),
                      binding.bi_attention(q, k[:, :2000], v[:, :2000], 1.0 / 16))
    # the largest problem of this shape family that fits still runs
    Tq2 = SCRATCH // (3 * L * (D + 2) * 4)
    q2 = inputs.normal_bf16((L, Tq2, D), 1.0, 73).cuda()
    k2 = inputs.normal_bf16((L, 6000, D), 1.0, 74).cuda()
    v2 = inputs.normal_bf16((L, 6000, D), 1.0, 75).cuda()
    assert binding.bi_attention_workspace_bytes(L, Tq2, 6000) <= SCRATCH
    assert bits_equal(binding.bi_attention_noalloc(q2, k2, v2, 0.0625), binding.bi_attention_ws(q2, k2, v2, 0.0625))
    assert binding.bi_device_status() == binding.BI_OK


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_narrow_heads_equal_caller_workspace(d):
    # the scratch holds ceil(Tk / 2048) * L * Tq * (d + 2) floats for a narrower head
    binding.load()
    L, Tq, Tk = 3, 260, 4500
    need = binding.bi_attention_workspace_bytes(L, Tq, Tk, d)
    assert need == 3 * L * Tq * (d + 2) * 4 and need <= SCRATCH
    q = inputs.normal_bf16((L, Tq, d), 1.0, 76).cuda()
    k = inputs.normal_bf16((L, Tk, d), 1.0, 77).cuda()
    v = inputs.normal_bf16((L, Tk, d), 1.0, 78).cuda()
    for od in (torch.float32, torch.bfloat16):
        assert bits_equal(binding.bi_attention_noalloc(q, k, v, d ** -0.5, out_dtype=od),
                          binding.bi_attention_ws(q, k, v, d ** -0.5, out_dtype=od))
    assert binding.bi_device_status() == binding.BI_OK
