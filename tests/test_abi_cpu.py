"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
it exports every entry point include/bi.h declares, and argument / shape /
dtype / layout errors come back as status codes before anything is launched
(the descriptors below point at fake addresses that are never touched)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from invariant_gemm_bi_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "bi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_documented_entry_points():
    names = _header_functions()
    for n in ("bi_mm", "bi_addmm", "bi_bmm", "bi_conv2d_patch", "bi_softmax_lastdim",
              "bi_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name
    assert set(_header_functions()) == set(binding.EXPORTED)


def test_library_has_no_oracle_or_host_math_dependency():
    # The product library must not link the oracle (it is test infrastructure).
    data = open(build.LIB_PATH, "rb").read()
    assert b"bio_mm" not in data and b"libbi_oracle" not in data


def test_status_strings(lib):
    assert binding.status_string(0) == "BI_OK"
    assert binding.status_string(6) == "BI_ERR_TIMEOUT"
    assert lib.bi_abi_version() == 8


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def _t(shape, stride=None, dtype=0, ptr=FAKE):
    d = binding.BiTensor()
    d.ptr = ptr
    d.ndim = len(shape)
    d.dtype = dtype
    if stride is None:
        stride, s = [], 1
        for n in reversed(shape):
            stride.insert(0, s)
            s *= n
    for i, (n, st) in enumerate(zip(shape, stride)):
        d.shape[i] = n
        d.stride[i] = st
    return d


def _r(d):
    return ctypes.byref(d) if d is not None else None


def _mm(lib, a, b, c):
    return lib.bi_mm(_r(a), _r(b), _r(c), None)


def test_mm_validation_errors(lib):
    ok_a, ok_b, ok_c = _t([4, 64]), _t([64, 32]), _t([4, 32], dtype=2)
    # inner dimension mismatch
    assert _mm(lib, ok_a, _t([48, 32]), ok_c) == binding.BI_ERR_SHAPE_MISMATCH
    # output extent mismatch
    assert _mm(lib, ok_a, ok_b, _t([4, 33], dtype=2)) == binding.BI_ERR_SHAPE_MISMATCH
    # fp32 inputs are not taken, and bf16 / fp16 operands are never mixed (the
    # tensor core's f16 kind takes one format for both)
    assert _mm(lib, _t([4, 64], dtype=2), ok_b, ok_c) == binding.BI_ERR_UNSUPPORTED_DTYPE
    assert _mm(lib, _t([4, 64], dtype=1), ok_b, ok_c) == binding.BI_ERR_UNSUPPORTED_DTYPE
    assert _mm(lib, ok_a, _t([64, 32], dtype=1), ok_c) == binding.BI_ERR_UNSUPPORTED_DTYPE
    assert lib.bi_bmm(_r(_t([2, 4, 64], dtype=1)), _r(_t([2, 64, 32])), _r(_t([2, 4, 32], dtype=2)), 1.0,
                      None) == binding.BI_ERR_UNSUPPORTED_DTYPE
    # wrong rank
    assert _mm(lib, _t([4, 64, 1]), ok_b, ok_c) == binding.BI_ERR_INVALID_ARG
    # null descriptor
    assert lib.bi_mm(None, _r(ok_b), _r(ok_c), None) == binding.BI_ERR_INVALID_ARG
    # A without a unit stride on K (column-major activations)
    assert _mm(lib, _t([4, 64], [1, 4]), ok_b, ok_c) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # A row stride not a multiple of 8 elements (16 bytes)
    assert _mm(lib, _t([4, 60], [60, 1]), _t([60, 32]), ok_c) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # misaligned base
    assert _mm(lib, _t([4, 64], ptr=FAKE + 2), ok_b, ok_c) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # B with neither unit stride
    assert _mm(lib, ok_a, _t([64, 32], [64, 2]), ok_c) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # output without unit stride on N
    assert _mm(lib, ok_a, ok_b, _t([4, 32], [1, 4], dtype=2)) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # negative stride
    assert _mm(lib, ok_a, _t([64, 32], [-32, 1]), ok_c) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    assert "stride" in binding.last_error_message()


def test_empty_problems_are_no_ops_without_touching_the_device(lib):
    # M == 0 / N == 0: nothing to compute, OK before any CUDA call
    assert _mm(lib, _t([0, 64]), _t([64, 32]), _t([0, 32], dtype=2)) == binding.BI_OK
    assert _mm(lib, _t([4, 64]), _t([64, 0]), _t([4, 0], dtype=2)) == binding.BI_OK
    assert lib.bi_softmax_lastdim(_r(_t([0, 8], dtype=2)), _r(_t([0, 8])), None) == binding.BI_OK


def test_valid_call_without_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = _mm(lib, _t([4, 64]), _t([64, 32]), _t([4, 32], dtype=2))
    assert st == binding.BI_ERR_NO_DEVICE
    # fp16 operands (both) with fp16 output pass validation the same way
    st = _mm(lib, _t([4, 64], dtype=1), _t([64, 32], dtype=1), _t([4, 32], dtype=1))
    assert st == binding.BI_ERR_NO_DEVICE


def test_addmm_bmm_softmax_conv_validation(lib):
    a, b, c = _t([4, 64]), _t([64, 32]), _t([4, 32])
    assert lib.bi_addmm(None, _r(a), _r(b), _r(c), None) == binding.BI_ERR_INVALID_ARG
    assert lib.bi_addmm(_r(_t([31])), _r(a), _r(b), _r(c), None) == binding.BI_ERR_SHAPE_MISMATCH
    # bmm batch mismatch
    assert lib.bi_bmm(_r(_t([2, 4, 64])), _r(_t([3, 64, 32])), _r(_t([2, 4, 32], dtype=2)), 1.0,
                      None) == binding.BI_ERR_SHAPE_MISMATCH
    # softmax needs fp32 scores
    assert lib.bi_softmax_lastdim(_r(_t([4, 8])), _r(_t([4, 8])), None) == binding.BI_ERR_UNSUPPORTED_DTYPE
    # conv: output shape must follow the size formula
    arr = ctypes.c_int32 * 2
    x, w = _t([2, 3, 224, 224]), _t([1152, 3, 14, 14])
    bad_y = _t([2, 1152, 15, 16])
    st = lib.bi_conv2d_patch(_r(x), _r(w), None, _r(bad_y), arr(14, 14), arr(0, 0), arr(1, 1), 1, None)
    assert st == binding.BI_ERR_SHAPE_MISMATCH
    # groups must divide the channels
    st = lib.bi_conv2d_patch(_r(x), _r(w), None, _r(_t([2, 1152, 16, 16])), arr(14, 14), arr(0, 0),
                             arr(1, 1), 2, None)
    assert st == binding.BI_ERR_SHAPE_MISMATCH
    # non-contiguous input
    xs = _t([2, 3, 224, 224], [3 * 224 * 224, 224 * 224, 1, 224])
    st = lib.bi_conv2d_patch(_r(xs), _r(w), None, _r(_t([2, 1152, 16, 16])), arr(14, 14), arr(0, 0),
                             arr(1, 1), 1, None)
    assert st == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # debug wait: limit out of range is refused before launching
    assert lib.bi_debug_expire_wait(10, None) == binding.BI_ERR_INVALID_ARG


def test_packed_weight_size_and_validation(lib):
    # [k blocks of 64] x [tiles of 256 columns] x 32 KB
    assert lib.bi_packed_weight_bytes(4096, 14336) == 64 * 56 * 32768
    assert lib.bi_packed_weight_bytes(65, 257) == 2 * 2 * 32768
    assert lib.bi_packed_weight_bytes(0, 8) == 0
    desc = binding.BiPackedWeightDesc()
    # destination too small
    st = lib.bi_pack_weight(_r(_t([64, 256])), FAKE, 1024, ctypes.byref(desc), None)
    assert st == binding.BI_ERR_INVALID_ARG
    # fp32 weight refused
    st = lib.bi_pack_weight(_r(_t([64, 256], dtype=2)), FAKE, 1 << 20, ctypes.byref(desc), None)
    assert st == binding.BI_ERR_UNSUPPORTED_DTYPE
    # packed descriptor with an element type other than bf16 / fp16
    pd = binding.BiPackedWeightDesc(FAKE, 1 << 20, 64, 256, 1, 256, 2)
    st = lib.bi_addmm_packed(None, _r(_t([4, 64])), ctypes.byref(pd), _r(_t([4, 256], dtype=2)), None)
    assert st == binding.BI_ERR_INVALID_ARG
    # an fp16 packed weight does not take bf16 activations
    pd = binding.BiPackedWeightDesc(FAKE, 1 << 20, 64, 256, 1, 256, 1)
    st = lib.bi_addmm_packed(None, _r(_t([4, 64])), ctypes.byref(pd), _r(_t([4, 256], dtype=2)), None)
    assert st == binding.BI_ERR_UNSUPPORTED_DTYPE
    # packed descriptor with a foreign tile width
    pd = binding.BiPackedWeightDesc(FAKE, 1 << 20, 64, 256, 1, 128)
    st = lib.bi_addmm_packed(None, _r(_t([4, 64])), ctypes.byref(pd), _r(_t([4, 256], dtype=2)), None)
    assert st == binding.BI_ERR_INVALID_ARG
    # K of the activations must match the packed weight
    pd = binding.BiPackedWeightDesc(FAKE, 1 << 20, 64, 256, 1, 256)
    st = lib.bi_addmm_packed(None, _r(_t([4, 128])), ctypes.byref(pd), _r(_t([4, 256], dtype=2)), None)
    assert st == binding.BI_ERR_SHAPE_MISMATCH


def test_conv_packed_weight_size_and_validation(lib):
    # [Co][C * (KH rounded up to 4) * 16] bf16
    assert lib.bi_conv_packed_weight_bytes(1152, 3, 14, 14) == 1152 * 3 * 16 * 16 * 2
    assert lib.bi_conv_packed_weight_bytes(8, 2, 5, 3) == 8 * 2 * 8 * 16 * 2
    assert lib.bi_conv_packed_weight_bytes(8, 2, 5, 17) == 0
    assert lib.bi_conv_packed_weight_bytes(0, 2, 5, 3) == 0
    desc = binding.BiConvPackedWeightDesc()
    big = 1 << 24
    # fp32 filter refused; KW > 16 refused; too-small destination refused
    assert lib.bi_conv_pack_weight(_r(_t([8, 3, 4, 4], dtype=2)), FAKE, big, ctypes.byref(desc),
                                   None) == binding.BI_ERR_UNSUPPORTED_DTYPE
    assert lib.bi_conv_pack_weight(_r(_t([8, 3, 4, 17])), FAKE, big, ctypes.byref(desc),
                                   None) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    assert lib.bi_conv_pack_weight(_r(_t([8, 3, 4, 4])), FAKE, 64, ctypes.byref(desc),
                                   None) == binding.BI_ERR_INVALID_ARG
    # the convolution itself: a consistent descriptor of a [1152, 3, 14, 14] filter
    pw = binding.BiConvPackedWeightDesc(FAKE, big, 1152, 3, 14, 14, 3 * 16 * 16)
    x = _t([2, 3, 224, 224])
    y = _t([2, 1152, 16, 16])

    def conv(x_, pw_, y_):
        return lib.bi_conv2d_patch_packed(_r(x_), ctypes.byref(pw_), None, _r(y_), None)

    # channel count differs from the filter's
    assert conv(_t([2, 4, 224, 224]), pw, y) == binding.BI_ERR_SHAPE_MISMATCH
    # output extent not [B, Co, H/KH, W/KW]
    assert conv(x, pw, _t([2, 1152, 16, 15])) == binding.BI_ERR_SHAPE_MISMATCH
    # image rows not a multiple of 8 elements (TMA reads whole 16-byte rows)
    assert conv(_t([2, 3, 224, 230]), pw, y) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # image wider than one staged row
    assert conv(_t([1, 3, 14, 264]), pw, _t([1, 1152, 1, 18])) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # misaligned image base
    assert conv(_t([2, 3, 224, 224], ptr=FAKE + 2), pw, y) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # descriptor whose row length does not match its shape
    bad = binding.BiConvPackedWeightDesc(FAKE, big, 1152, 3, 14, 14, 588)
    assert conv(x, bad, y) == binding.BI_ERR_INVALID_ARG
    # bf16 / fp32 only for y
    assert conv(x, pw, _t([2, 1152, 16, 16], dtype=1)) == binding.BI_ERR_UNSUPPORTED_DTYPE
    # nothing to compute: OK before any CUDA call
    assert conv(_t([0, 3, 224, 224]), pw, _t([0, 1152, 16, 16])) == binding.BI_OK


def test_row_reduction_validation(lib):
    import ctypes as ct
    x, y = _t([4, 100]), _t([4, 100])
    eps = ct.c_float(1e-6)
    # shapes
    assert lib.bi_rmsnorm_lastdim(_r(x), None, eps, _r(_t([4, 99])), None) == binding.BI_ERR_SHAPE_MISMATCH
    assert lib.bi_rmsnorm_lastdim(_r(x), _r(_t([99])), eps, _r(y), None) == binding.BI_ERR_SHAPE_MISMATCH
    assert lib.bi_log_softmax_lastdim(_r(x), _r(_t([3, 100])), None) == binding.BI_ERR_SHAPE_MISMATCH
    assert lib.bi_mean_lastdim(_r(x), _r(_t([5])), None) == binding.BI_ERR_SHAPE_MISMATCH
    assert lib.bi_mean_lastdim(_r(x), _r(_t([4, 1])), None) == binding.BI_ERR_INVALID_ARG  # rank
    # layouts: no unit stride on the reduced dimension, misaligned element
    assert lib.bi_log_softmax_lastdim(_r(_t([4, 100], [1, 4])), _r(y), None) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    assert lib.bi_rmsnorm_lastdim(_r(x), None, eps, _r(_t([4, 100], [1, 4])), None) == \
        binding.BI_ERR_UNSUPPORTED_LAYOUT
    assert lib.bi_mean_lastdim(_r(_t([4, 100], dtype=2, ptr=FAKE + 2)), _r(_t([4])), None) == \
        binding.BI_ERR_UNSUPPORTED_LAYOUT
    # eps must be finite and >= 0
    for bad in (-1.0, float("nan"), float("inf")):
        assert lib.bi_rmsnorm_lastdim(_r(x), None, ct.c_float(bad), _r(y), None) == binding.BI_ERR_INVALID_ARG
    # rows longer than 2^24 are refused; an empty row has no mean
    assert lib.bi_mean_lastdim(_r(_t([1, (1 << 24) + 1])), _r(_t([1])), None) == binding.BI_ERR_INVALID_ARG
    assert lib.bi_mean_lastdim(_r(_t([3, 0])), _r(_t([3])), None) == binding.BI_ERR_INVALID_ARG
    # empty problems are no-ops before any CUDA call
    assert lib.bi_rmsnorm_lastdim(_r(_t([0, 8])), None, eps, _r(_t([0, 8])), None) == binding.BI_OK
    assert lib.bi_log_softmax_lastdim(_r(_t([5, 0])), _r(_t([5, 0])), None) == binding.BI_OK
    assert lib.bi_mean_lastdim(_r(_t([0, 8])), _r(_t([0])), None) == binding.BI_OK
    # a valid call of every input / output type combination gets as far as the device
    import torch
    if not torch.cuda.is_available():
        for dx in (0, 1, 2):
            for dy in (0, 1, 2):
                assert lib.bi_rmsnorm_lastdim(_r(_t([4, 100], dtype=dx)), _r(_t([100], dtype=dy)), eps,
                                              _r(_t([4, 100], dtype=dy)), None) == binding.BI_ERR_NO_DEVICE
                assert lib.bi_log_softmax_lastdim(_r(_t([4, 100], dtype=dx)), _r(_t([4, 100], dtype=dy)),
                                                  None) == binding.BI_ERR_NO_DEVICE
                assert lib.bi_mean_lastdim(_r(_t([4, 100], dtype=dx)), _r(_t([4], dtype=dy)),
                                           None) == binding.BI_ERR_NO_DEVICE


def test_attention_validation(lib):
    def call(q, k, v, o, scale=0.0625):
        return lib.bi_attention(_r(q), _r(k), _r(v), ctypes.c_float(scale), _r(o), None)
    q, k, v, o = _t([2, 100, 256]), _t([2, 90, 256]), _t([2, 90, 256]), _t([2, 100, 256], dtype=2)
    # shapes
    assert call(q, _t([2, 91, 256]), v, o) == binding.BI_ERR_SHAPE_MISMATCH
    assert call(q, k, v, _t([2, 99, 256], dtype=2)) == binding.BI_ERR_SHAPE_MISMATCH
    assert call(q, _t([3, 90, 256]), _t([3, 90, 256]), o) == binding.BI_ERR_SHAPE_MISMATCH
    # head dimension 64, 128 or 256 only; dtypes
    for d in (32, 96, 192, 512):
        assert call(_t([2, 100, d]), _t([2, 90, d]), _t([2, 90, d]), _t([2, 100, d], dtype=2)) == \
            binding.BI_ERR_INVALID_ARG
        assert "head dimension" in binding.last_error_message()
    assert call(_t([2, 100, 256], dtype=1), k, v, o) == binding.BI_ERR_UNSUPPORTED_DTYPE
    assert call(q, k, v, _t([2, 100, 256], dtype=1)) == binding.BI_ERR_UNSUPPORTED_DTYPE
    # layouts: non-unit head stride, a row stride that is not 16 bytes, a misaligned base
    assert call(_t([2, 100, 256], [256 * 100, 1, 100]), k, v, o) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    assert call(_t([2, 100, 256], [100 * 260, 260, 1]), k, v, o) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    assert call(q, _t([2, 90, 256], ptr=FAKE + 8), v, o) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    # scale must be finite; an empty key range has no softmax
    assert call(q, k, v, o, float("inf")) == binding.BI_ERR_INVALID_ARG
    assert call(q, _t([2, 0, 256]), _t([2, 0, 256]), o) == binding.BI_ERR_INVALID_ARG
    # no query rows or no heads: nothing to do, before any CUDA call
    assert call(_t([2, 0, 256]), k, v, _t([2, 0, 256], dtype=2)) == binding.BI_OK
    assert call(_t([0, 100, 256]), _t([0, 90, 256]), _t([0, 90, 256]), _t([0, 100, 256], dtype=2)) == binding.BI_OK
    # a valid call reaches the device check
    import torch
    if not torch.cuda.is_available():
        assert call(q, k, v, o) == binding.BI_ERR_NO_DEVICE
        assert call(q, k, v, _t([2, 100, 256], dtype=0)) == binding.BI_ERR_NO_DEVICE


def test_attention_workspace_rules(lib):
    # no workspace up to 2048 keys; ceil(Tk / 2048) splits of L*Tq*(D+2) floats beyond
    for d in (64, 128, 256):
        assert lib.bi_attention_workspace_bytes(2, 100, 2048, d) == 0
        assert lib.bi_attention_workspace_bytes(2, 100, 2049, d) == 2 * 2 * 100 * (d + 2) * 4
        assert lib.bi_attention_workspace_bytes(3, 7, 6145, d) == 4 * 3 * 7 * (d + 2) * 4
        assert lib.bi_attention_workspace_bytes(0, 7, 6145, d) == 0
    assert lib.bi_attention_workspace_bytes(2, 100, 6145, 96) == 0  # no such kernel
    q, k, v, o = _t([2, 100, 256]), _t([2, 3000, 256]), _t([2, 3000, 256]), _t([2, 100, 256], dtype=2)
    f = ctypes.c_float(0.0625)
    need = lib.bi_attention_workspace_bytes(2, 100, 3000, 256)
    # a long key range without (enough) workspace is refused before any launch
    assert lib.bi_attention(_r(q), _r(k), _r(v), f, _r(o), None) == binding.BI_ERR_INVALID_ARG
    assert "workspace" in binding.last_error_message()
    assert lib.bi_attention_ws(_r(q), _r(k), _r(v), f, _r(o), ctypes.c_void_p(FAKE), ctypes.c_int64(need - 1),
                               None) == binding.BI_ERR_INVALID_ARG
    assert lib.bi_attention_ws(_r(q), _r(k), _r(v), f, _r(o), ctypes.c_void_p(FAKE + 8), ctypes.c_int64(need),
                               None) == binding.BI_ERR_UNSUPPORTED_LAYOUT
    assert lib.bi_attention_ws(_r(q), _r(k), _r(v), f, _r(o), ctypes.c_void_p(FAKE), ctypes.c_int64(-1),
                               None) == binding.BI_ERR_INVALID_ARG
    import torch
    if not torch.cuda.is_available():
        assert lib.bi_attention_ws(_r(q), _r(k), _r(v), f, _r(o), ctypes.c_void_p(FAKE), ctypes.c_int64(need),
                                   None) == binding.BI_ERR_NO_DEVICE
