"""ctypes binding of the C ABI in ``include/bi.h`` (argument marshalling only).

Each function takes CUDA torch tensors, describes them as ``bi_tensor``
structs (pointer, shape, element strides, dtype code), allocates the output
with torch when ``out`` is not given, and calls the entry point of the same
name on the current torch stream.  All arithmetic happens in the library's
CUDA kernels; a missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

BI_OK = 0
BI_ERR_INVALID_ARG = 1
BI_ERR_SHAPE_MISMATCH = 2
BI_ERR_UNSUPPORTED_DTYPE = 3
BI_ERR_UNSUPPORTED_LAYOUT = 4
BI_ERR_CUDA = 5
BI_ERR_TIMEOUT = 6
BI_ERR_NO_DEVICE = 7

EXPORTED = ("bi_mm", "bi_addmm", "bi_bmm", "bi_conv2d_patch", "bi_softmax_lastdim",
            "bi_rmsnorm_lastdim", "bi_log_softmax_lastdim", "bi_mean_lastdim", "bi_attention",
            "bi_attention_workspace_bytes", "bi_attention_ws", "bi_attention_noalloc",
            "bi_packed_weight_bytes", "bi_pack_weight", "bi_addmm_packed",
            "bi_conv_packed_weight_bytes", "bi_conv_pack_weight", "bi_conv2d_patch_packed",
            "bi_device_status", "bi_debug_expire_wait", "bi_status_string",
            "bi_last_error_message", "bi_abi_version")

_DTYPES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}


class BiTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("ndim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class BiPackedWeightDesc(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("bytes", ctypes.c_int64), ("K", ctypes.c_int64),
                ("N", ctypes.c_int64), ("layout", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class BiConvPackedWeightDesc(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("bytes", ctypes.c_int64), ("Co", ctypes.c_int64),
                ("C", ctypes.c_int64), ("KH", ctypes.c_int64), ("KW", ctypes.c_int64),
                ("Kp", ctypes.c_int64)]


class ConvPackedWeight:
    """A patch-embedding filter packed on the device by ``bi_conv_pack_weight``:
    owns the torch buffer that holds it and the descriptor the library reads."""

    def __init__(self, buffer: torch.Tensor, desc: BiConvPackedWeightDesc):
        self.buffer = buffer
        self.desc = desc

    @property
    def shape(self):
        return (int(self.desc.Co), int(self.desc.C), int(self.desc.KH), int(self.desc.KW))


class PackedWeight:
    """A weight packed on the device by ``bi_pack_weight``: owns the torch
    buffer that holds it and the descriptor the library reads."""

    def __init__(self, buffer: torch.Tensor, desc: BiPackedWeightDesc):
        self.buffer = buffer
        self.desc = desc

    @property
    def shape(self):
        return (int(self.desc.K), int(self.desc.N))


class BiError(RuntimeError):
    def __init__(self, op: str, status: int, name: str, detail: str):
        super().__init__(f"{op}: {name}: {detail}")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Loads the shared library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"CUDA library {p} is missing: run invariant_gemm_bi_gb300.build.build()")
            lib = ctypes.CDLL(p)
            ptr = ctypes.POINTER(BiTensor)
            i32x2 = ctypes.POINTER(ctypes.c_int32)
            st = ctypes.c_int
            sig = {
                "bi_mm": ([ptr, ptr, ptr, ctypes.c_void_p], st),
                "bi_addmm": ([ptr, ptr, ptr, ptr, ctypes.c_void_p], st),
                "bi_bmm": ([ptr, ptr, ptr, ctypes.c_float, ctypes.c_void_p], st),
                "bi_conv2d_patch": ([ptr, ptr, ptr, ptr, i32x2, i32x2, i32x2, ctypes.c_int32,
                                     ctypes.c_void_p], st),
                "bi_softmax_lastdim": ([ptr, ptr, ctypes.c_void_p], st),
                "bi_rmsnorm_lastdim": ([ptr, ptr, ctypes.c_float, ptr, ctypes.c_void_p], st),
                "bi_log_softmax_lastdim": ([ptr, ptr, ctypes.c_void_p], st),
                "bi_mean_lastdim": ([ptr, ptr, ctypes.c_void_p], st),
                "bi_attention": ([ptr, ptr, ptr, ctypes.c_float, ptr, ctypes.c_void_p], st),
                "bi_attention_workspace_bytes": ([ctypes.c_int64] * 4, ctypes.c_int64),
                "bi_attention_noalloc": ([ptr, ptr, ptr, ctypes.c_float, ptr, ctypes.c_void_p], st),
                "bi_attention_ws": ([ptr, ptr, ptr, ctypes.c_float, ptr, ctypes.c_void_p, ctypes.c_int64,
                                     ctypes.c_void_p], st),
                "bi_packed_weight_bytes": ([ctypes.c_int64, ctypes.c_int64], ctypes.c_int64),
                "bi_pack_weight": ([ptr, ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.POINTER(BiPackedWeightDesc), ctypes.c_void_p], st),
                "bi_addmm_packed": ([ptr, ptr, ctypes.POINTER(BiPackedWeightDesc), ptr,
                                     ctypes.c_void_p], st),
                "bi_conv_packed_weight_bytes": ([ctypes.c_int64] * 4, ctypes.c_int64),
                "bi_conv_pack_weight": ([ptr, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.POINTER(BiConvPackedWeightDesc), ctypes.c_void_p], st),
                "bi_conv2d_patch_packed": ([ptr, ctypes.POINTER(BiConvPackedWeightDesc), ptr, ptr,
                                            ctypes.c_void_p], st),
                "bi_device_status": ([ctypes.c_void_p], st),
                "bi_debug_expire_wait": ([ctypes.c_uint64, ctypes.c_void_p], st),
                "bi_status_string": ([st], ctypes.c_char_p),
                "bi_last_error_message": ([], ctypes.c_char_p),
                "bi_abi_version": ([], ctypes.c_int32),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _desc(t: torch.Tensor | None, name: str) -> BiTensor | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: expected a CUDA tensor, got {t.device}")
    if t.dtype not in _DTYPES:
        raise TypeError(f"{name}: unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError(f"{name}: rank {t.dim()} > 4")
    d = BiTensor()
    d.ptr = t.data_ptr() if t.numel() else (t.data_ptr() or None)
    d.ndim = t.dim()
    d.dtype = _DTYPES[t.dtype]
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _ref(d: BiTensor | None):
    return ctypes.byref(d) if d is not None else None


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(lib, op: str, status: int):
    if status != BI_OK:
        name = lib.bi_status_string(status).decode()
        detail = lib.bi_last_error_message().decode()
        raise BiError(op, status, name, detail)


def bi_mm(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
          out_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """out[m,n] = sum_k a[m,k] b[k,n]  (bf16 inputs, fp32 accumulation)."""
    lib = load()
    if out is None:
        out = torch.empty((a.shape[0], b.shape[1]), dtype=out_dtype, device=a.device)
    da, db, dc = _desc(a, "a"), _desc(b, "b"), _desc(out, "out")
    _check(lib, "bi_mm", lib.bi_mm(_ref(da), _ref(db), _ref(dc), _stream(stream)))
    return out


def bi_addmm(bias: torch.Tensor, a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
             out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """out[m,n] = sum_k a[m,k] b[k,n] + bias[n]."""
    lib = load()
    if out is None:
        out = torch.empty((a.shape[0], b.shape[1]), dtype=out_dtype, device=a.device)
    dbias, da, db, dc = _desc(bias, "bias"), _desc(a, "a"), _desc(b, "b"), _desc(out, "out")
    _check(lib, "bi_addmm", lib.bi_addmm(_ref(dbias), _ref(da), _ref(db), _ref(dc), _stream(stream)))
    return out


def bi_bmm(a: torch.Tensor, b: torch.Tensor, alpha: float = 1.0, out: torch.Tensor | None = None,
           out_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """out[l] = alpha * a[l] @ b[l]."""
    lib = load()
    if out is None:
        out = torch.empty((a.shape[0], a.shape[1], b.shape[2]), dtype=out_dtype, device=a.device)
    da, db, dc = _desc(a, "a"), _desc(b, "b"), _desc(out, "out")
    _check(lib, "bi_bmm", lib.bi_bmm(_ref(da), _ref(db), _ref(dc), float(alpha), _stream(stream)))
    return out


def _pair(v):
    return (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))


def conv_out_hw(h, w, kh, kw, stride, padding, dilation):
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    dh, dw = _pair(dilation)
    return (h + 2 * ph - dh * (kh - 1) - 1) // sh + 1, (w + 2 * pw - dw * (kw - 1) - 1) // sw + 1


def bi_conv2d_patch(x: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None = None, stride=1,
                    padding=0, dilation=1, groups: int = 1, out: torch.Tensor | None = None,
                    out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """2-D convolution (as nn.Conv2d) computed per sample as an implicit-im2col product."""
    lib = load()
    if out is None:
        ho, wo = conv_out_hw(x.shape[2], x.shape[3], w.shape[2], w.shape[3], stride, padding, dilation)
        out = torch.empty((x.shape[0], w.shape[0], max(ho, 0), max(wo, 0)), dtype=out_dtype,
                          device=x.device)
    arr = ctypes.c_int32 * 2
    st, pd, dl = arr(*_pair(stride)), arr(*_pair(padding)), arr(*_pair(dilation))
    dx, dw_, db, dy = _desc(x, "x"), _desc(w, "w"), _desc(bias, "bias"), _desc(out, "out")
    _check(lib, "bi_conv2d_patch",
           lib.bi_conv2d_patch(_ref(dx), _ref(dw_), _ref(db), _ref(dy), st, pd, dl, int(groups),
                               _stream(stream)))
    return out


def bi_softmax_lastdim(s: torch.Tensor, out: torch.Tensor | None = None,
                       out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """Row softmax of a 2-D fp32 tensor over its last dimension."""
    lib = load()
    if out is None:
        out = torch.empty(s.shape, dtype=out_dtype, device=s.device)
    ds, dp = _desc(s, "s"), _desc(out, "out")
    _check(lib, "bi_softmax_lastdim", lib.bi_softmax_lastdim(_ref(ds), _ref(dp), _stream(stream)))
    return out


def bi_rmsnorm_lastdim(x: torch.Tensor, weight: torch.Tensor | None = None, eps: float = 1e-6,
                       out: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
                       stream=None) -> torch.Tensor:
    """RMSNorm of each row of a 2-D tensor over its last dimension (output in x's
    dtype unless out / out_dtype says otherwise)."""
    lib = load()
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    dx, dw, dy = _desc(x, "x"), _desc(weight, "weight"), _desc(out, "out")
    _check(lib, "bi_rmsnorm_lastdim",
           lib.bi_rmsnorm_lastdim(_ref(dx), _ref(dw), ctypes.c_float(eps), _ref(dy), _stream(stream)))
    return out


def bi_log_softmax_lastdim(s: torch.Tensor, out: torch.Tensor | None = None,
                           out_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """Row log-softmax of a 2-D tensor over its last dimension."""
    lib = load()
    if out is None:
        out = torch.empty(s.shape, dtype=out_dtype, device=s.device)
    ds, dy = _desc(s, "s"), _desc(out, "out")
    _check(lib, "bi_log_softmax_lastdim", lib.bi_log_softmax_lastdim(_ref(ds), _ref(dy), _stream(stream)))
    return out


def bi_mean_lastdim(x: torch.Tensor, out: torch.Tensor | None = None,
                    out_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """Mean of each row of a 2-D tensor over its last dimension: a [R] result."""
    lib = load()
    if out is None:
        out = torch.empty((x.shape[0],), dtype=out_dtype, device=x.device)
    dx, dy = _desc(x, "x"), _desc(out, "out")
    _check(lib, "bi_mean_lastdim", lib.bi_mean_lastdim(_ref(dx), _ref(dy), _stream(stream)))
    return out


def bi_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                 out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                 stream=None) -> torch.Tensor:
    """Fused attention softmax(scale * q k^T) v per head: q [L, Tq, D], k / v
    [L, Tk, D] bf16, D = 64, 128 or 256; returns [L, Tq, D] (fp32 unless out /
    out_dtype)."""
    lib = load()
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], q.shape[2]), dtype=out_dtype, device=q.device)
    dq, dk, dv, do = _desc(q, "q"), _desc(k, "k"), _desc(v, "v"), _desc(out, "out")
    _check(lib, "bi_attention",
           lib.bi_attention(_ref(dq), _ref(dk), _ref(dv), ctypes.c_float(scale), _ref(do), _stream(stream)))
    return out


def bi_attention_workspace_bytes(L: int, Tq: int, Tk: int, D: int = 256) -> int:
    return int(load().bi_attention_workspace_bytes(int(L), int(Tq), int(Tk), int(D)))


def bi_attention_ws(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                    out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Fused attention for any key range: for Tk > 2048 a workspace of
    bi_attention_workspace_bytes(L, Tq, Tk, D) bytes is used (allocated here when
    not given)."""
    lib = load()
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], q.shape[2]), dtype=out_dtype, device=q.device)
    need = bi_attention_workspace_bytes(q.shape[0], q.shape[1], k.shape[1], q.shape[2])
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wptr = ctypes.c_void_p(workspace.data_ptr() if workspace is not None else None)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    dq, dk, dv, do = _desc(q, "q"), _desc(k, "k"), _desc(v, "v"), _desc(out, "out")
    _check(lib, "bi_attention_ws",
           lib.bi_attention_ws(_ref(dq), _ref(dk), _ref(dv), ctypes.c_float(scale), _ref(do), wptr,
                               ctypes.c_int64(wbytes), _stream(stream)))
    return out


def bi_attention_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float,
                         out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                         stream=None) -> torch.Tensor:
    """Fused attention for any key range without a workspace argument: long
    key ranges use the library's static device scratch (64 MiB per device)."""
    lib = load()
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], q.shape[2]), dtype=out_dtype, device=q.device)
    dq, dk, dv, do = _desc(q, "q"), _desc(k, "k"), _desc(v, "v"), _desc(out, "out")
    _check(lib, "bi_attention_noalloc",
           lib.bi_attention_noalloc(_ref(dq), _ref(dk), _ref(dv), ctypes.c_float(scale), _ref(do), _stream(stream)))
    return out


def bi_packed_weight_bytes(K: int, N: int) -> int:
    return int(load().bi_packed_weight_bytes(int(K), int(N)))


def bi_pack_weight(b: torch.Tensor, stream=None) -> PackedWeight:
    """Packs a [K, N] bf16 weight (row-major, or a transposed view of [N, K])."""
    lib = load()
    K, N = b.shape
    nbytes = bi_packed_weight_bytes(K, N)
    buf = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=b.device)
    desc = BiPackedWeightDesc()
    db = _desc(b, "b")
    _check(lib, "bi_pack_weight",
           lib.bi_pack_weight(_ref(db), ctypes.c_void_p(buf.data_ptr()), nbytes, ctypes.byref(desc),
                              _stream(stream)))
    return PackedWeight(buf, desc)


def bi_addmm_packed(bias: torch.Tensor | None, a: torch.Tensor, b: PackedWeight,
                    out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.bfloat16,
                    stream=None) -> torch.Tensor:
    """out = a @ B (+ bias) with B packed; bit-identical to bi_mm / bi_addmm on the plain weight."""
    lib = load()
    if out is None:
        out = torch.empty((a.shape[0], b.shape[1]), dtype=out_dtype, device=a.device)
    dbias, da, dc = _desc(bias, "bias"), _desc(a, "a"), _desc(out, "out")
    _check(lib, "bi_addmm_packed",
           lib.bi_addmm_packed(_ref(dbias), _ref(da), ctypes.byref(b.desc), _ref(dc), _stream(stream)))
    return out


def bi_conv_packed_weight_bytes(Co: int, C: int, KH: int, KW: int) -> int:
    return int(load().bi_conv_packed_weight_bytes(int(Co), int(C), int(KH), int(KW)))


def bi_conv_pack_weight(w: torch.Tensor, stream=None) -> ConvPackedWeight:
    """Packs a [Co, C, KH, KW] bf16 patch-embedding filter (KW <= 16)."""
    lib = load()
    Co, C, KH, KW = w.shape
    nbytes = bi_conv_packed_weight_bytes(Co, C, KH, KW)
    buf = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=w.device)
    desc = BiConvPackedWeightDesc()
    dw_ = _desc(w, "w")
    _check(lib, "bi_conv_pack_weight",
           lib.bi_conv_pack_weight(_ref(dw_), ctypes.c_void_p(buf.data_ptr()), nbytes, ctypes.byref(desc),
                                   _stream(stream)))
    return ConvPackedWeight(buf, desc)


def bi_conv2d_patch_packed(x: torch.Tensor, w: ConvPackedWeight, bias: torch.Tensor | None = None,
                           out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.bfloat16,
                           stream=None) -> torch.Tensor:
    """Non-overlapping patch convolution (stride = kernel size) with a packed filter."""
    lib = load()
    Co, C, KH, KW = w.shape
    if out is None:
        out = torch.empty((x.shape[0], Co, x.shape[2] // KH, x.shape[3] // KW), dtype=out_dtype,
                          device=x.device)
    dx, db, dy = _desc(x, "x"), _desc(bias, "bias"), _desc(out, "out")
    _check(lib, "bi_conv2d_patch_packed",
           lib.bi_conv2d_patch_packed(_ref(dx), ctypes.byref(w.desc), _ref(db), _ref(dy), _stream(stream)))
    return out


def bi_device_status(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device status word as a status code."""
    lib = load()
    return int(lib.bi_device_status(_stream(stream)))


def bi_debug_expire_wait(limit_ns: int, stream=None) -> None:
    """Launches the bounded-wait test kernel (a wait that nothing ends)."""
    lib = load()
    _check(lib, "bi_debug_expire_wait", lib.bi_debug_expire_wait(int(limit_ns), _stream(stream)))


def last_error_message() -> str:
    return load().bi_last_error_message().decode()


def status_string(status: int) -> str:
    return load().bi_status_string(int(status)).decode()
