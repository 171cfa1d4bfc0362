"""fp64 CPU oracle for the batch-invariant contractions -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package never imports the product library: the two share no code.

The arithmetic lives in ``bi_oracle.c`` (plain C, double precision, one
sequential ascending-k sum per output element).  This module compiles it with
gcc on first use and marshals torch CPU tensors through ctypes.

Operation definitions followed (page title, section):
  * mm / addmm  -- "Unmasking the True Culprit: Why Temperature=0 Doesn't Mean
    Deterministic LLM Inference", section "Implementation Analysis: The
    matmul_persistent Function" (c = a @ b, optional bias added to every row);
  * bmm         -- "Batch-Invariant Kernel Design: Conv2d and Attention BMM",
    section "Kernel 2: Attention BMM" (one independent product per element of
    the flattened B*H dimension);
  * conv2d      -- same page, section "Kernel 1: Conv2d" (non-transposed 2-D
    convolution with stride, padding, dilation, groups) and "Batch-Invariant
    VLAs", section "Replacing nn.Conv2d" (unfold, flattened weight @ patches,
    plus bias);
  * softmax     -- the last-dimension softmax of the attention scores, one row
    at a time ("ai-infra handbook: deterministic inference", section on
    normalisation / softmax reductions).
  * attention   -- o = softmax(scale * q @ k^T) @ v per head over the whole
    key range ("ai-infra handbook: deterministic inference", section on fixed
    splitting: attention's key/value range split by a fixed length or not at
    all, its result independent of how queries are chunked).

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bi_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libbi_oracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_dbl = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile bi_oracle.c into libbi_oracle.so next to it (gcc, OpenMP).

    ``-ffp-contract=off`` keeps every multiply and add a separate rounding
    step on every host architecture (no fused multiply-add contraction).
    """
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            _int = ctypes.c_int
            lib.bio_mm.argtypes = [_i64, _i64, _i64, _int, _vp, _i64, _i64, _vp, _i64, _i64,
                                   _int, _vp, _i64, _dbl, _vp, _i64, _vp, _vp]
            lib.bio_mm.restype = None
            lib.bio_bmm.argtypes = [_i64, _i64, _i64, _i64, _int, _vp, _i64, _i64, _i64,
                                    _vp, _i64, _i64, _i64, _dbl, _vp, _vp]
            lib.bio_bmm.restype = None
            lib.bio_conv2d.argtypes = [_i64] * 14 + [_vp, _vp, _vp, _vp, _vp]
            lib.bio_conv2d.restype = None
            lib.bio_unfold.argtypes = [_i64] * 12 + [_vp, _vp]
            lib.bio_unfold.restype = None
            lib.bio_conv_out_size.argtypes = [_i64] * 5
            lib.bio_conv_out_size.restype = _i64
            lib.bio_softmax_rows.argtypes = [_i64, _i64, _vp, _i64, _vp]
            lib.bio_softmax_rows.restype = None
            lib.bio_rmsnorm_rows.argtypes = [_i64, _i64, _vp, _i64, _vp, _dbl, _vp]
            lib.bio_rmsnorm_rows.restype = None
            lib.bio_log_softmax_rows.argtypes = [_i64, _i64, _vp, _i64, _vp]
            lib.bio_log_softmax_rows.restype = None
            lib.bio_mean_rows.argtypes = [_i64, _i64, _vp, _i64, _vp, _vp]
            lib.bio_mean_rows.restype = None
            lib.bio_attention.argtypes = [_i64, _i64, _i64, _i64, _vp, _vp, _vp, _dbl, _vp, _vp, _vp]
            lib.bio_attention.restype = None
            lib.bio_round_bf16.argtypes = [_vp, _vp, _i64]
            lib.bio_round_bf16.restype = None
            lib.bio_round_f32.argtypes = [_vp, _vp, _i64]
            lib.bio_round_f32.restype = None
            lib.bio_sum_seq_f64.argtypes = [_vp, _i64]
            lib.bio_sum_seq_f64.restype = _dbl
            lib.bio_sum_seq_f32.argtypes = [_vp, _i64]
            lib.bio_sum_seq_f32.restype = ctypes.c_float
            lib.bio_bf16_bits_to_double.argtypes = [ctypes.c_uint16]
            lib.bio_bf16_bits_to_double.restype = _dbl
            lib.bio_f16_bits_to_double.argtypes = [ctypes.c_uint16]
            lib.bio_f16_bits_to_double.restype = _dbl
            lib.bio_num_threads.argtypes = []
            lib.bio_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _bf16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.bfloat16 or t.device.type != "cpu":
        raise TypeError(f"oracle expects CPU bfloat16 tensors, got {t.dtype} on {t.device}")
    return t


def _half(t: torch.Tensor) -> int:
    """1 for an fp16 tensor, 0 for bf16 (the 16-bit types the products take)."""
    if t.device.type != "cpu" or t.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"oracle expects CPU bfloat16 or float16 tensors, got {t.dtype} on {t.device}")
    return 1 if t.dtype == torch.float16 else 0


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if isinstance(t, torch.Tensor) else t.ctypes.data)


def num_threads() -> int:
    return int(_load().bio_num_threads())


def mm(a: torch.Tensor, b: torch.Tensor, bias: torch.Tensor | None = None,
       alpha: float = 1.0, rows=None):
    """fp64 ``alpha * a @ b (+ bias)`` for bf16 or fp16 a [M,K], b [K,N] of the
    same type (any strides); bias bf16 or fp16.

    Returns ``(c, absum)``: both float64 numpy arrays of shape [R, N], where
    R = M, or len(rows) when only the listed output rows are computed.
    ``absum = |alpha| * sum_k |a[m,k] b[k,n]| (+ |bias[n]|)`` -- the scale of
    the error bound the GPU result is held to.
    """
    lib = _load()
    in_f16 = _half(a)
    if _half(b) != in_f16:
        raise TypeError("a and b must have the same dtype")
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    rows_arr = None
    R = M
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        R = int(rows_arr.size)
    c = np.empty((R, N), dtype=np.float64)
    absum = np.empty((R, N), dtype=np.float64)
    bias_f16 = _half(bias) if bias is not None else 0
    lib.bio_mm(M, N, K, in_f16, _ptr(a), a.stride(0), a.stride(1), _ptr(b), b.stride(0), b.stride(1),
               bias_f16, _ptr(bias) if bias is not None else None, bias.stride(0) if bias is not None else 0,
               float(alpha), _ptr(rows_arr) if rows_arr is not None else None, R,
               _ptr(c), _ptr(absum))
    return c, absum


def bmm(a: torch.Tensor, b: torch.Tensor, alpha: float = 1.0):
    """fp64 ``alpha * a[l] @ b[l]`` for bf16 or fp16 a [L,M,K], b [L,K,N] of the same type (any strides).

    Returns ``(c, absum)`` float64 arrays of shape [L, M, N].
    """
    lib = _load()
    in_f16 = _half(a)
    if _half(b) != in_f16:
        raise TypeError("a and b must have the same dtype")
    L, M, K = a.shape
    L2, K2, N = b.shape
    if L != L2 or K != K2:
        raise ValueError("batch or inner dimensions differ")
    c = np.empty((L, M, N), dtype=np.float64)
    absum = np.empty((L, M, N), dtype=np.float64)
    lib.bio_bmm(L, M, N, K, in_f16, _ptr(a), a.stride(0), a.stride(1), a.stride(2),
                _ptr(b), b.stride(0), b.stride(1), b.stride(2), float(alpha), _ptr(c), _ptr(absum))
    return c, absum


def _pair(v):
    return (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))


def conv_out_size(n, k, s, p, d) -> int:
    return int(_load().bio_conv_out_size(n, k, s, p, d))


def conv2d(x: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None = None,
           stride=1, padding=0, dilation=1, groups: int = 1):
    """Direct fp64 2-D convolution (cross-correlation, as nn.Conv2d).

    x [B,C,H,W], w [Co,C/groups,KH,KW], bias [Co] or None; bf16, made
    contiguous here.  Returns ``(y, absum)`` float64 arrays [B,Co,Ho,Wo].
    """
    lib = _load()
    x = _bf16(x).contiguous()
    w = _bf16(w).contiguous()
    if bias is not None:
        bias = _bf16(bias).contiguous()
    B, C, H, W = x.shape
    Co, Cig, KH, KW = w.shape
    if C != Cig * groups or Co % groups:
        raise ValueError("channel / group mismatch")
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    dh, dw = _pair(dilation)
    Ho = conv_out_size(H, KH, sh, ph, dh)
    Wo = conv_out_size(W, KW, sw, pw, dw)
    y = np.empty((B, Co, Ho, Wo), dtype=np.float64)
    absum = np.empty((B, Co, Ho, Wo), dtype=np.float64)
    lib.bio_conv2d(B, C, H, W, Co, KH, KW, sh, sw, ph, pw, dh, dw, groups,
                   _ptr(x), _ptr(w), _ptr(bias) if bias is not None else None, _ptr(y), _ptr(absum))
    return y, absum


def unfold(x: torch.Tensor, kernel_size, stride=1, padding=0, dilation=1) -> torch.Tensor:
    """Explicit im2col: bf16 [B, C*KH*KW, Ho*Wo] in torch.nn.functional.unfold's layout."""
    lib = _load()
    x = _bf16(x).contiguous()
    B, C, H, W = x.shape
    KH, KW = _pair(kernel_size)
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    dh, dw = _pair(dilation)
    Ho = conv_out_size(H, KH, sh, ph, dh)
    Wo = conv_out_size(W, KW, sw, pw, dw)
    cols = torch.empty((B, C * KH * KW, Ho * Wo), dtype=torch.bfloat16)
    lib.bio_unfold(B, C, H, W, KH, KW, sh, sw, ph, pw, dh, dw, _ptr(x), _ptr(cols))
    return cols


def conv2d_via_unfold(x: torch.Tensor, w: torch.Tensor, bias: torch.Tensor | None = None,
                      stride=1, padding=0, dilation=1, groups: int = 1):
    """The unfold form: per sample and group, W_flat @ unfold(x) + bias (fp64).

    Shares the fp64 product routine with :func:`mm` but none of the direct
    convolution's index arithmetic, so agreement of the two pins both.
    """
    Co, Cig, KH, KW = w.shape
    B, C, H, W = x.shape
    cols = unfold(x, (KH, KW), stride, padding, dilation)
    L = cols.shape[2]
    Cog = Co // groups
    Kg = Cig * KH * KW
    wf = w.contiguous().reshape(Co, Kg)
    y = np.empty((B, Co, L), dtype=np.float64)
    absum = np.empty((B, Co, L), dtype=np.float64)
    for b in range(B):
        for g in range(groups):
            wg = wf[g * Cog:(g + 1) * Cog]
            colg = cols[b, g * Kg:(g + 1) * Kg]
            bg = bias[g * Cog:(g + 1) * Cog] if bias is not None else None
            # out[co, l] = sum_k wg[co,k] cols[k,l] + bias[co]: a product with
            # rows = output channels; bias per row, so add it here in fp64.
            c, ab = mm(wg, colg)
            if bg is not None:
                bv = bg.to(torch.float64).numpy()[:, None]
                c = c + bv
                ab = ab + np.abs(bv)
            y[b, g * Cog:(g + 1) * Cog] = c
            absum[b, g * Cog:(g + 1) * Cog] = ab
    Ho = conv_out_size(H, KH, _pair(stride)[0], _pair(padding)[0], _pair(dilation)[0])
    Wo = conv_out_size(W, KW, _pair(stride)[1], _pair(padding)[1], _pair(dilation)[1])
    return y.reshape(B, Co, Ho, Wo), absum.reshape(B, Co, Ho, Wo)


def softmax_rows(s: torch.Tensor) -> np.ndarray:
    """fp64 softmax over the last dim of an fp32 [R, N] tensor (row stride any)."""
    lib = _load()
    if s.dtype != torch.float32 or s.device.type != "cpu" or s.dim() != 2 or s.stride(1) != 1:
        raise TypeError("softmax_rows expects a CPU float32 [R, N] tensor with unit column stride")
    R, N = s.shape
    p = np.empty((R, N), dtype=np.float64)
    lib.bio_softmax_rows(R, N, _ptr(s), s.stride(0), _ptr(p))
    return p


def _rows_f64(x: torch.Tensor) -> np.ndarray:
    """A CPU [R, N] tensor of a floating type as a C-contiguous float64 array (exact)."""
    if x.device.type != "cpu" or x.dim() != 2 or x.dtype not in (torch.float32, torch.bfloat16, torch.float16):
        raise TypeError("expects a CPU fp32 / bf16 / fp16 [R, N] tensor")
    return np.ascontiguousarray(x.to(torch.float64).numpy())


def rmsnorm_rows(x: torch.Tensor, weight: torch.Tensor | None = None, eps: float = 1e-6) -> np.ndarray:
    """fp64 RMSNorm over the last dim: y = x * (1 / sqrt(mean(x^2) + eps)) * weight."""
    lib = _load()
    xd = _rows_f64(x)
    R, N = xd.shape
    wd = None
    if weight is not None:
        wd = np.ascontiguousarray(weight.to(torch.float64).numpy())
        if wd.shape != (N,):
            raise ValueError("weight must have N elements")
    y = np.empty((R, N), dtype=np.float64)
    lib.bio_rmsnorm_rows(R, N, _ptr(xd), N, _ptr(wd) if wd is not None else None, float(eps), _ptr(y))
    return y


def log_softmax_rows(s: torch.Tensor) -> np.ndarray:
    """fp64 log-softmax over the last dim: (s - max) - log(sum exp(s - max))."""
    lib = _load()
    sd = _rows_f64(s)
    R, N = sd.shape
    y = np.empty((R, N), dtype=np.float64)
    lib.bio_log_softmax_rows(R, N, _ptr(sd), N, _ptr(y))
    return y


def mean_rows(x: torch.Tensor):
    """fp64 mean over the last dim; returns (mean [R], mean of |x| [R])."""
    lib = _load()
    xd = _rows_f64(x)
    R, N = xd.shape
    y = np.empty((R,), dtype=np.float64)
    ya = np.empty((R,), dtype=np.float64)
    lib.bio_mean_rows(R, N, _ptr(xd), N, _ptr(y), _ptr(ya))
    return y, ya


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float):
    """fp64 attention per head: q [L, Tq, D], k / v [L, Tk, D] (bf16, fp16 or
    fp32 CPU tensors, any strides).  Returns (o [L, Tq, D], absum [L, Tq, D]
    = sum_j p_j |v_jd|, smax [L, Tq] = |scale| max_j sum_d |q_d k_jd|)."""
    lib = _load()
    for t in (q, k, v):
        if t.device.type != "cpu" or t.dim() != 3 or t.dtype not in (torch.float32, torch.bfloat16, torch.float16):
            raise TypeError("attention expects CPU fp32 / bf16 / fp16 [L, T, D] tensors")
    L, Tq, D = q.shape
    Tk = k.shape[1]
    if k.shape != (L, Tk, D) or v.shape != (L, Tk, D):
        raise ValueError("k and v must be [L, Tk, D] with q's L and D")
    qd, kd, vd = (np.ascontiguousarray(t.to(torch.float64).numpy()) for t in (q, k, v))
    o = np.empty((L, Tq, D), dtype=np.float64)
    ab = np.empty((L, Tq, D), dtype=np.float64)
    sm = np.empty((L, Tq), dtype=np.float64)
    lib.bio_attention(L, Tq, Tk, D, _ptr(qd), _ptr(kd), _ptr(vd), float(scale), _ptr(o), _ptr(ab), _ptr(sm))
    return o, ab, sm


def round_bf16(x: np.ndarray) -> torch.Tensor:
    """fp64 -> bf16 with one round-to-nearest-even step (bf16 tensor, same shape)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = torch.empty(x.shape, dtype=torch.bfloat16)
    lib.bio_round_bf16(_ptr(x), _ptr(out), x.size)
    return out


def round_f32(x: np.ndarray) -> torch.Tensor:
    """fp64 -> fp32 with one round-to-nearest-even step."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = torch.empty(x.shape, dtype=torch.float32)
    lib.bio_round_f32(_ptr(x), _ptr(out), x.size)
    return out


def sum_seq_f64(values) -> float:
    lib = _load()
    x = np.ascontiguousarray(np.asarray(values, dtype=np.float64))
    return float(lib.bio_sum_seq_f64(_ptr(x), x.size))


def sum_seq_f32(values) -> float:
    lib = _load()
    x = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    return float(lib.bio_sum_seq_f32(_ptr(x), x.size))


def bf16_bits_to_double(bits: int) -> float:
    return float(_load().bio_bf16_bits_to_double(bits & 0xFFFF))


def f16_bits_to_double(bits: int) -> float:
    return float(_load().bio_f16_bits_to_double(bits & 0xFFFF))
