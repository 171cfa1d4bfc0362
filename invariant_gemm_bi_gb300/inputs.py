"""Seeded synthetic inputs for the five contraction workloads and the row
reductions.

This module draws random numbers and nothing else: it holds none of the
contractions' arithmetic, so both the CUDA path and the CPU oracle can take
their inputs from it.  Every tensor is drawn in fp32 from a seeded
``torch.Generator`` and rounded once to bf16 or fp16 (round-to-nearest-even),
except the fp32 logits, which are kept as drawn.

Seed scheme: the activation-like operand (A, x, images, Q) uses seed 0, the
weight-like operand (W, K) seed 1, bias / V seed 2.  Sweeps over M (or B)
draw the largest size once and slice prefixes, so row 0 / sample 0 / head 0
are the same bits at every size.

The shapes and distributions mirror the layers the pages trace: a tiny
linear layer, an LLM MLP projection (4096 -> 14336), the SigLIP patch
embedding (3x224x224 images, 14x14 patches, 1152 channels), joint-model
attention (816 tokens, head dim 256, 8 heads) and a large square product.
No dataset or trained weight is involved.
"""
from __future__ import annotations

import torch

SEED_ACT, SEED_WEIGHT, SEED_AUX = 0, 1, 2


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded to bf16."""
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=_gen(seed, device))
    return t.to(torch.bfloat16)


def normal_f16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded to fp16."""
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=_gen(seed, device))
    return t.to(torch.float16)


def uniform_bf16(shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    """U(lo, hi) drawn in fp32, rounded to bf16."""
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.uniform_(lo, hi, generator=_gen(seed, device))
    return t.to(torch.bfloat16)


def normal_f32(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 (no rounding)."""
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=_gen(seed, device))
    return t


def small_int_bf16(shape, lo: int, hi: int, seed: int, device="cpu") -> torch.Tensor:
    """Integers uniform in [lo, hi] stored as bf16 (exact for |v| <= 256)."""
    t = torch.randint(lo, hi + 1, shape, generator=_gen(seed, device), device=device)
    return t.to(torch.bfloat16)


# -- the five workloads -------------------------------------------------------

TINY_MM_M = (1, 2, 3, 8, 31, 32, 64)
LLM_ADDMM_M = (1, 2, 4, 8, 16, 32, 63, 64, 128, 512, 2048, 8192)
PATCH_EMBED_B = (1, 8, 32)
ATTENTION_B = (1, 4, 32)
SQUARE_MM_M = (1, 16, 256, 4096, 16384)


def tiny_mm(m_max: int = 64, device="cpu"):
    """A [M,256] ~N(0,1), W [256,128] ~N(0,0.02); fp32 output."""
    a = normal_bf16((m_max, 256), 1.0, SEED_ACT, device)
    w = normal_bf16((256, 128), 0.02, SEED_WEIGHT, device)
    return a, w


LLM_ADDMM_F16_M = (1, 16, 512, 8192)


def llm_addmm_f16(m_max: int = 8192, device="cpu", k: int = 4096, n: int = 14336):
    """The LLM-linear workload with fp16 operands (same distributions and seeds), fp16 output."""
    x = normal_f16((m_max, k), 1.0, SEED_ACT, device)
    w = normal_f16((k, n), 0.02, SEED_WEIGHT, device)
    bias = normal_f16((n,), 0.01, SEED_AUX, device)
    return x, w, bias


def llm_addmm(m_max: int = 8192, device="cpu", k: int = 4096, n: int = 14336):
    """x [M,4096] ~N(0,1), W [4096,14336] ~N(0,0.02), bias [14336] ~N(0,0.01); bf16 output."""
    x = normal_bf16((m_max, k), 1.0, SEED_ACT, device)
    w = normal_bf16((k, n), 0.02, SEED_WEIGHT, device)
    bias = normal_bf16((n,), 0.01, SEED_AUX, device)
    return x, w, bias


def patch_embed(b_max: int = 32, device="cpu"):
    """images [B,3,224,224] ~U(-1,1), weight [1152,3,14,14] ~N(0,0.02), bias [1152] ~N(0,0.01)."""
    x = uniform_bf16((b_max, 3, 224, 224), -1.0, 1.0, SEED_ACT, device)
    w = normal_bf16((1152, 3, 14, 14), 0.02, SEED_WEIGHT, device)
    bias = normal_bf16((1152,), 0.01, SEED_AUX, device)
    return x, w, bias


def attention(b_max: int = 32, heads: int = 8, t: int = 816, d: int = 256, device="cpu"):
    """Q, K, V [B*heads, T, D] ~N(0,1) (Q seed 0, K seed 1, V seed 2)."""
    q = normal_bf16((b_max * heads, t, d), 1.0, SEED_ACT, device)
    k = normal_bf16((b_max * heads, t, d), 1.0, SEED_WEIGHT, device)
    v = normal_bf16((b_max * heads, t, d), 1.0, SEED_AUX, device)
    return q, k, v


def square_mm(m_max: int = 16384, device="cpu", n: int = 8192):
    """A [M,8192] ~N(0,1), W [8192,8192] ~N(0,0.01); fp32 output."""
    a = normal_bf16((m_max, n), 1.0, SEED_ACT, device)
    w = normal_bf16((n, n), 0.01, SEED_WEIGHT, device)
    return a, w


# -- row reductions over the last dimension -----------------------------------

RMSNORM_ROWS = (1, 8, 64, 512, 8192)
LOGITS_ROWS = (1, 8, 64)


def rmsnorm_hidden(rows: int = 8192, device="cpu", n: int = 4096):
    """Hidden states x [rows, 4096] ~N(0,1) bf16 and an RMSNorm gain [4096] ~U(0.5,1.5) bf16."""
    x = normal_bf16((rows, n), 1.0, SEED_ACT, device)
    w = uniform_bf16((n,), 0.5, 1.5, SEED_WEIGHT, device)
    return x, w


def vocab_logits(rows: int = 64, device="cpu", n: int = 128256):
    """Next-token logits [rows, 128256] ~N(0, 3^2) in fp32 (a Llama-3-sized vocabulary)."""
    return normal_f32((rows, n), 3.0, SEED_ACT, device)
