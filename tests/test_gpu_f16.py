"""GPU parity of the fp16-input products (mm / addmm / bmm / packed) against the
fp64 oracle: the same fixed tile and K order as bf16, with A and B both fp16
("Unmasking the True Culprit: Why Temperature=0 Doesn't Mean Deterministic LLM
Inference", section "Implementation Analysis: The matmul_persistent Function":
one fixed configuration per input dtype), row-0 bit invariance across M, and
values only fp16 can hold arriving exactly."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_gemm_bi_gb300 import binding
from tests.gpu_helpers import bits_equal, check_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load()
    yield
    assert binding.bi_device_status() == binding.BI_OK


def _normal_f16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.float16)


def test_f16_small_integers_and_fine_fractions_exact():
    # half-integers up to 1024 and small integers (K = 304: rows of a whole
    # number of 16-byte units): every product and partial
    # sum is exact in fp32, so the fp32 output equals the oracle exactly
    g = torch.Generator().manual_seed(1)
    a = torch.randint(-1024, 1024, (37, 304), generator=g).to(torch.float16) + 0.5
    b = torch.randint(-8, 9, (304, 72), generator=g).to(torch.float16)
    ref, _ = oracle.mm(a, b)
    c = binding.bi_mm(a.cuda(), b.cuda(), out_dtype=torch.float32)
    assert np.array_equal(c.cpu().double().numpy(), ref)
    # 1 + 2^-10 is an fp16 value bf16 cannot hold
    one = torch.full((1, 1), 1.0 + 2.0 ** -10, dtype=torch.float16)
    c = binding.bi_mm(one.cuda(), torch.ones(1, 1, dtype=torch.float16).cuda(), out_dtype=torch.float32)
    assert c.item() == 1.0 + 2.0 ** -10


@pytest.mark.parametrize("b_layout", ["mn", "k"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", [(1, 264, 200), (130, 520, 1000), (257, 136, 72)])
def test_f16_mm_and_addmm_match_oracle(shape, out_dtype, b_layout):
    M, N, K = shape
    a = _normal_f16((M, K), 1.0, 2)
    w = _normal_f16((K, N), 0.05, 3)
    bias = _normal_f16((N,), 0.1, 4)
    wg = w.cuda() if b_layout == "mn" else w.t().contiguous().cuda().t()
    ref, absum = oracle.mm(a, w)
    check_tolerance(binding.bi_mm(a.cuda(), wg, out_dtype=out_dtype), ref, absum, f"f16 mm {shape}")
    ref, absum = oracle.mm(a, w, bias=bias)
    check_tolerance(binding.bi_addmm(bias.cuda(), a.cuda(), wg, out_dtype=out_dtype), ref, absum,
                    f"f16 addmm {shape}")


def test_f16_row0_invariant_across_m_and_run_to_run():
    K, N = 2048, 776
    a = _normal_f16((1000, K), 1.0, 5).cuda()
    w = _normal_f16((K, N), 0.02, 6).cuda()
    bias = _normal_f16((N,), 0.01, 7).cuda()
    full = binding.bi_addmm(bias, a, w, out_dtype=torch.float16)
    for M in (1, 2, 17, 32, 33, 128, 129, 300):
        c = binding.bi_addmm(bias, a[:M], w, out_dtype=torch.float16)
        assert bits_equal(c, full[:M]), M
    assert bits_equal(binding.bi_addmm(bias, a, w, out_dtype=torch.float16), full)
    rows = [0, 1, 500, 999]
    ref, absum = oracle.mm(a.cpu(), w.cpu(), bias=bias.cpu(), rows=rows)
    check_tolerance(full[rows], ref, absum, "f16 sampled rows")


def test_f16_bmm_with_alpha_and_batch_invariance():
    L, M, K, N = 6, 100, 136, 72
    a = _normal_f16((L, M, K), 1.0, 8)
    bt = _normal_f16((L, N, K), 1.0, 9)
    b = bt.transpose(1, 2)                        # K-major view, as Q @ K^T
    ref, absum = oracle.bmm(a, b, alpha=1.0 / 16)
    c = binding.bi_bmm(a.cuda(), bt.cuda().transpose(1, 2), alpha=1.0 / 16, out_dtype=torch.float32)
    check_tolerance(c, ref, absum, "f16 bmm")
    c0 = binding.bi_bmm(a[:1].cuda(), bt[:1].cuda().transpose(1, 2), alpha=1.0 / 16, out_dtype=torch.float32)
    assert bits_equal(c0, c[:1])


@pytest.mark.parametrize("layout", ["mn", "k"])
def test_f16_packed_weight_is_bit_identical_to_plain(layout):
    M, N, K = 19, 520, 1000
    a = _normal_f16((M, K), 1.0, 10).cuda()
    w = _normal_f16((K, N), 0.02, 11).cuda()
    bias = _normal_f16((N,), 0.01, 12).cuda()
    wv = w if layout == "mn" else w.t().contiguous().t()
    packed = binding.bi_pack_weight(wv)
    assert packed.desc.dtype == 1
    for od in (torch.float32, torch.float16):
        assert bits_equal(binding.bi_addmm_packed(bias, a, packed, out_dtype=od),
                          binding.bi_addmm(bias, a, wv, out_dtype=od))
    # a bf16 activation with an fp16 packed weight is refused before launch
    with pytest.raises(binding.BiError) as ei:
        binding.bi_addmm_packed(bias, a.to(torch.bfloat16), packed)
    assert ei.value.status == binding.BI_ERR_UNSUPPORTED_DTYPE


def test_mixed_operand_types_are_refused_before_launch():
    a = _normal_f16((8, 64), 1.0, 13).cuda()
    w = _normal_f16((64, 32), 0.1, 14).cuda().to(torch.bfloat16)
    out = torch.full((8, 32), 7.0, device="cuda")
    with pytest.raises(binding.BiError) as ei:
        binding.bi_mm(a, w, out=out)
    assert ei.value.status == binding.BI_ERR_UNSUPPORTED_DTYPE
    assert bool((out == 7.0).all())
