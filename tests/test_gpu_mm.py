"""GPU parity of bi_mm / bi_addmm against the fp64 oracle, operand layouts,
ragged tails, exact integer cases, and bitwise batch invariance / run-to-run
determinism ("Batch-Invariant Kernel Design: Conv2d and Attention BMM",
section "The two correctness tests": agreement with a reference within a
tolerance, and sample 0 alone vs in a batch bit for bit)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_gemm_bi_gb300 import binding, inputs
from tests.gpu_helpers import bits_equal, check_tolerance, padded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load()
    yield
    assert binding.bi_device_status() == binding.BI_OK


def _to_gpu(*ts):
    return [t.cuda() for t in ts]


# -- first: the smallest possible case, exact --------------------------------

def test_single_tile_small_integers_exact():
    a = inputs.small_int_bf16((8, 64), -3, 3, 1)
    b = inputs.small_int_bf16((64, 16), -3, 3, 2)
    ref, _ = oracle.mm(a, b)
    c = binding.bi_mm(*_to_gpu(a, b))
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().double().numpy(), ref)


@pytest.mark.parametrize("b_layout", ["mn", "k"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 24, 40), (128, 256, 64), (129, 264, 72),
                                   (300, 520, 200), (77, 1000, 1000)])
def test_small_integers_bit_exact(shape, b_layout):
    # every partial sum is an integer below 2^24: exact in fp32 in any order,
    # so the GPU must match the oracle bit for bit (fp32 output)
    M, N, K = shape
    a = inputs.small_int_bf16((M, K), -4, 4, 3)
    bt = inputs.small_int_bf16((N, K), -4, 4, 4)
    b = bt.t().contiguous() if b_layout == "mn" else bt.t()
    ref, _ = oracle.mm(a, b)
    ag = a.cuda()
    bg = b.contiguous().cuda() if b_layout == "mn" else bt.cuda().t()
    c = binding.bi_mm(ag, bg)
    assert np.array_equal(c.cpu().double().numpy(), ref)


# -- tolerance on real-valued inputs, every layout and ragged tails ----------

RAGGED = [(1, 128, 256), (3, 136, 72), (31, 264, 200), (130, 392, 520), (257, 128, 64),
          (64, 520, 1000), (200, 8, 8)]


@pytest.mark.parametrize("b_layout", ["mn", "k"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", RAGGED)
def test_mm_matches_oracle(shape, out_dtype, b_layout):
    M, N, K = shape
    a = inputs.normal_bf16((M, K), 1.0, 10)
    w = inputs.normal_bf16((K, N), 0.05, 11)
    ref, absum = oracle.mm(a, w)
    bg = w.cuda() if b_layout == "mn" else w.t().contiguous().cuda().t()
    c = binding.bi_mm(a.cuda(), bg, out_dtype=out_dtype)
    check_tolerance(c, ref, absum, f"mm {shape} {out_dtype} {b_layout}")


@pytest.mark.parametrize("bias_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(1, 264, 128), (45, 520, 200), (130, 136, 1024)])
def test_addmm_matches_oracle(shape, bias_dtype):
    M, N, K = shape
    x = inputs.normal_bf16((M, K), 1.0, 12)
    w = inputs.normal_bf16((K, N), 0.02, 13)
    bias = inputs.normal_bf16((N,), 0.01, 14)
    ref, absum = oracle.mm(x, w, bias=bias)
    if bias_dtype == torch.float32:
        bias_g = bias.float().cuda()   # same values, fp32 storage
    else:
        bias_g = bias.cuda()
    for out_dtype in (torch.bfloat16, torch.float32):
        c = binding.bi_addmm(bias_g, x.cuda(), w.cuda(), out_dtype=out_dtype)
        check_tolerance(c, ref, absum, f"addmm {shape} {out_dtype}")


def test_strided_operands_and_output_stay_in_their_views():
    M, N, K = 70, 200, 136
    a = inputs.normal_bf16((M, K), 1.0, 20)
    w = inputs.normal_bf16((K, N), 0.05, 21)
    bias = inputs.normal_bf16((N,), 0.01, 22)
    ref, absum = oracle.mm(a, w, bias=bias)
    _, ag = padded(M, K, K + 24)
    ag.copy_(a.cuda())
    _, wg = padded(K, N, N + 40)
    wg.copy_(w.cuda())
    # output view with row stride 256 inside a canary-filled buffer
    store = torch.full((M + 2, 256), 12345.0, dtype=torch.float32, device="cuda")
    out = store[1:M + 1, 8:8 + N]
    bg = torch.empty(N * 3, dtype=torch.bfloat16, device="cuda")
    bias_view = bg[::3]
    bias_view.copy_(bias.cuda())
    binding.bi_addmm(bias_view, ag, wg, out=out)
    check_tolerance(out, ref, absum, "strided addmm")
    mask = torch.ones_like(store, dtype=torch.bool)
    mask[1:M + 1, 8:8 + N] = False
    assert torch.all(store[mask] == 12345.0), "a write landed outside the output view"


def test_empty_and_degenerate_shapes():
    a = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, 32, dtype=torch.bfloat16, device="cuda")
    assert binding.bi_mm(a, w).shape == (0, 32)
    # K == 0: an empty reduction gives exactly the bias
    bias = inputs.normal_bf16((40,), 1.0, 5).cuda()
    c = binding.bi_addmm(bias, torch.zeros(3, 0, dtype=torch.bfloat16, device="cuda"),
                         torch.zeros(0, 40, dtype=torch.bfloat16, device="cuda"), out_dtype=torch.float32)
    assert torch.equal(c, bias.float().expand(3, 40))
    c = binding.bi_mm(torch.zeros(2, 0, dtype=torch.bfloat16, device="cuda"),
                      torch.zeros(0, 8, dtype=torch.bfloat16, device="cuda"))
    assert torch.equal(c, torch.zeros(2, 8, device="cuda"))


def test_unsupported_layout_reports_and_leaves_output_untouched():
    a = torch.zeros(4, 60, dtype=torch.bfloat16, device="cuda")     # row stride 60: not 16-byte
    w = torch.zeros(60, 32, dtype=torch.bfloat16, device="cuda")
    out = torch.full((4, 32), 7.0, device="cuda")
    with pytest.raises(binding.BiError) as ei:
        binding.bi_mm(a, w, out=out)
    assert ei.value.status == binding.BI_ERR_UNSUPPORTED_LAYOUT
    assert torch.all(out == 7.0)


# -- batch invariance --------------------------------------------------------

def test_tiny_workload_row0_invariant_and_exact_rows():
    # A [M,256] ~N(0,1), W [256,128] ~N(0,0.02), fp32 output, M in {1,2,3,8,31,32,64}
    a, w = inputs.tiny_mm(64)
    ref, absum = oracle.mm(a, w)
    ag, wg = a.cuda(), w.cuda()
    full = binding.bi_mm(ag, wg)
    check_tolerance(full, ref, absum, "tiny mm M=64")
    for M in inputs.TINY_MM_M:
        c = binding.bi_mm(ag[:M], wg)
        check_tolerance(c, ref[:M], absum[:M], f"tiny mm M={M}")
        # every row, not only row 0, is bit-identical to the same row in the M=64 run
        assert bits_equal(c, full[:M]), f"M={M}"


def test_distractor_rows_do_not_touch_row0():
    K, N = 1024, 520
    a = inputs.normal_bf16((300, K), 1.0, 30).cuda()
    w = inputs.normal_bf16((K, N), 0.02, 31).cuda()
    alone = binding.bi_mm(a[:1], w)
    for fill in (2.0 ** 100, -(2.0 ** 100), float("nan"), float("inf")):
        batch = a.clone()
        batch[1:] = fill
        c = binding.bi_mm(batch, w)
        assert bits_equal(c[:1], alone), fill


def test_run_to_run_bitwise():
    # "Unmasking the True Culprit", section "Why Most GPU Kernels Don't Use
    # Atomic Operations": repeated products of the same inputs are identical.
    a = inputs.normal_bf16((2048, 2048), 1.0, 40).cuda()
    w = inputs.normal_bf16((2048, 2048), 1.0, 41).cuda()
    ref = binding.bi_mm(a, w)
    for _ in range(50):
        assert bits_equal(binding.bi_mm(a, w), ref)


def test_linspace_batch_vs_single_row():
    # the page's structured example: mm(a[:1], b) vs mm(a, b)[:1] with
    # linspace inputs ("Unmasking the True Culprit", section "The Batch
    # Invariance Problem Revealed")
    B, D = 2048, 4096
    a = torch.linspace(-100, 100, B * D).reshape(B, D).to(torch.bfloat16).cuda()
    b = torch.linspace(-100, 100, D * D).reshape(D, D).to(torch.bfloat16).cuda()
    out1 = binding.bi_mm(a[:1], b)
    out2 = binding.bi_mm(a, b)[:1]
    assert bits_equal(out1, out2)
    ref, absum = oracle.mm(a[:1].cpu(), b.cpu())
    check_tolerance(out1, ref, absum, "linspace row 0")


# -- packed weights ----------------------------------------------------------

@pytest.mark.parametrize("layout", ["mn", "k"])
@pytest.mark.parametrize("shape", [(1, 264, 200), (17, 256, 64), (130, 520, 1000), (257, 136, 72),
                                   (3, 14336, 4096)])
def test_packed_weight_is_bit_identical_to_plain(shape, layout):
    M, N, K = shape
    a = inputs.normal_bf16((M, K), 1.0, 80).cuda()
    w = inputs.normal_bf16((K, N), 0.02, 81).cuda()
    bias = inputs.normal_bf16((N,), 0.01, 82).cuda()
    wv = w if layout == "mn" else w.t().contiguous().t()
    packed = binding.bi_pack_weight(wv)
    assert packed.desc.layout == (1 if layout == "mn" else 2)
    for out_dtype in (torch.float32, torch.bfloat16):
        plain = binding.bi_addmm(bias, a, wv, out_dtype=out_dtype)
        got = binding.bi_addmm_packed(bias, a, packed, out_dtype=out_dtype)
        assert bits_equal(got, plain)
        plain_mm = binding.bi_mm(a, wv, out_dtype=out_dtype)
        assert bits_equal(binding.bi_addmm_packed(None, a, packed, out_dtype=out_dtype), plain_mm)
    if M <= 300 and K <= 1000:
        ref, absum = oracle.mm(a.cpu(), w.cpu(), bias=bias.cpu())
        check_tolerance(binding.bi_addmm_packed(bias, a, packed, out_dtype=torch.float32), ref, absum,
                        f"packed {shape}")


def test_packed_weight_row0_invariant_and_validation():
    K, N = 1024, 520
    a = inputs.normal_bf16((300, K), 1.0, 83).cuda()
    w = inputs.normal_bf16((K, N), 0.02, 84).cuda()
    packed = binding.bi_pack_weight(w)
    full = binding.bi_addmm_packed(None, a, packed)
    for M in (1, 2, 7, 64, 129, 300):
        assert bits_equal(binding.bi_addmm_packed(None, a[:M], packed), full[:M])
    # a mismatched K is refused before launch
    with pytest.raises(binding.BiError) as ei:
        binding.bi_addmm_packed(None, a[:, :512], packed)
    assert ei.value.status == binding.BI_ERR_SHAPE_MISMATCH
    # a descriptor claiming a too-small buffer is refused
    bad = binding.PackedWeight(packed.buffer, binding.BiPackedWeightDesc(
        packed.desc.ptr, packed.desc.bytes - 16, K, N, packed.desc.layout, packed.desc.tile_n))
    with pytest.raises(binding.BiError) as ei:
        binding.bi_addmm_packed(None, a, bad)
    assert ei.value.status == binding.BI_ERR_INVALID_ARG


def test_short_a_layout_matches_general_layout_bitwise():
    # M <= 32 runs with 32-row A stages, larger M with 128-row stages; every
    # row must come out with the same bits either way, distractors included.
    K, N = 2048, 776
    a = inputs.normal_bf16((300, K), 1.0, 90).cuda()
    w = inputs.normal_bf16((K, N), 0.02, 91).cuda()
    bias = inputs.normal_bf16((N,), 0.01, 92).cuda()
    general = binding.bi_addmm(bias, a, w, out_dtype=torch.float32)       # M = 300
    packed = binding.bi_pack_weight(w)
    for M in (1, 2, 17, 31, 32, 33):
        assert bits_equal(binding.bi_addmm(bias, a[:M], w, out_dtype=torch.float32), general[:M]), M
        assert bits_equal(binding.bi_addmm_packed(bias, a[:M], packed, out_dtype=torch.float32),
                          general[:M]), M
    for fill in (float("nan"), float("inf"), 2.0 ** 100):
        d = a[:32].clone()
        d[1:] = fill
        assert bits_equal(binding.bi_addmm(bias, d, w, out_dtype=torch.float32)[:1], general[:1])


@pytest.mark.parametrize("b_layout", ["k", "mn"])
def test_weight_streaming_launches_match_the_others_bitwise(b_layout):
    # up to two 256-row tiles (M <= 512) the launch loads the weight with the
    # evict-first and A with the evict-last L2 priority; larger M, without;
    # the rows they share must carry the same bits (plain and packed weight)
    K, N = 1024, 1000
    a = inputs.normal_bf16((1100, K), 1.0, 93).cuda()
    w = inputs.normal_bf16((K, N), 0.02, 94)
    wg = w.t().contiguous().cuda().t() if b_layout == "k" else w.cuda()
    bias = inputs.normal_bf16((N,), 0.01, 95).cuda()
    full = binding.bi_addmm(bias, a, wg)                                  # 5 row tiles
    packed = binding.bi_pack_weight(wg)
    for M in (1, 33, 256, 257, 511, 512, 513, 768):
        assert bits_equal(binding.bi_addmm(bias, a[:M], wg), full[:M]), M
        assert bits_equal(binding.bi_addmm_packed(bias, a[:M], packed), full[:M]), M
    ref, absum = oracle.mm(a[:3].cpu(), w, bias=bias.cpu())
    check_tolerance(full[:3], ref, absum, "streamed-weight rows")


# -- tile count vs resident CTA pairs ---------------------------------------

@pytest.mark.parametrize("K", [64, 320, 4096])
def test_column_count_does_not_change_shared_columns(K):
    # 38 column tiles leave pairs idle, 76 fill the GPU, 80 make pairs take a
    # second tile; the columns the three problems share must agree bit for
    # bit, for plain MN-major and packed weights, with a ragged last tile.
    a = inputs.normal_bf16((40, K), 1.0, 93).cuda()
    w = inputs.normal_bf16((K, 256 * 80), 0.02, 94).cuda()
    bias = inputs.normal_bf16((256 * 80,), 0.01, 95).cuda()
    widths = (256 * 37 + 72, 256 * 75 + 8, 256 * 80)
    for M in (1, 29, 40):
        outs = [binding.bi_addmm(bias[:n], a[:M], w[:, :n], out_dtype=torch.float32) for n in widths]
        packs = [binding.bi_addmm_packed(bias[:n], a[:M], binding.bi_pack_weight(w[:, :n]),
                                         out_dtype=torch.float32) for n in widths]
        for o, pk, n in zip(outs, packs, widths):
            assert bits_equal(o, outs[-1][:, :n]), (M, n)
            assert bits_equal(pk, o), (M, n)
    cols = [0, 1, 256 * 37 + 71, 256 * 75 + 7, 256 * 80 - 1]
    ref, absum = oracle.mm(a[:3].cpu(), w[:, cols].cpu(), bias=bias[cols].cpu())
    check_tolerance(outs[-1][:, cols][:3], ref, absum, f"split stream K={K}")
