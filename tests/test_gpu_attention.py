"""GPU parity of the fused attention (bi_attention) against the fp64 oracle,
and its invariances: a head computed alone or among any number of heads, and a
query row computed among any other query rows, give the same bits ("ai-infra
handbook: deterministic inference", section on fixed splitting: attention's
key range is not split by load, and its result must not change with how
queries are chunked; "Batch-Invariant Kernel Design: Conv2d and Attention
BMM", section "Kernel 2: Attention BMM").

Tolerance per output element, from the oracle's o = ref, absum = sum_j p_j |v_jd|
and smax = |scale| max_j sum_d |q_d k_jd| of its row:
    |o - ref| <= (2^-8 + 2.2e-4 smax + 2^-20 smax + 1e-4 + Tk 2^-23) absum + u_out |ref|
2^-8: p is rounded to bf16 before it multiplies v (relative 2^-9, doubled for
the normalisation it does not share); 1e-4 smax bounds the fp32 tensor-core
error of a score (as the GEMM tests' 1e-4 sum |ab|), which moves a weight by
that much relative, twice over (numerator and denominator); 2^-20 smax covers
rounding the scaled score and the SFU's 2^x; 1e-4 the fp32 accumulation of
P V; Tk 2^-23 the running sum of weights; u_out (2^-8 bf16, 2^-24 fp32) the
final rounding.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_gemm_bi_gb300 import binding
from invariant_gemm_bi_gb300 import inputs
from tests.gpu_helpers import bits_equal

pytestmark = pytest.mark.gpu

U_OUT = {torch.bfloat16: 2.0 ** -8, torch.float32: 2.0 ** -24}
D = 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load()
    yield
    assert binding.bi_device_status() == binding.BI_OK


def _qkv(L, Tq, Tk, seed, d=D):
    q = inputs.normal_bf16((L, Tq, d), 1.0, seed)
    k = inputs.normal_bf16((L, Tk, d), 1.0, seed + 1)
    v = inputs.normal_bf16((L, Tk, d), 1.0, seed + 2)
    return q, k, v


def check_attention(o: torch.Tensor, ref, absum, smax, Tk: int, what: str = ""):
    g = o.detach().to("cpu", torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    sm = smax[..., None]
    bound = (2.0 ** -8 + 2.2e-4 * sm + 2.0 ** -20 * sm + 1e-4 + Tk * 2.0 ** -23) * absum + \
        U_OUT[o.dtype] * np.abs(ref)
    err = np.abs(g - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        det = [(tuple(i), g[tuple(i)], ref[tuple(i)], bound[tuple(i)]) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, e.g. {det}")


# (L, Tq, Tk): one query and one key; exactly one tile and one key block;
# ragged tails in both; more keys than queries and the reverse; the
# attention workload's sequence length (816 = 6 x 128 + 48)
SHAPES = [(1, 1, 1), (1, 128, 128), (2, 129, 64), (3, 200, 333), (1, 50, 1000), (2, 816, 816)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_attention_matches_oracle(shape, out_dtype):
    L, Tq, Tk = shape
    q, k, v = _qkv(L, Tq, Tk, 10)
    ref, absum, smax = oracle.attention(q, k, v, 1.0 / 16)
    o = binding.bi_attention(q.cuda(), k.cuda(), v.cuda(), 1.0 / 16, out_dtype=out_dtype)
    check_attention(o, ref, absum, smax, Tk, f"attention {shape} -> {out_dtype}")


@pytest.mark.parametrize("rising", [True, False])
def test_attention_running_maximum_rescales(rising):
    # scores that climb by ~20 per block (~30 in log2 units) force the running maximum to move
    # (and O and the running sum to be rescaled) at every block; falling
    # scores never move it after the first block
    L, Tq, Tk = 2, 130, 700
    q = (torch.ones(L, Tq, D) * 0.25).to(torch.bfloat16)
    ramp = torch.arange(Tk, dtype=torch.float32) / 10.0
    if not rising:
        ramp = ramp.flip(0)
    k = (ramp[None, :, None] * torch.ones(L, Tk, D)).to(torch.bfloat16)
    k[:, :, 1::2] *= -0.5                                   # vary the scores' mix of signs
    v = inputs.normal_bf16((L, Tk, D), 1.0, 20)
    ref, absum, smax = oracle.attention(q, k, v, 0.1)
    o = binding.bi_attention(q.cuda(), k.cuda(), v.cuda(), 0.1)
    check_attention(o, ref, absum, smax, Tk, f"rescale rising={rising}")


def test_attention_head_alone_equals_head_in_batch():
    # head 0 of sample 0 alone vs among 16 heads, with distractor heads full
    # of huge, infinite and NaN values
    q, k, v = _qkv(16, 300, 300, 30)
    q[5], k[6], v[7] = 2.0 ** 100, float("inf"), float("nan")
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    full = binding.bi_attention(qg, kg, vg, 1.0 / 16)
    for L in (1, 2, 8):
        assert bits_equal(binding.bi_attention(qg[:L], kg[:L], vg[:L], 1.0 / 16), full[:L]), L
    assert bits_equal(binding.bi_attention(qg[3:4], kg[3:4], vg[3:4], 1.0 / 16), full[3:4])
    ref, absum, smax = oracle.attention(q[:2], k[:2], v[:2], 1.0 / 16)
    check_attention(full[:2], ref, absum, smax, 300, "head 0/1 among distractors")
    # and run to run
    assert bits_equal(binding.bi_attention(qg, kg, vg, 1.0 / 16), full)


def test_attention_query_chunking_invariance():
    # a query row gives the same bits whatever other query rows come with it
    # and wherever it falls in a 128-row tile (chunked prefill)
    q, k, v = _qkv(2, 400, 500, 40)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    full = binding.bi_attention(qg, kg, vg, 1.0 / 16)
    for a, b in ((0, 1), (0, 300), (50, 400), (127, 129), (399, 400), (200, 333)):
        part = binding.bi_attention(qg[:, a:b].contiguous(), kg, vg, 1.0 / 16)
        assert bits_equal(part, full[:, a:b]), (a, b)


def test_attention_strided_inputs_and_output():
    # q, k, v as views of one packed [L, T, 3, 256] tensor (row stride 768),
    # output into a padded buffer: the same bits as contiguous operands
    L, T = 3, 250
    qkv = inputs.normal_bf16((L, T, 3, D), 1.0, 50)
    g = qkv.cuda()
    q, k, v = g[:, :, 0], g[:, :, 1], g[:, :, 2]
    ref_o = binding.bi_attention(q.contiguous(), k.contiguous(), v.contiguous(), 0.0625)
    big = torch.full((L, T + 3, D + 64), 7.0, device="cuda")
    out = big[:, 1:T + 1, 32:32 + D]
    binding.bi_attention(q, k, v, 0.0625, out=out)
    assert bits_equal(out.contiguous(), ref_o)
    assert bool((big[:, 0] == 7.0).all()) and bool((big[:, T + 1:] == 7.0).all())
    assert bool((big[:, :, :32] == 7.0).all()) and bool((big[:, :, 32 + D:] == 7.0).all())


def test_attention_every_head_of_the_workload_equals_the_head_alone():
    # B = 32: every CTA runs about twelve tiles, including tiles whose last
    # row quadrants hold no output rows (816 = 6 x 128 + 48); each head of
    # the batched run must give the bits of the same head run alone, where
    # every CTA runs one tile
    q, k, v = inputs.attention(32)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    o = binding.bi_attention(qg, kg, vg, 1.0 / 16)
    assert bool(torch.isfinite(o).all())
    for h in range(0, 256, 5):
        assert bits_equal(binding.bi_attention(qg[h:h + 1], kg[h:h + 1], vg[h:h + 1], 1.0 / 16), o[h:h + 1]), h
    assert bits_equal(binding.bi_attention(qg, kg, vg, 1.0 / 16), o)


def test_attention_workload_sampled_heads():
    # the timed shape at B = 32: Q, K, V [256, 816, 256]; heads 0, 100 and 255
    # against the oracle, head 0 bit-equal to the B = 1 run
    q, k, v = inputs.attention(32)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    o = binding.bi_attention(qg, kg, vg, 1.0 / 16)
    for h in (0, 100, 255):
        ref, absum, smax = oracle.attention(q[h:h + 1], k[h:h + 1], v[h:h + 1], 1.0 / 16)
        check_attention(o[h:h + 1], ref, absum, smax, 816, f"B=32 head {h}")
    o1 = binding.bi_attention(qg[:8], kg[:8], vg[:8], 1.0 / 16)
    assert bits_equal(o1, o[:8])


# ---------------------------------------------------------------------------
# Key ranges longer than 2048: fixed 2048-key splits merged in split order
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(2, 130, 2049), (1, 300, 4096), (3, 64, 5000), (1, 40, 9000)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_attention_split_key_range_matches_oracle(shape, out_dtype):
    L, Tq, Tk = shape
    q, k, v = _qkv(L, Tq, Tk, 60)
    ref, absum, smax = oracle.attention(q, k, v, 1.0 / 16)
    o = binding.bi_attention_ws(q.cuda(), k.cuda(), v.cuda(), 1.0 / 16, out_dtype=out_dtype)
    check_attention(o, ref, absum, smax, Tk, f"split attention {shape} -> {out_dtype}")


def test_attention_split_invariances():
    # heads alone vs in a batch, query chunks, run to run, and a caller-given
    # workspace full of garbage: all the same bits
    L, Tq, Tk = 6, 260, 4500
    q, k, v = _qkv(L, Tq, Tk, 61)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    full = binding.bi_attention_ws(qg, kg, vg, 1.0 / 16)
    for h in (0, 3, 5):
        assert bits_equal(binding.bi_attention_ws(qg[h:h + 1], kg[h:h + 1], vg[h:h + 1], 1.0 / 16),
                          full[h:h + 1]), h
    for a, b in ((0, 1), (100, 260), (127, 131)):
        assert bits_equal(binding.bi_attention_ws(qg[:, a:b].contiguous(), kg, vg, 1.0 / 16), full[:, a:b])
    ws = torch.full((binding.bi_attention_workspace_bytes(L, Tq, Tk),), 0xFF, dtype=torch.uint8, device="cuda")
    assert bits_equal(binding.bi_attention_ws(qg, kg, vg, 1.0 / 16, workspace=ws), full)
    ref, absum, smax = oracle.attention(q[:2], k[:2], v[:2], 1.0 / 16)
    check_attention(full[:2], ref, absum, smax, Tk, "split attention heads 0-1")


def test_attention_split_rescales_across_splits():
    # scores rising along the keys: the maximum moves in every block and the
    # later splits dominate the merge
    L, Tq, Tk = 1, 70, 5000
    q = (torch.ones(L, Tq, D) * 0.25).to(torch.bfloat16)
    ramp = torch.arange(Tk, dtype=torch.float32) / 40.0
    k = (ramp[None, :, None] * torch.ones(L, Tk, D)).to(torch.bfloat16)
    k[:, :, 1::2] *= -0.5
    v = inputs.normal_bf16((L, Tk, D), 1.0, 62)
    ref, absum, smax = oracle.attention(q, k, v, 0.1)
    o = binding.bi_attention_ws(q.cuda(), k.cuda(), v.cuda(), 0.1)
    check_attention(o, ref, absum, smax, Tk, "split attention, rising scores")


def test_attention_unsplit_range_is_the_same_with_or_without_workspace():
    q, k, v = _qkv(2, 200, 2048, 63)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    assert binding.bi_attention_workspace_bytes(2, 200, 2048) == 0
    assert bits_equal(binding.bi_attention_ws(qg, kg, vg, 0.0625), binding.bi_attention(qg, kg, vg, 0.0625))
    with pytest.raises(binding.BiError) as ei:
        binding.bi_attention(qg, torch.cat([kg, kg[:, :1]], 1), torch.cat([vg, vg[:, :1]], 1), 0.0625)
    assert ei.value.status == binding.BI_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# Head dimensions 64 and 128: the same kernel built for a narrower D (fewer
# tensor-core steps per score, a narrower O), held to the same bar
# ---------------------------------------------------------------------------

SMALL_D = [64, 128]


@pytest.mark.parametrize("d", SMALL_D)
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 129, 64), (3, 200, 333), (2, 816, 816)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_attention_head_dims_match_oracle(d, shape, out_dtype):
    L, Tq, Tk = shape
    q, k, v = _qkv(L, Tq, Tk, 70, d)
    scale = d ** -0.5
    ref, absum, smax = oracle.attention(q, k, v, scale)
    o = binding.bi_attention(q.cuda(), k.cuda(), v.cuda(), scale, out_dtype=out_dtype)
    check_attention(o, ref, absum, smax, Tk, f"attention D={d} {shape} -> {out_dtype}")


@pytest.mark.parametrize("d", SMALL_D)
def test_attention_head_dims_rescale(d):
    L, Tq, Tk = 2, 130, 700
    q = (torch.ones(L, Tq, d) * 0.5).to(torch.bfloat16)
    ramp = torch.arange(Tk, dtype=torch.float32) / 10.0
    k = (ramp[None, :, None] * torch.ones(L, Tk, d)).to(torch.bfloat16)
    k[:, :, 1::2] *= -0.5
    v = inputs.normal_bf16((L, Tk, d), 1.0, 71)
    ref, absum, smax = oracle.attention(q, k, v, 0.2)
    o = binding.bi_attention(q.cuda(), k.cuda(), v.cuda(), 0.2)
    check_attention(o, ref, absum, smax, Tk, f"rescale D={d}")


@pytest.mark.parametrize("d", SMALL_D)
def test_attention_head_dims_invariances(d):
    # heads alone vs in a batch of 40 (more tiles than SMs), query chunks, run to run
    q, k, v = _qkv(40, 300, 450, 72, d)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    full = binding.bi_attention(qg, kg, vg, d ** -0.5)
    for h in (0, 17, 39):
        assert bits_equal(binding.bi_attention(qg[h:h + 1], kg[h:h + 1], vg[h:h + 1], d ** -0.5), full[h:h + 1]), h
    for a, b in ((0, 1), (127, 129), (200, 300)):
        assert bits_equal(binding.bi_attention(qg[:, a:b].contiguous(), kg, vg, d ** -0.5), full[:, a:b]), (a, b)
    assert bits_equal(binding.bi_attention(qg, kg, vg, d ** -0.5), full)
    ref, absum, smax = oracle.attention(q[38:40], k[38:40], v[38:40], d ** -0.5)
    check_attention(full[38:40], ref, absum, smax, 450, f"D={d} heads 38-39")


@pytest.mark.parametrize("d", SMALL_D)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_attention_head_dims_strided(d, out_dtype):
    # packed [L, T, 3, d] operands and a padded output: the bits of contiguous ones
    L, T = 3, 250
    g = inputs.normal_bf16((L, T, 3, d), 1.0, 73).cuda()
    q, k, v = g[:, :, 0], g[:, :, 1], g[:, :, 2]
    ref_o = binding.bi_attention(q.contiguous(), k.contiguous(), v.contiguous(), 0.125, out_dtype=out_dtype)
    big = torch.full((L, T + 3, d + 64), 7.0, device="cuda", dtype=out_dtype)
    out = big[:, 1:T + 1, 32:32 + d]
    binding.bi_attention(q, k, v, 0.125, out=out)
    assert bits_equal(out.contiguous(), ref_o)
    assert bool((big[:, 0] == 7.0).all()) and bool((big[:, T + 1:] == 7.0).all())
    assert bool((big[:, :, :32] == 7.0).all()) and bool((big[:, :, 32 + d:] == 7.0).all())


@pytest.mark.parametrize("d", SMALL_D)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_attention_head_dims_split(d, out_dtype):
    L, Tq, Tk = 3, 140, 4500
    q, k, v = _qkv(L, Tq, Tk, 74, d)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    assert binding.bi_attention_workspace_bytes(L, Tq, Tk, d) == 3 * L * Tq * (d + 2) * 4
    full = binding.bi_attention_ws(qg, kg, vg, d ** -0.5, out_dtype=out_dtype)
    ref, absum, smax = oracle.attention(q, k, v, d ** -0.5)
    check_attention(full, ref, absum, smax, Tk, f"split D={d} -> {out_dtype}")
    assert bits_equal(binding.bi_attention_ws(qg[1:2], kg[1:2], vg[1:2], d ** -0.5, out_dtype=out_dtype), full[1:2])
    assert bits_equal(binding.bi_attention_ws(qg[:, 130:].contiguous(), kg, vg, d ** -0.5, out_dtype=out_dtype),
                      full[:, 130:])


@pytest.mark.parametrize("d", SMALL_D)
def test_attention_two_tile_kernel_equals_one_tile_kernel(d):
    # Heads of 64 or 128 with two or more query tiles run two tiles per CTA
    # (pairs of tiles, then the odd last tile of each head alone: 100 heads x
    # 5 tiles = 300 units, more than one per SM); a 128-row chunk on its own
    # runs the one-tile kernel.  Every row has the same bits in both, also
    # when the running maximum rises by more than 2^8 between key blocks.
    L, Tq, Tk = 100, 640, 700
    q, k, v = _qkv(L, Tq, Tk, 75, d)
    k[:, 300:310] *= 6.0  # scores rise sharply at the third key block
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    for out_dtype in (torch.float32, torch.bfloat16):
        full = binding.bi_attention(qg, kg, vg, d ** -0.5, out_dtype=out_dtype)
        for c in range(Tq // 128):
            part = binding.bi_attention(qg[:, 128 * c:128 * (c + 1)].contiguous(), kg, vg, d ** -0.5,
                                        out_dtype=out_dtype)
            assert bits_equal(part, full[:, 128 * c:128 * (c + 1)]), (out_dtype, c)
    ref, absum, smax = oracle.attention(q[98:100], k[98:100], v[98:100], d ** -0.5)
    check_attention(full[98:100], ref, absum, smax, Tk, f"two-tile D={d}")
