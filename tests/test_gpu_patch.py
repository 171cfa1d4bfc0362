"""GPU parity of the packed patch-embedding convolution (bi_conv2d_patch_packed)
against the fp64 oracle's direct convolution ("Batch-Invariant VLAs", section
"Replacing nn.Conv2d": the patch embedding as a per-sample product of the
unfolded patches and the flattened filter), sample-0 bit invariance across the
batch, and isolation of each output position from every pixel outside its own
window."""
from __future__ import annotations

import pytest
import torch

import oracle
from invariant_gemm_bi_gb300 import binding, inputs
from tests.gpu_helpers import bits_equal, check_tolerance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load()
    yield
    assert binding.bi_device_status() == binding.BI_OK


def _conv(x, w, bias, out_dtype=torch.bfloat16):
    packed = binding.bi_conv_pack_weight(w.cuda())
    return binding.bi_conv2d_patch_packed(x.cuda(), packed, None if bias is None else bias.cuda(),
                                          out_dtype=out_dtype)


def test_packed_filter_layout_is_the_padded_filter():
    # [Co][ci][kh < KHp][kw < 16], zeros where kh >= KH or kw >= KW
    Co, C, KH, KW = 5, 3, 6, 7
    w = inputs.normal_bf16((Co, C, KH, KW), 1.0, 40)
    packed = binding.bi_conv_pack_weight(w.cuda())
    torch.cuda.synchronize()
    KHp = (KH + 3) // 4 * 4
    expect = torch.zeros((Co, C, KHp, 16), dtype=torch.bfloat16)
    expect[:, :, :KH, :KW] = w
    got = packed.buffer[: Co * C * KHp * 16 * 2].cpu().view(torch.bfloat16).view(Co, C, KHp, 16)
    assert bits_equal(got, expect)
    assert packed.desc.Kp == C * KHp * 16


def test_siglip_patch_embed_matches_oracle_and_is_sample0_invariant():
    # images [B,3,224,224] ~U(-1,1), weight [1152,3,14,14] ~N(0,0.02), bias [1152]
    B_max = max(inputs.PATCH_EMBED_B)
    x, w, bias = inputs.patch_embed(B_max)
    xg, bg = x.cuda(), bias.cuda()
    packed = binding.bi_conv_pack_weight(w.cuda())
    y_full = binding.bi_conv2d_patch_packed(xg, packed, bg)
    for b in (0, B_max - 1):
        ref, absum = oracle.conv2d(x[b:b + 1], w, bias, 14, 0, 1, 1)
        check_tolerance(y_full[b:b + 1], ref, absum, f"packed conv sample {b}")
    for B in inputs.PATCH_EMBED_B:
        y = binding.bi_conv2d_patch_packed(xg[:B], packed, bg)
        assert bits_equal(y[:1], y_full[:1]), f"sample 0 differs at B={B}"
        assert bits_equal(y, y_full[:B])
    assert bits_equal(binding.bi_conv2d_patch_packed(xg, packed, bg), y_full)
    # fp32 output agrees with the oracle too
    y32 = binding.bi_conv2d_patch_packed(xg[:2], packed, bg, out_dtype=torch.float32)
    ref, absum = oracle.conv2d(x[:2], w, bias, 14, 0, 1, 1)
    check_tolerance(y32, ref, absum, "packed conv fp32")


PATCH_CASES = [
    # B, C, H, W, Co, KH, KW, out dtype, bias dtype (None: no bias)
    (2, 3, 224, 224, 768, 16, 16, torch.bfloat16, torch.bfloat16),  # 14 x 14 patches: 126-row tiles
    (3, 1, 40, 48, 130, 8, 8, torch.float32, torch.float32),         # one channel, ragged Co
    (2, 4, 30, 56, 40, 7, 7, torch.float32, torch.bfloat16),         # odd KW, leftover image rows
    (1, 2, 33, 64, 16, 5, 3, torch.float32, None),                   # leftover rows and columns
    (2, 3, 32, 256, 64, 2, 2, torch.bfloat16, torch.float32),        # widest image, 128 patches a row
    (1, 3, 64, 64, 300, 16, 16, torch.bfloat16, None),
    (1, 3, 224, 224, 1153, 14, 14, torch.float32, torch.bfloat16),  # 6 whole 192-channel tiles + 1 channel
]


@pytest.mark.parametrize("case", PATCH_CASES)
def test_patch_cases_match_oracle(case):
    B, C, H, W, Co, KH, KW, od, bd = case
    x = inputs.uniform_bf16((B, C, H, W), -1, 1, 41)
    w = inputs.normal_bf16((Co, C, KH, KW), 0.1, 42)
    bias = None if bd is None else inputs.normal_bf16((Co,), 0.1, 43)  # bf16 values (the oracle's input)
    ref, absum = oracle.conv2d(x, w, bias, (KH, KW), 0, 1, 1)
    kb = None if bias is None else bias.to(bd)                          # same values in the bias dtype under test
    y = _conv(x, w, kb, od)
    check_tolerance(y, ref, absum, f"packed conv {case}")
    y0 = _conv(x[:1], w, kb, od)
    assert bits_equal(y0, y[:1])


def test_each_position_reads_only_its_own_window():
    # Non-finite pixels in the neighbouring windows (right, below, and in the
    # columns / rows past the last whole patch) leave position (0, 0) unchanged.
    C, H, W, Co, KH, KW = 3, 30, 48, 64, 7, 6   # Ho = 4 (2 rows left over), Wo = 8
    x = inputs.uniform_bf16((1, C, H, W), -1, 1, 44)
    w = inputs.normal_bf16((Co, C, KH, KW), 0.1, 45)
    clean = _conv(x, w, None, torch.float32)
    dirty = x.clone()
    dirty[0, 1, 0, KW] = float("inf")        # right neighbour's first column
    dirty[0, 2, 3, KW + 1] = float("nan")
    dirty[0, 0, KH, 2] = float("-inf")       # window below
    dirty[0, 1, 28:, :] = float("nan")       # rows past the last whole patch
    y = _conv(dirty, w, None, torch.float32)
    assert bits_equal(y[:, :, 0, 0], clean[:, :, 0, 0])
    assert torch.isfinite(y[:, :, 0, 0]).all()


def test_distractor_samples_do_not_touch_sample0():
    x, w, bias = inputs.patch_embed(3)
    packed = binding.bi_conv_pack_weight(w.cuda())
    alone = binding.bi_conv2d_patch_packed(x[:1].cuda(), packed, bias.cuda())
    for fill in (float("nan"), float("inf"), 2.0 ** 100):
        d = x.clone()
        d[1:] = fill
        y = binding.bi_conv2d_patch_packed(d.cuda(), packed, bias.cuda())
        assert bits_equal(y[:1], alone)


@pytest.mark.parametrize("case", [c for c in PATCH_CASES if c[6] == 16 or (c[6] == 14 and c[5] % 2 == 0)] +
                         [(32, 3, 224, 224, 1152, 14, 14, torch.bfloat16, torch.bfloat16),
                          (2, 3, 45, 64, 200, 9, 16, torch.float32, None)])  # KH = 9: a lone kernel row per channel
def test_plain_filter_entry_point_equals_packed(case):
    # bi_conv2d_patch on non-overlapping 16-wide patches, or 14-wide ones with
    # an even patch height, builds the packed filter layout in shared memory
    # from w itself: the bits of the packed path.
    B, C, H, W, Co, KH, KW, od, bd = case
    x = inputs.uniform_bf16((B, C, H, W), -1, 1, 46)
    w = inputs.normal_bf16((Co, C, KH, KW), 0.05, 47)
    bias = None if bd is None else inputs.normal_bf16((Co,), 0.1, 48).to(bd).cuda()
    xg, wg = x.cuda(), w.cuda()
    packed = binding.bi_conv2d_patch_packed(xg, binding.bi_conv_pack_weight(wg), bias, out_dtype=od)
    plain = binding.bi_conv2d_patch(xg, wg, bias, stride=(KH, KW), out_dtype=od)
    assert bits_equal(plain, packed)
    for b in (1, B):
        assert bits_equal(binding.bi_conv2d_patch(xg[:b], wg, bias, stride=(KH, KW), out_dtype=od), packed[:b])


def test_plain_filter_entry_point_misaligned_image_takes_the_general_kernel():
    # An image view that is not 16-byte aligned cannot be copied by rows: the
    # general kernel runs (the unfold order in steps of 16), within the
    # oracle's bound.
    B, C, H, W, Co, KH, KW = 2, 3, 32, 48, 40, 8, 8
    x = inputs.uniform_bf16((B, C, H, W), -1, 1, 49)
    w = inputs.normal_bf16((Co, C, KH, KW), 0.1, 50)
    buf = torch.zeros(x.numel() + 1, dtype=torch.bfloat16, device="cuda")
    xs = buf[1:].view(B, C, H, W)
    xs.copy_(x.cuda())
    y = binding.bi_conv2d_patch(xs, w.cuda(), None, stride=(KH, KW), out_dtype=torch.float32)
    ref, absum = oracle.conv2d(x, w, None, (KH, KW), 0, 1, 1)
    check_tolerance(y, ref, absum, "misaligned image")
