"""The five workloads at their full sizes, in the launch configuration the
benchmark times: oracle parity on sampled rows (every row where the oracle
finishes in seconds), row 0 / sample 0 / head 0 bit-equal across the whole
M (or B) sweep, and run-to-run bit equality."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_gemm_bi_gb300 import binding, inputs
from tests.gpu_helpers import bits_equal, check_tolerance

pytestmark = pytest.mark.gpu


def _sample_rows(M: int, n_extra: int, seed: int) -> list[int]:
    rng = np.random.default_rng(seed)
    rows = {0, M - 1}
    rows.update(int(r) for r in rng.integers(0, M, n_extra))
    return sorted(rows)


def test_llm_addmm_sweep():
    # x [M,4096] ~N(0,1), W [4096,14336] ~N(0,0.02), bias ~N(0,0.01), bf16 out
    M_max = max(inputs.LLM_ADDMM_M)
    x, w, bias = inputs.llm_addmm(M_max)
    xg, wg, bg = x.cuda(), w.cuda(), bias.cuda()
    row0 = None
    full = binding.bi_addmm(bg, xg, wg)
    check_rows = _sample_rows(M_max, 14, 0)
    ref, absum = oracle.mm(x, w, bias=bias, rows=check_rows)
    check_tolerance(full[check_rows], ref, absum, "addmm M=8192 sampled rows")
    for M in inputs.LLM_ADDMM_M:
        c = binding.bi_addmm(bg, xg[:M], wg)
        if row0 is None:
            row0 = c[:1].clone()
        assert bits_equal(c[:1], row0), f"row 0 differs at M={M}"
        assert bits_equal(c[M - 1:M], full[M - 1:M]), f"row M-1 differs at M={M}"
    check_tolerance(row0, ref[:1], absum[:1], "addmm row 0")
    # run to run
    assert bits_equal(binding.bi_addmm(bg, xg, wg), full)


def test_llm_addmm_packed_weight_equals_plain_full_size():
    # The benchmark times the plain [4096,14336] weight; its packed form
    # (bi_pack_weight) must give the same bits at every M of the sweep,
    # including the full M = 8192 launch.
    M_max = max(inputs.LLM_ADDMM_M)
    x, w, bias = inputs.llm_addmm(M_max)
    xg, wg, bg = x.cuda(), w.cuda(), bias.cuda()
    wp = binding.bi_pack_weight(wg)
    for M in inputs.LLM_ADDMM_M:
        plain = binding.bi_addmm(bg, xg[:M], wg)
        packed = binding.bi_addmm_packed(bg, xg[:M], wp)
        assert bits_equal(plain, packed), f"packed and plain weights differ at M={M}"
        del plain, packed


def test_square_mm_sweep():
    # A [M,8192] ~N(0,1), W [8192,8192] ~N(0,0.01), fp32 out
    M_max = max(inputs.SQUARE_MM_M)
    a, w = inputs.square_mm(M_max)
    ag, wg = a.cuda(), w.cuda()
    full = binding.bi_mm(ag, wg)
    check_rows = _sample_rows(M_max, 10, 1)
    ref, absum = oracle.mm(a, w, rows=check_rows)
    check_tolerance(full[check_rows], ref, absum, "square mm M=16384 sampled rows")
    for M in inputs.SQUARE_MM_M:
        c = binding.bi_mm(ag[:M], wg)
        assert bits_equal(c[:1], full[:1]), f"row 0 differs at M={M}"
        assert bits_equal(c[M - 1:M], full[M - 1:M]), f"row M-1 differs at M={M}"
        del c
    assert bits_equal(binding.bi_mm(ag, wg), full)


def _attention_gpu(q, k, v):
    s = binding.bi_bmm(q, k.transpose(1, 2), alpha=1.0 / 16)          # [L,T,T] fp32
    p = binding.bi_softmax_lastdim(s.view(-1, s.shape[-1])).view(s.shape)  # bf16
    o = binding.bi_bmm(p, v)                                          # [L,T,D] fp32
    return s, p, o


def test_attention_stagewise_parity_and_head0_invariance():
    # Q, K, V [B*8, 816, 256] ~N(0,1); S = Q K^T / 16; P = softmax(S) -> bf16; O = P V
    B_max = max(inputs.ATTENTION_B)
    q, k, v = inputs.attention(B_max)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    s_full, p_full, o_full = _attention_gpu(qg, kg, vg)
    # stage-wise parity on heads 0 and the last one, each stage on its own GPU inputs
    for h in (0, q.shape[0] - 1):
        ref_s, abs_s = oracle.bmm(q[h:h + 1], k[h:h + 1].transpose(1, 2), alpha=1.0 / 16)
        check_tolerance(s_full[h:h + 1], ref_s, abs_s, f"S head {h}")
        ref_p = oracle.softmax_rows(s_full[h].cpu())
        pg = p_full[h].cpu().double().numpy()
        assert np.all(np.abs(pg - ref_p) <= 2.0 ** -8 * ref_p + 1e-4 * ref_p + 1e-30), f"P head {h}"
        ref_o, abs_o = oracle.bmm(p_full[h:h + 1].cpu(), v[h:h + 1])
        check_tolerance(o_full[h:h + 1], ref_o, abs_o, f"O head {h}")
    for B in inputs.ATTENTION_B:
        L = B * 8
        s, p, o = _attention_gpu(qg[:L], kg[:L], vg[:L])
        assert bits_equal(s[:1], s_full[:1]) and bits_equal(p[:1], p_full[:1])
        assert bits_equal(o[:1], o_full[:1]), f"head 0 differs at B={B}"
    s2, p2, o2 = _attention_gpu(qg, kg, vg)
    assert bits_equal(o2, o_full) and bits_equal(p2, p_full)


def test_patch_embed_conv_parity_and_sample0_invariance():
    # images [B,3,224,224] ~U(-1,1), weight [1152,3,14,14] ~N(0,0.02), bias [1152],
    # stride 14 -> [B,1152,16,16] bf16
    B_max = max(inputs.PATCH_EMBED_B)
    x, w, bias = inputs.patch_embed(B_max)
    xg, wg, bg = x.cuda(), w.cuda(), bias.cuda()
    y_full = binding.bi_conv2d_patch(xg, wg, bg, stride=14)
    for b in (0, B_max - 1):
        ref, absum = oracle.conv2d(x[b:b + 1], w, bias, 14, 0, 1, 1)
        check_tolerance(y_full[b:b + 1], ref, absum, f"conv sample {b}")
    for B in inputs.PATCH_EMBED_B:
        y = binding.bi_conv2d_patch(xg[:B], wg, bg, stride=14)
        assert bits_equal(y[:1], y_full[:1]), f"sample 0 differs at B={B}"
        assert bits_equal(y, y_full[:B])
    assert bits_equal(binding.bi_conv2d_patch(xg, wg, bg, stride=14), y_full)


CONV_CASES = [
    # B, C, H, W, Co, KH, KW, stride, padding, dilation, groups, out dtype
    (2, 4, 9, 11, 6, 3, 3, 1, 1, 1, 1, torch.float32),
    (1, 4, 10, 10, 4, 3, 2, (2, 1), (1, 0), (2, 1), 2, torch.bfloat16),
    (3, 6, 17, 15, 9, 2, 3, 2, 2, 1, 3, torch.float32),
    (2, 3, 28, 28, 200, 14, 14, 14, 0, 1, 1, torch.bfloat16),
    (1, 16, 40, 40, 130, 3, 3, 1, 1, 1, 1, torch.float32),
    # non-overlapping patches (the row-wise patch loader): grouped, partial tile,
    # rows not 16-byte aligned, K not a multiple of 4
    (2, 4, 30, 45, 6, 5, 3, (5, 3), 0, 1, 2, torch.float32),
    (3, 3, 64, 48, 130, 8, 8, 8, 0, 1, 1, torch.bfloat16),
    (2, 3, 70, 70, 40, 7, 7, 7, 0, 1, 1, torch.float32),
    # pair path with image columns past the last patch (W = 48, Wo*KW = 42)
    (2, 2, 20, 48, 24, 4, 6, (4, 6), 0, 1, 1, torch.float32),
    (1, 3, 32, 40, 16, 4, 4, 4, 0, 1, 1, torch.bfloat16),
]


@pytest.mark.parametrize("case", CONV_CASES)
def test_general_conv_matches_oracle(case):
    B, C, H, W, Co, KH, KW, st, pd, dl, gr, od = case
    x = inputs.uniform_bf16((B, C, H, W), -1, 1, 50)
    w = inputs.normal_bf16((Co, C // gr, KH, KW), 0.2, 51)
    bias = inputs.normal_bf16((Co,), 0.1, 52)
    ref, absum = oracle.conv2d(x, w, bias, st, pd, dl, gr)
    y = binding.bi_conv2d_patch(x.cuda(), w.cuda(), bias.cuda(), st, pd, dl, gr, out_dtype=od)
    check_tolerance(y, ref, absum, f"conv {case}")
    y0 = binding.bi_conv2d_patch(x[:1].cuda(), w.cuda(), bias.cuda(), st, pd, dl, gr, out_dtype=od)
    assert bits_equal(y0, y[:1])


def test_softmax_matches_oracle_both_paths_and_ragged_rows():
    for N in (1, 7, 816, 1024, 1025, 3000):
        s = (inputs.normal_bf16((37, N), 3.0, 60 + N).float())
        ref = oracle.softmax_rows(s)
        for od in (torch.bfloat16, torch.float32):
            p = binding.bi_softmax_lastdim(s.cuda(), out_dtype=od).cpu().double().numpy()
            tol = (2.0 ** -8 if od == torch.bfloat16 else 0.0) * ref + 1e-4 * ref + 1e-38
            assert np.all(np.abs(p - ref) <= tol), (N, od)
        one = binding.bi_softmax_lastdim(s[:1].cuda())
        many = binding.bi_softmax_lastdim(s.cuda())
        assert bits_equal(one, many[:1])


def test_bmm_bf16_output_and_batch_strides():
    L, M, K, N = 5, 100, 136, 72
    a = inputs.normal_bf16((L, M, K), 1.0, 70)
    b = inputs.normal_bf16((L, K, N), 0.1, 71)
    ref, absum = oracle.bmm(a, b, alpha=0.5)
    c = binding.bi_bmm(a.cuda(), b.cuda(), alpha=0.5, out_dtype=torch.bfloat16)
    check_tolerance(c, ref, absum, "bmm bf16")
    c1 = binding.bi_bmm(a[2:3].cuda(), b[2:3].cuda(), alpha=0.5, out_dtype=torch.bfloat16)
    assert bits_equal(c1, c[2:3])


def test_softmax_alignment_does_not_change_bits():
    # 16-byte rows take the vector path, shifted rows the scalar one: same order, same bits
    s = inputs.normal_bf16((64, 816), 2.0, 61).float().cuda()
    store = torch.zeros(64, 820, device="cuda")
    shifted = store[:, 1:817]
    shifted.copy_(s)
    for od in (torch.bfloat16, torch.float32):
        a = binding.bi_softmax_lastdim(s, out_dtype=od)
        b = binding.bi_softmax_lastdim(shifted, out_dtype=od)
        assert bits_equal(a, b)
