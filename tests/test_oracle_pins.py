"""Pins for the fp64 CPU oracle: checks against values the pages print, closed
forms, exact rational arithmetic, integer arithmetic and independent library
routines -- never against the oracle itself or the CUDA path.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong rounding) fails it.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from invariant_gemm_bi_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(t: torch.Tensor):
    """Exact rationals of a bf16/fp32 tensor's values (nested lists)."""
    return [[Fraction(float(v)) for v in row] for row in t.to(torch.float64).tolist()]


# ---------------------------------------------------------------------------
# Summation order (values printed on the pages)
# ---------------------------------------------------------------------------

def _read_nonassoc():
    rows = []
    with open(os.path.join(GOLDEN, "nonassociativity.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                typ, order, a, b, c, exp = line.split()
                rows.append((typ, order, float(a), float(b), float(c), float(exp)))
    return rows


@pytest.mark.parametrize("row", _read_nonassoc())
def test_sequential_sum_helpers_match_printed_values(row):
    typ, order, a, b, c, expected = row
    # A sequential sum from zero evaluates (((0 + x0) + x1) + x2):
    #   left  = (a + b) + c   -> order [a, b, c]
    #   right = a + (b + c)   -> compute (b + c) first: order [b, c, a]
    seq = [a, b, c] if order == "left" else [b, c, a]
    got = oracle.sum_seq_f32(seq) if typ == "f32" else oracle.sum_seq_f64(seq)
    assert got == expected


def test_mm_accumulates_in_ascending_k_in_double():
    # products [1, 2^60, -2^60]: ascending-k double sum gives (1 + 2^60) - 2^60 = 0,
    # any other grouping of the last two terms first gives 1.
    a = torch.tensor([[1.0, 2.0 ** 30, -(2.0 ** 30)]], dtype=torch.bfloat16)
    b = torch.tensor([[1.0], [2.0 ** 30], [2.0 ** 30]], dtype=torch.bfloat16)
    c, _ = oracle.mm(a, b)
    assert c[0, 0] == 0.0
    # reversed k order gives 1
    c2, _ = oracle.mm(a.flip(1).contiguous(), b.flip(0).contiguous())
    assert c2[0, 0] == 1.0
    # products [1, 2^24, -2^24]: exact in double (=1), lost in a float sum (=0)
    a = torch.tensor([[1.0, 2.0 ** 12, -(2.0 ** 12)]], dtype=torch.bfloat16)
    b = torch.tensor([[1.0], [2.0 ** 12], [2.0 ** 12]], dtype=torch.bfloat16)
    c, _ = oracle.mm(a, b)
    assert c[0, 0] == 1.0


# ---------------------------------------------------------------------------
# mm / addmm / bmm
# ---------------------------------------------------------------------------

def _exact_mm(a, b, bias, alpha):
    A, B = _frac(a), _frac(b)
    M, K, N = len(A), len(B), len(B[0])
    bv = [Fraction(float(v)) for v in bias.to(torch.float64).tolist()] if bias is not None else None
    al = Fraction(alpha)
    out, outabs = [], []
    for m in range(M):
        r, ra = [], []
        for n in range(N):
            terms = [A[m][k] * B[k][n] for k in range(K)]
            v = al * sum(terms, Fraction(0))
            va = abs(al) * sum((abs(t) for t in terms), Fraction(0))
            if bv is not None:
                v += bv[n]
                va += abs(bv[n])
            r.append(v)
            ra.append(va)
        out.append(r)
        outabs.append(ra)
    return out, outabs


@pytest.mark.parametrize("seed", range(12))
def test_mm_against_exact_rationals(seed):
    g = torch.Generator().manual_seed(100 + seed)
    M, N, K = (int(v) for v in torch.randint(1, 6, (3,), generator=g))
    a = (torch.randn(M, K, generator=g) * 3).to(torch.bfloat16)
    b = (torch.randn(K, N, generator=g) * 0.5).to(torch.bfloat16)
    bias = (torch.randn(N, generator=g)).to(torch.bfloat16) if seed % 2 else None
    alpha = [1.0, 0.0625, 3.0][seed % 3]
    # strided views: a transposed operand must give the same numbers
    if seed % 4 == 1:
        a = a.t().contiguous().t()
    if seed % 4 == 2:
        b = b.t().contiguous().t()
    c, absum = oracle.mm(a, b, bias=bias, alpha=alpha)
    ex, exabs = _exact_mm(a, b, bias, alpha)
    for m in range(M):
        for n in range(N):
            # fp64 sum of <= 6 exact products: error <= 6 * 2^-53 * sum|terms|
            assert abs(Fraction(c[m, n]) - ex[m][n]) <= Fraction(6, 2 ** 53) * exabs[m][n]
            assert abs(Fraction(absum[m, n]) - exabs[m][n]) <= Fraction(6, 2 ** 53) * exabs[m][n]


def test_mm_identity_permutation_onehot_exact():
    a = inputs.normal_bf16((7, 16), 1.0, 3)
    eye = torch.eye(16, dtype=torch.bfloat16)
    c, _ = oracle.mm(a, eye)
    assert np.array_equal(c, a.to(torch.float64).numpy())
    perm = torch.randperm(16, generator=torch.Generator().manual_seed(5))
    P = eye[:, perm]                      # column n of P is e_{perm[n]}
    c, _ = oracle.mm(a, P)
    assert np.array_equal(c, a[:, perm].to(torch.float64).numpy())
    onehot = torch.zeros(16, 3, dtype=torch.bfloat16)
    onehot[5, 0] = 1
    onehot[0, 1] = 2                      # power of two: still exact
    onehot[15, 2] = -1
    c, _ = oracle.mm(a, onehot)
    ref = torch.stack([a[:, 5], 2 * a[:, 0], -a[:, 15]], 1).to(torch.float64).numpy()
    assert np.array_equal(c, ref)


def test_mm_small_integers_exact_against_integer_matmul():
    a = inputs.small_int_bf16((9, 300), -4, 4, 11)
    b = inputs.small_int_bf16((300, 13), -4, 4, 12)
    bias = inputs.small_int_bf16((13,), -100, 100, 13)
    c, absum = oracle.mm(a, b, bias=bias)
    ai = a.to(torch.int64).numpy()
    bi = b.to(torch.int64).numpy()
    ref = ai @ bi + bias.to(torch.int64).numpy()[None, :]
    assert np.array_equal(c, ref.astype(np.float64))
    refabs = np.abs(ai)[:, :, None] * np.abs(bi)[None, :, :]
    assert np.array_equal(absum, refabs.sum(1) + np.abs(bias.to(torch.int64).numpy())[None, :])


def test_addmm_bias_only():
    a = torch.zeros(4, 32, dtype=torch.bfloat16)
    b = inputs.normal_bf16((32, 24), 1.0, 1)
    bias = inputs.normal_bf16((24,), 1.0, 2)
    c, _ = oracle.mm(a, b, bias=bias)
    assert np.array_equal(c, np.broadcast_to(bias.to(torch.float64).numpy(), (4, 24)))


def test_mm_sampled_rows_match_full_rows():
    a = inputs.normal_bf16((40, 64), 1.0, 0)
    b = inputs.normal_bf16((64, 48), 0.02, 1)
    full, fabs_ = oracle.mm(a, b)
    rows = [0, 39, 17, 3]
    part, pabs = oracle.mm(a, b, rows=rows)
    assert np.array_equal(part, full[rows]) and np.array_equal(pabs, fabs_[rows])


def test_bmm_against_exact_rationals_and_alpha():
    g = torch.Generator().manual_seed(7)
    L, M, K, N = 3, 4, 5, 3
    a = torch.randn(L, M, K, generator=g).to(torch.bfloat16)
    bt = torch.randn(L, N, K, generator=g).to(torch.bfloat16)
    b = bt.transpose(1, 2)                 # K-major view, as Q @ K^T
    c, absum = oracle.bmm(a, b, alpha=1.0 / 16)
    for l in range(L):
        ex, exabs = _exact_mm(a[l], b[l], None, 1.0 / 16)
        for m in range(M):
            for n in range(N):
                assert abs(Fraction(c[l, m, n]) - ex[m][n]) <= Fraction(5, 2 ** 53) * exabs[m][n]
    # alpha = 2^-4 only moves the exponent
    c1, _ = oracle.bmm(a, b, alpha=1.0)
    assert np.array_equal(c, c1 / 16)


# ---------------------------------------------------------------------------
# fp16 operands
# ---------------------------------------------------------------------------

def test_f16_decoding_matches_numpy_on_every_bit_pattern():
    # IEEE binary16 from its definition (oracle) vs numpy's float16 (independent)
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_bits_to_double(int(v)) for v in bits[::7]])
    exp = ref[::7]
    nan = np.isnan(exp)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], exp[~nan])
    for v in (0x0001, 0x03FF, 0x0400, 0x7BFF, 0x7C00, 0xFC00, 0x8000, 0x3C00):
        assert oracle.f16_bits_to_double(v) == float(np.uint16(v).view(np.float16))


@pytest.mark.parametrize("seed", range(6))
def test_mm_f16_against_exact_rationals(seed):
    g = torch.Generator().manual_seed(300 + seed)
    M, N, K = (int(v) for v in torch.randint(1, 6, (3,), generator=g))
    a = (torch.randn(M, K, generator=g) * 3).to(torch.float16)
    b = (torch.randn(K, N, generator=g) * 0.5).to(torch.float16)
    bias = (torch.randn(N, generator=g)).to(torch.float16) if seed % 2 else None
    alpha = [1.0, 0.0625, 3.0][seed % 3]
    if seed % 3 == 1:
        b = b.t().contiguous().t()
    c, absum = oracle.mm(a, b, bias=bias, alpha=alpha)
    ex, exabs = _exact_mm(a, b, bias, alpha)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(c[m, n]) - ex[m][n]) <= Fraction(6, 2 ** 53) * exabs[m][n]
            assert abs(Fraction(absum[m, n]) - exabs[m][n]) <= Fraction(6, 2 ** 53) * exabs[m][n]


def test_mm_and_bmm_f16_small_integers_and_fractions_exact():
    # fp16 holds 11 significant bits: values like 1023.5 or 2^-14 that bf16
    # cannot hold must arrive exactly
    g = torch.Generator().manual_seed(9)
    a = torch.randint(-1024, 1024, (5, 40), generator=g).to(torch.float16) + 0.5
    b = torch.randint(-8, 8, (40, 6), generator=g).to(torch.float16)
    c, _ = oracle.mm(a, b)
    ref = a.to(torch.float64).numpy() @ b.to(torch.float64).numpy()   # exact: small dyadics
    assert np.array_equal(c, ref)
    tiny = torch.full((1, 4), 2.0 ** -14, dtype=torch.float16)
    c, _ = oracle.mm(tiny, torch.ones(4, 1, dtype=torch.float16))
    assert c[0, 0] == 4 * 2.0 ** -14
    cb, _ = oracle.bmm(a[None], b[None], alpha=0.5)
    assert np.array_equal(cb[0], ref * 0.5)
    with pytest.raises(TypeError):
        oracle.mm(a, b.to(torch.bfloat16))


# ---------------------------------------------------------------------------
# Row reductions: RMSNorm, log-softmax, mean
# ---------------------------------------------------------------------------

def test_rmsnorm_closed_forms_and_invariances():
    # constant row 2^k, eps = 0: every output is exactly sign(x) (times w)
    x = torch.full((2, 12), -8.0)
    x[1] = 0.25
    y = oracle.rmsnorm_rows(x, eps=0.0)
    assert np.array_equal(y, np.sign(x.numpy()).astype(np.float64))
    # scaling x by a power of two changes nothing when eps = 0
    g = torch.Generator().manual_seed(21)
    x = torch.randn(5, 37, generator=g)
    assert np.array_equal(oracle.rmsnorm_rows(x, eps=0.0), oracle.rmsnorm_rows(x * 64, eps=0.0))
    # with w = 1 and eps = 0 the output's root mean square is 1
    y = oracle.rmsnorm_rows(x, eps=0.0)
    assert np.allclose(np.sqrt((y ** 2).mean(1)), 1.0, rtol=1e-14, atol=0)
    # the weight scales each column: one-hot weight keeps one column
    w = torch.zeros(37)
    w[5] = 2.0
    yw = oracle.rmsnorm_rows(x, w, eps=0.0)
    assert np.array_equal(yw[:, 5], 2 * y[:, 5]) and not yw[:, :5].any() and not yw[:, 6:].any()


def test_rmsnorm_matches_numpy_with_eps():
    g = torch.Generator().manual_seed(22)
    x = torch.randn(7, 300, generator=g).to(torch.bfloat16)
    w = (torch.rand(300, generator=g) + 0.5).to(torch.bfloat16)
    xd, wd = x.double().numpy(), w.double().numpy()
    ref = xd * (1.0 / np.sqrt((xd ** 2).mean(1, keepdims=True) + 1e-6)) * wd
    assert np.allclose(oracle.rmsnorm_rows(x, w, eps=1e-6), ref, rtol=1e-14, atol=0)


def test_log_softmax_closed_forms_and_library():
    # [0, log 3]: softmax is [1/4, 3/4]
    x = torch.tensor([[0.0, float(np.log(3.0))]], dtype=torch.float64).float()
    y = oracle.log_softmax_rows(x)
    xs = x.double().numpy()
    assert np.allclose(y, xs - np.log(np.exp(xs).sum()), rtol=0, atol=1e-15)
    # constant row: -log N
    y = oracle.log_softmax_rows(torch.full((1, 10), 3.5))
    assert np.allclose(y, -np.log(10.0), rtol=1e-15, atol=0)
    # exp(y) sums to one; shifting the row by a constant changes nothing
    g = torch.Generator().manual_seed(23)
    x = (torch.randn(6, 777, generator=g) * 4).to(torch.bfloat16).float()
    x[x.abs() < 2.0 ** -12] = 0.0              # so that x + 8 is exact in fp32
    y = oracle.log_softmax_rows(x)
    assert np.allclose(np.exp(y).sum(1), 1.0, rtol=1e-13)
    assert np.allclose(oracle.log_softmax_rows(x + 8.0), y, rtol=0, atol=1e-13)
    # against scipy's log_softmax (an independent library routine)
    special = pytest.importorskip("scipy.special")
    assert np.allclose(y, special.log_softmax(x.double().numpy(), axis=1), rtol=0, atol=1e-12)


def test_mean_rows_exact_cases_and_library():
    # small integers over a power-of-two length: exact
    g = torch.Generator().manual_seed(24)
    x = torch.randint(-50, 50, (4, 64), generator=g).float()
    m, ma = oracle.mean_rows(x)
    assert np.array_equal(m, x.double().numpy().sum(1) / 64)
    assert np.array_equal(ma, np.abs(x.double().numpy()).sum(1) / 64)
    # constant row
    assert oracle.mean_rows(torch.full((1, 7), -1.5, dtype=torch.bfloat16))[0][0] == -1.5
    # against numpy's mean
    x = torch.randn(5, 1001, generator=g).to(torch.float16)
    assert np.allclose(oracle.mean_rows(x)[0], x.double().numpy().mean(1), rtol=1e-13, atol=1e-16)


def _qkv(L, Tq, Tk, D, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn(shape, generator=g).to(dtype) for shape in ((L, Tq, D), (L, Tk, D), (L, Tk, D)))


def test_attention_special_cases():
    q, k, v = _qkv(2, 5, 7, 16, 31)
    # one key: every query row returns that key's value row, exactly
    o, ab, _ = oracle.attention(q, k[:, :1], v[:, :1], 0.25)
    assert np.array_equal(o, np.broadcast_to(v[:, :1].double().numpy(), o.shape))
    # identical keys: uniform weights, the mean of the value rows
    ksame = k[:, :1].expand(2, 7, 16).contiguous()
    o, _, _ = oracle.attention(q, ksame, v, 0.25)
    assert np.allclose(o, np.broadcast_to(v.double().numpy().mean(1, keepdims=True), o.shape), rtol=1e-14, atol=1e-15)
    # all-ones values: every output is 1
    o, _, _ = oracle.attention(q, k, torch.ones_like(v), 0.25)
    assert np.allclose(o, 1.0, rtol=1e-15, atol=0)
    # one dominant key (score 900 above the rest): its value row, exactly
    qd = torch.zeros(1, 3, 8)
    qd[0, :, 0] = 30.0
    kd = torch.zeros(1, 6, 8)
    kd[0, 4, 0] = 30.0
    vd = torch.randn(1, 6, 8, generator=torch.Generator().manual_seed(32))
    o, _, _ = oracle.attention(qd, kd, vd, 1.0)
    assert np.array_equal(o[0], np.broadcast_to(vd[0, 4].double().numpy(), (3, 8)))
    # two keys with a known score gap: weights 1/(1+e^-g) and e^-g/(1+e^-g)
    q2 = torch.tensor([[[1.0, 0.0]]])
    k2 = torch.tensor([[[2.0, 0.0], [0.5, 0.0]]])
    v2 = torch.tensor([[[1.0, 0.0], [0.0, 1.0]]])
    o, _, sm = oracle.attention(q2, k2, v2, 0.5)
    g = 0.5 * (2.0 - 0.5)
    assert np.allclose(o[0, 0], [1 / (1 + np.exp(-g)), np.exp(-g) / (1 + np.exp(-g))], rtol=1e-15, atol=0)
    assert sm[0, 0] == 1.0  # 0.5 * max(|1*2|, |1*0.5|)


def test_attention_invariances_and_library():
    q, k, v = _qkv(3, 9, 40, 24, 33)
    o, ab, sm = oracle.attention(q, k, v, 0.2)
    # permuting keys and values together changes nothing
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(34))
    op, _, _ = oracle.attention(q, k[:, perm], v[:, perm], 0.2)
    assert np.allclose(op, o, rtol=1e-13, atol=1e-15)
    # adding one vector u to every key shifts all scores of a row by q.u: no change
    u = torch.randn(24, generator=torch.Generator().manual_seed(35)).to(torch.bfloat16).float()
    os_, _, _ = oracle.attention(q.float(), k.float() + u, v, 0.2)
    assert np.allclose(os_, o, rtol=1e-12, atol=1e-14)
    # scale 2 equals doubling q (exact in binary floating point)
    o2, _, _ = oracle.attention(q, k, v, 0.4)
    o2b, _, _ = oracle.attention(q.float() * 2, k, v, 0.2)
    assert np.array_equal(o2, o2b)
    # each head and each query row stands alone
    o1, _, _ = oracle.attention(q[1:2, 4:5], k[1:2], v[1:2], 0.2)
    assert np.array_equal(o1[0, 0], o[1, 4])
    # absum bounds |o|, equals o for non-negative values; smax by brute force
    assert np.all(ab >= np.abs(o) - 1e-15)
    vp = v.abs()
    op_, abp, _ = oracle.attention(q, k, vp, 0.2)
    assert np.allclose(abp, op_, rtol=1e-15, atol=0)
    qd, kd = q.double().numpy(), k.double().numpy()
    assert np.allclose(sm, 0.2 * np.abs(qd[:, :, None, :] * kd[:, None, :, :]).sum(-1).max(-1), rtol=1e-14)
    # against scipy's softmax and numpy's matrix products (independent routines)
    special = pytest.importorskip("scipy.special")
    ref = special.softmax(0.2 * qd @ kd.transpose(0, 2, 1), axis=-1) @ v.double().numpy()
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# Rounding
# ---------------------------------------------------------------------------

def test_round_bf16_matches_torch_on_fp32_values():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 2 ** 31, (200000,), generator=g, dtype=torch.int64)
    bits = torch.cat([bits, (bits[:1000] & ~0xFFFF) | 0x8000])      # exact ties
    bits = torch.cat([bits, torch.arange(0, 70000, dtype=torch.int64)])  # subnormals
    sign = torch.randint(0, 2, bits.shape, generator=g) << 31
    u32 = ((bits | sign) & 0xFFFFFFFF).to(torch.int64)
    f = torch.from_numpy(u32.numpy().astype(np.uint32).view(np.float32))
    f = f[~torch.isnan(f)]
    ref = f.to(torch.bfloat16)
    got = oracle.round_bf16(f.to(torch.float64).numpy())
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def _rne_bf16_fraction(x: float) -> float:
    """Independent exact reference: round a double to 8 significant bits, RNE."""
    if x == 0:
        return x
    fx = Fraction(x)
    ax = abs(fx)
    e = math.frexp(x)[1]                 # |x| in [2^(e-1), 2^e)
    q_exp = max(e - 8, -133)             # bf16 quantum (subnormal floor 2^-133)
    q = Fraction(2) ** q_exp
    n = ax / q
    lo = math.floor(n)
    rem = n - lo
    r = lo + 1 if (rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1)) else lo
    val = r * q
    if val >= Fraction(2) ** 128:
        return math.copysign(math.inf, x)
    return math.copysign(float(val), x)


def test_round_bf16_double_inputs_against_exact_rationals():
    rng = np.random.default_rng(9)
    xs = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000),
                         rng.standard_normal(200) * 1e-39,
                         np.array([3.3895313892515355e38, 3.3961775292304135e38, 1.0 + 2 ** -8,
                                   1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -40])])
    got = oracle.round_bf16(xs).to(torch.float64).numpy()
    for x, gv in zip(xs, got):
        ref = _rne_bf16_fraction(float(x))
        assert gv == ref, (x, gv, ref)


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(4)
    xs = rng.standard_normal(10000) * 10.0 ** rng.integers(-45, 39, 10000)
    assert np.array_equal(oracle.round_f32(xs).numpy(), xs.astype(np.float32))


# ---------------------------------------------------------------------------
# Softmax
# ---------------------------------------------------------------------------

def test_softmax_closed_forms():
    # constant row of length 2^k: every entry exactly 2^-k
    s = torch.full((3, 64), 0.75, dtype=torch.float32)
    p = oracle.softmax_rows(s)
    assert np.all(p == 1.0 / 64)
    # two entries [0, x]: p = [1/(1+e^x), 1/(1+e^-x)]
    xs = torch.tensor([[0.0, 2.5], [0.0, -7.0], [0.0, 0.0]], dtype=torch.float32)
    p = oracle.softmax_rows(xs)
    for (_, x), row in zip(xs.tolist(), p):
        assert abs(row[0] - 1.0 / (1.0 + math.exp(x))) <= 4e-16
        assert abs(row[1] - 1.0 / (1.0 + math.exp(-x))) <= 4e-16
    # one dominant logit
    s = torch.zeros(1, 816)
    s[0, 123] = 200.0
    p = oracle.softmax_rows(s)
    assert p[0, 123] == 1.0 / (1.0 + 815 * math.exp(-200.0))
    assert abs(p[0, 0] - math.exp(-200.0)) <= 1e-15 * math.exp(-200.0)


def test_softmax_invariances():
    s = inputs.normal_bf16((5, 816), 4.0, 3).to(torch.float32)
    p = oracle.softmax_rows(s)
    assert np.allclose(p.sum(1), 1.0, rtol=0, atol=1e-13)
    # exact shift invariance (shift by 4 is exact for these fp32 values)
    assert np.array_equal(oracle.softmax_rows(s + 4.0), p)
    # permutation equivariance (the sum order changes, so up to double rounding)
    perm = torch.randperm(816, generator=torch.Generator().manual_seed(1))
    pp = oracle.softmax_rows(s[:, perm].contiguous())
    assert np.allclose(pp, p[:, perm.numpy()], rtol=1e-13, atol=0)
    # the row argmax is preserved
    assert np.array_equal(p.argmax(1), s.argmax(1).numpy())
    # strided rows: a row stride larger than N gives the same rows
    wide = torch.zeros(5, 1000)
    wide[:, :816] = s
    assert np.array_equal(oracle.softmax_rows(wide[:, :816]), p)


# ---------------------------------------------------------------------------
# Convolution
# ---------------------------------------------------------------------------

CONV_CASES = [
    # B, C, H, W, Co, KH, KW, stride, padding, dilation, groups
    (2, 3, 28, 28, 8, 14, 14, 14, 0, 1, 1),      # the patch-embedding shape, small
    (2, 4, 9, 11, 6, 3, 3, 1, 1, 1, 1),
    (1, 4, 10, 10, 4, 3, 2, (2, 1), (1, 0), (2, 1), 2),
    (3, 6, 7, 8, 9, 2, 3, 2, 2, 1, 3),
]


@pytest.mark.parametrize("case", CONV_CASES)
def test_conv_direct_equals_unfold_form_exactly(case):
    B, C, H, W, Co, KH, KW, st, pd, dl, gr = case
    x = inputs.uniform_bf16((B, C, H, W), -1, 1, 0)
    w = inputs.normal_bf16((Co, C // gr, KH, KW), 0.5, 1)
    bias = inputs.normal_bf16((Co,), 0.1, 2)
    y, ya = oracle.conv2d(x, w, bias, st, pd, dl, gr)
    y2, ya2 = oracle.conv2d_via_unfold(x, w, bias, st, pd, dl, gr)
    # same products summed in the same order: bit-identical doubles
    assert np.array_equal(y, y2) and np.array_equal(ya, ya2)


@pytest.mark.parametrize("case", CONV_CASES)
def test_unfold_matches_torch_unfold(case):
    B, C, H, W, Co, KH, KW, st, pd, dl, gr = case
    x = inputs.uniform_bf16((B, C, H, W), -1, 1, 0)
    cols = oracle.unfold(x, (KH, KW), st, pd, dl)
    ref = F.unfold(x, (KH, KW), dilation=dl, padding=pd, stride=st)
    assert torch.equal(cols, ref)


def test_conv_output_size_formula():
    assert oracle.conv_out_size(224, 14, 14, 0, 1) == 16
    for n, k, s, p, d in [(10, 3, 1, 1, 1), (11, 3, 2, 0, 2), (7, 7, 1, 3, 1), (5, 2, 3, 2, 2)]:
        ref = F.conv2d(torch.zeros(1, 1, n, n), torch.zeros(1, 1, k, k), stride=s, padding=p,
                       dilation=d).shape[-1]
        assert oracle.conv_out_size(n, k, s, p, d) == ref


def test_conv_onehot_weight_samples_the_image():
    x = inputs.uniform_bf16((2, 3, 28, 28), -1, 1, 0)
    w = torch.zeros(3, 3, 14, 14, dtype=torch.bfloat16)
    w[0, 0, 0, 0] = 1     # out channel 0 picks x[:, 0, 14*oh, 14*ow]
    w[1, 2, 5, 9] = 1     # out channel 1 picks x[:, 2, 14*oh+5, 14*ow+9]
    w[2, 1, 13, 13] = -1  # out channel 2 picks -x[:, 1, 14*oh+13, 14*ow+13]
    y, _ = oracle.conv2d(x, w, None, 14, 0, 1, 1)
    xd = x.to(torch.float64).numpy()
    assert np.array_equal(y[:, 0], xd[:, 0, 0::14, 0::14])
    assert np.array_equal(y[:, 1], xd[:, 2, 5::14, 9::14])
    assert np.array_equal(y[:, 2], -xd[:, 1, 13::14, 13::14])


def test_conv_against_exact_rationals_tiny():
    x = inputs.normal_bf16((1, 2, 5, 4), 1.0, 4)
    w = inputs.normal_bf16((2, 1, 2, 3), 1.0, 5)
    bias = inputs.normal_bf16((2,), 1.0, 6)
    st, pd, dl, gr = (2, 1), (1, 1), (1, 2), 2
    y, _ = oracle.conv2d(x, w, bias, st, pd, dl, gr)
    X = x.to(torch.float64).numpy()
    Wt = w.to(torch.float64).numpy()
    bv = bias.to(torch.float64).numpy()
    Ho, Wo = y.shape[2], y.shape[3]
    for co in range(2):
        g = co  # one channel per group
        for oh in range(Ho):
            for ow in range(Wo):
                acc, accabs = Fraction(float(bv[co])), abs(Fraction(float(bv[co])))
                for kh in range(2):
                    for kw in range(3):
                        ih, iw = oh * 2 - 1 + kh, ow * 1 - 1 + kw * 2
                        if 0 <= ih < 5 and 0 <= iw < 4:
                            t = Fraction(float(X[0, g, ih, iw])) * Fraction(float(Wt[co, 0, kh, kw]))
                            acc += t
                            accabs += abs(t)
                assert abs(Fraction(y[0, co, oh, ow]) - acc) <= Fraction(8, 2 ** 53) * accabs


def test_conv_matches_torch_conv2d_in_double():
    # an independent library convolution in float64 on the same bf16 values
    x = inputs.uniform_bf16((2, 3, 28, 28), -1, 1, 0)
    w = inputs.normal_bf16((5, 3, 14, 14), 0.02, 1)
    bias = inputs.normal_bf16((5,), 0.01, 2)
    y, ya = oracle.conv2d(x, w, bias, 14, 0, 1, 1)
    ref = F.conv2d(x.double(), w.double(), bias.double(), stride=14).numpy()
    assert np.all(np.abs(y - ref) <= 1e-13 * ya)


# ---------------------------------------------------------------------------
# The invariance checker, against the page's split-K toy (negative control)
# ---------------------------------------------------------------------------

def _read_toy_pattern():
    out = {}
    with open(os.path.join(GOLDEN, "splitk_toy_pattern.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                pol, m, flag = line.split()
                out[(pol, int(m))] = flag == "True"
    return out


def _toy_row0(x_row: np.ndarray, w: np.ndarray, M: int, by_batch: bool) -> np.ndarray:
    """Row 0 of the toy split-K GEMM in float32: 4 K-chunks if M < 64 (by_batch), else 1.
    Each chunk is a sequential float32 sum over its k range; chunks are then
    added in order."""
    K = w.shape[0]
    splits = 4 if (by_batch and M < 64) else 1
    bounds = np.linspace(0, K, splits + 1).astype(int)
    parts = []
    for s, e in zip(bounds[:-1], bounds[1:]):
        acc = np.zeros(w.shape[1], dtype=np.float32)
        for k in range(s, e):
            acc = (acc + np.float32(x_row[k]) * w[k]).astype(np.float32)
        parts.append(acc)
    total = np.zeros(w.shape[1], dtype=np.float32)
    for p in parts:
        total = (total + p).astype(np.float32)
    return total


def test_invariance_checker_flags_batch_dependent_split():
    from tests.invariance import row0_bit_equal
    expected = _read_toy_pattern()
    rng = np.random.default_rng(0)
    K, N = 1024, 64
    w = rng.standard_normal((K, N)).astype(np.float32)
    x0 = rng.standard_normal(K).astype(np.float32)
    for pol in ("by_batch", "fixed"):
        alone = _toy_row0(x0, w, 1, pol == "by_batch")
        for M in (8, 63, 64, 200):
            batched = _toy_row0(x0, w, M, pol == "by_batch")
            assert row0_bit_equal(torch.from_numpy(alone), torch.from_numpy(batched)) == expected[(pol, M)]
