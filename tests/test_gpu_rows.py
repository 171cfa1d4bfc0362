"""GPU parity of the invariant row reductions (RMSNorm, log-softmax, row mean
over the last dimension) against the fp64 oracle, and their invariances
("Unmasking the True Culprit: Why Temperature=0 Doesn't Mean Deterministic LLM
Inference", section "Beyond Matrix Multiplication: Other Critical Operations":
each row is reduced in one fixed order whatever the batch).

Tolerances, per element, from the fp64 oracle value ``ref`` (u_out the unit
roundoff of the output type: 2^-8 bf16, 2^-11 fp16, 2^-24 fp32; d = N/32 + 32
bounds the number of fp32 roundings on any path of the reduction tree: at most
ceil(N/32) sequential adds per thread, 5 butterfly levels and 16 warp partials):
    RMSNorm      |y - ref| <= (d + 16) * 2^-24 * |ref| + u_out |ref| + floor
    log-softmax  |y - ref| <= 2^-22 (|x - m| + |lse|) + (d + 8) * 2^-23 + u_out |ref|
    mean         |y - ref| <= (d + 2) * 2^-24 * mean|x| + u_out |ref| + floor
The sum of squares (RMSNorm) and of exponentials (log-softmax) add positive
terms, so their relative error is at most about d * 2^-24; the square root
halves it; the remaining terms are the few separately rounded scalar steps
(divide, add eps, square root, reciprocal, two multiplies; expf and logf
within 2 ulp).  floor = 2^-25 for fp16 output (half its subnormal spacing),
0 otherwise.
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

U_OUT = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11, torch.float32: 2.0 ** -24}
FLOOR = {torch.bfloat16: 0.0, torch.float16: 2.0 ** -25, torch.float32: 0.0}
DTYPES = (torch.bfloat16, torch.float16, torch.float32)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    binding.load()
    yield
    assert binding.bi_device_status() == binding.BI_OK


def _x(shape, dtype, std, seed):
    return inputs.normal_f32(shape, std, seed).to(dtype)


def _assert_within(y: torch.Tensor, ref: np.ndarray, bound: np.ndarray, what: str):
    g = y.detach().to("cpu", torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    bad = ~(err <= bound)  # NaN fails
    if bad.any():
        idx = np.argwhere(bad)[:5]
        det = [(tuple(i), g[tuple(i)], ref[tuple(i)], bound[tuple(i)]) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, e.g. {det}")


def _d(N: int) -> float:
    return N / 32 + 32


def check_rmsnorm(y, ref, N, what=""):
    bound = ((_d(N) + 16) * 2.0 ** -24 + U_OUT[y.dtype]) * np.abs(ref) + FLOOR[y.dtype]
    _assert_within(y, ref, bound, what)


def check_log_softmax(y, ref, N, what=""):
    # lse = -max_j ref (the largest input gives y = -lse); |x - m| = |ref + lse|
    g = y.detach().to("cpu", torch.float64).numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    fin = np.isfinite(ref)
    assert np.array_equal(g[~fin], ref[~fin]), f"{what}: non-finite entries differ"
    lse = -np.max(np.where(fin, ref, -np.inf), axis=1, keepdims=True)
    bound = (2.0 ** -22 * (np.abs(ref + lse) + np.abs(lse)) + (_d(N) + 8) * 2.0 ** -23 +
             U_OUT[y.dtype] * np.abs(ref))
    err = np.where(fin, np.abs(g - ref), 0.0)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        det = [(tuple(i), g[tuple(i)], ref[tuple(i)], bound[tuple(i)]) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, e.g. {det}")


def check_mean(y, ref, absmean, N, what=""):
    bound = (_d(N) + 2) * 2.0 ** -24 * absmean + U_OUT[y.dtype] * np.abs(ref) + FLOOR[y.dtype]
    _assert_within(y, ref, bound, what)


# shapes spanning every team size (32, 64, 256 and 1024 threads), rows split
# over a cluster of 2, 3 or 8 CTAs (N > 4096 G: 32768 fp32 / 65536 16-bit
# elements per CTA) including more than one register chunk per thread,
# ragged tails (N mod 4 != 0), a single element, a single row and odd row
# counts (teams of a block left without a row)
SHAPES = [(1, 1), (3, 7), (37, 1000), (11, 2000), (9, 3001), (19, 4099), (9, 8192), (3, 12345),
          (2, 40003), (3, 70001), (1, 600001)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("x_dtype", DTYPES)
def test_rmsnorm_matches_oracle(shape, x_dtype):
    R, N = shape
    x = _x(shape, x_dtype, 1.0, 1)
    w = inputs.uniform_bf16((N,), 0.5, 1.5, 2)
    for wt, yd in ((None, x_dtype), (w, x_dtype), (w.float(), torch.float32), (w.half(), torch.bfloat16)):
        ref = oracle.rmsnorm_rows(x, wt, eps=1e-6)
        y = binding.bi_rmsnorm_lastdim(x.cuda(), None if wt is None else wt.cuda(), 1e-6, out_dtype=yd)
        check_rmsnorm(y, ref, N, f"rmsnorm {shape} {x_dtype} w={None if wt is None else wt.dtype} -> {yd}")


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("x_dtype", DTYPES)
def test_log_softmax_matches_oracle(shape, x_dtype):
    R, N = shape
    s = _x(shape, x_dtype, 3.0, 3)
    ref = oracle.log_softmax_rows(s)
    for yd in (torch.float32, x_dtype):
        y = binding.bi_log_softmax_lastdim(s.cuda(), out_dtype=yd)
        check_log_softmax(y, ref, N, f"log_softmax {shape} {x_dtype} -> {yd}")


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("x_dtype", DTYPES)
def test_mean_matches_oracle(shape, x_dtype):
    R, N = shape
    x = _x(shape, x_dtype, 1.0, 4)
    ref, absmean = oracle.mean_rows(x)
    for yd in (torch.float32, x_dtype):
        y = binding.bi_mean_lastdim(x.cuda(), out_dtype=yd)
        check_mean(y, ref, absmean, N, f"mean {shape} {x_dtype} -> {yd}")


@pytest.mark.parametrize("N", [1000, 3001, 12345, 40003])
def test_rows_alone_equal_rows_in_a_batch(N):
    # every row's bits are the same whatever rows are reduced with it
    x = _x((300, N), torch.bfloat16, 1.0, 5).cuda()
    w = inputs.uniform_bf16((N,), 0.5, 1.5, 6).cuda()
    full = (binding.bi_rmsnorm_lastdim(x, w), binding.bi_log_softmax_lastdim(x), binding.bi_mean_lastdim(x))
    for M in (1, 2, 7, 8, 9, 64, 299):
        part = (binding.bi_rmsnorm_lastdim(x[:M], w), binding.bi_log_softmax_lastdim(x[:M]),
                binding.bi_mean_lastdim(x[:M]))
        for a, b in zip(part, full):
            assert bits_equal(a, b[:M]), M
    for r in (0, 151, 299):
        assert bits_equal(binding.bi_rmsnorm_lastdim(x[r:r + 1], w), full[0][r:r + 1])
        assert bits_equal(binding.bi_log_softmax_lastdim(x[r:r + 1]), full[1][r:r + 1])
        assert bits_equal(binding.bi_mean_lastdim(x[r:r + 1]), full[2][r:r + 1])
    # and run to run
    assert bits_equal(binding.bi_rmsnorm_lastdim(x, w), full[0])
    assert bits_equal(binding.bi_log_softmax_lastdim(x), full[1])


@pytest.mark.parametrize("N", [1001, 12347])
def test_misaligned_and_strided_rows_give_the_same_bits(N):
    # a row that starts off a 4-element boundary is loaded element by element
    # but summed in the same order: identical results; row strides and a
    # strided weight are honoured
    x = _x((40, N), torch.bfloat16, 1.0, 7)
    w = inputs.uniform_bf16((N,), 0.5, 1.5, 8)
    store = torch.zeros((40, N + 5), dtype=torch.bfloat16)
    store[:, 1:N + 1] = x
    xs = store.cuda()[:, 1:N + 1]          # misaligned base, row stride N + 5
    pad = N + (-N) % 4
    xa = torch.zeros((40, pad), dtype=torch.bfloat16)
    xa[:, :N] = x
    xa = xa.cuda()[:, :N]                  # every row on a 4-element boundary
    wstore = torch.zeros((2 * N,), dtype=torch.bfloat16)
    wstore[::2] = w
    ws = wstore.cuda()[::2]                # weight with stride 2
    ya = binding.bi_rmsnorm_lastdim(xa, w.cuda())
    assert bits_equal(binding.bi_rmsnorm_lastdim(xs, w.cuda()), ya)
    assert bits_equal(binding.bi_rmsnorm_lastdim(xa, ws), ya)
    assert bits_equal(binding.bi_log_softmax_lastdim(xs), binding.bi_log_softmax_lastdim(xa))
    assert bits_equal(binding.bi_mean_lastdim(xs), binding.bi_mean_lastdim(xa))
    # a strided output row and a strided mean vector
    ybig = torch.full((40, N + 3), 7.0, dtype=torch.float32, device="cuda")
    binding.bi_log_softmax_lastdim(xa, out=ybig[:, 1:N + 1])
    assert bits_equal(ybig[:, 1:N + 1].contiguous(), binding.bi_log_softmax_lastdim(xa))
    assert bool((ybig[:, 0] == 7.0).all()) and bool((ybig[:, N + 1:] == 7.0).all())
    mbig = torch.full((80,), 7.0, dtype=torch.float32, device="cuda")
    binding.bi_mean_lastdim(xa, out=mbig[::2])
    assert bits_equal(mbig[::2].contiguous(), binding.bi_mean_lastdim(xa))
    assert bool((mbig[1::2] == 7.0).all())


# RMSNorm with more than four blocks per SM runs a register-capped form of
# the same kernel (four resident blocks per SM): the row count picks it, the
# bits must not depend on it.  Teams of 32 (8 rows a block), 64 (4) and 256
# (1) threads; weight of the input's type, and no weight.
DENSE_ROWS = [(torch.bfloat16, 1000, 5200), (torch.bfloat16, 4096, 2600), (torch.float32, 3000, 700),
              (torch.float16, 12345, 700)]


@pytest.mark.parametrize("x_dtype,N,R", DENSE_ROWS)
def test_rmsnorm_dense_form_equals_small_grids(x_dtype, N, R):
    x = _x((R, N), x_dtype, 1.0, 12)
    w = inputs.uniform_bf16((N,), 0.5, 1.5, 13).to(x_dtype)
    xg, wg = x.cuda(), w.cuda()
    for wt in (wg, None):
        full = binding.bi_rmsnorm_lastdim(xg, wt, 1e-6)
        for r in (0, R // 2, R - 1):
            assert bits_equal(binding.bi_rmsnorm_lastdim(xg[r:r + 1], wt, 1e-6), full[r:r + 1]), (r, wt is None)
        assert bits_equal(binding.bi_rmsnorm_lastdim(xg[:9], wt, 1e-6), full[:9])
        rows = [0, R - 1]
        ref = oracle.rmsnorm_rows(x[rows], None if wt is None else w, eps=1e-6)
        check_rmsnorm(full[rows], ref, N, f"rmsnorm dense {x_dtype} {N} w={wt is not None}")


# Long rows reduced by clusters of 1024-thread CTAs: when the rows' clusters
# take more than one wave of SMs the kernel streams each thread's groups from
# memory on every pass instead of holding them in registers.  The row count
# picks the form; the bits must not depend on it.
LONG_ROWS = [(torch.float32, 128256, 40), (torch.float32, 40003, 90), (torch.bfloat16, 70001, 80),
             (torch.float16, 600001, 20), (torch.bfloat16, 40003, 160)]


@pytest.mark.parametrize("x_dtype,N,R", LONG_ROWS)
def test_log_softmax_streaming_form_equals_register_form(x_dtype, N, R):
    s = _x((R, N), x_dtype, 3.0, 11)
    s[3, ::5] = float("-inf")  # a masked row
    sg = s.cuda()
    for yd in (torch.float32, x_dtype):
        full = binding.bi_log_softmax_lastdim(sg, out_dtype=yd)  # more clusters than SMs
        for r in (0, 3, R // 2, R - 1):
            assert bits_equal(binding.bi_log_softmax_lastdim(sg[r:r + 1], out_dtype=yd), full[r:r + 1]), (yd, r)
        assert bits_equal(binding.bi_log_softmax_lastdim(sg[:7], out_dtype=yd), full[:7]), yd
        rows = [0, 3, R - 1]
        check_log_softmax(full[rows], oracle.log_softmax_rows(s[rows]), N, f"streamed {x_dtype} {N} -> {yd}")
    # rows off a 4-element boundary (element loads) give the same bits
    store = torch.zeros((R, N + 3), dtype=x_dtype)
    store[:, 1:N + 1] = s
    xs = store.cuda()[:, 1:N + 1]
    assert bits_equal(binding.bi_log_softmax_lastdim(xs), binding.bi_log_softmax_lastdim(sg))
    assert bits_equal(binding.bi_log_softmax_lastdim(xs[:1]), binding.bi_log_softmax_lastdim(sg[:1]))


def test_log_softmax_masked_and_large_entries():
    # -inf entries (a mask) give exactly -inf and weight nothing; large logits
    # do not overflow because the row maximum is subtracted first
    s = _x((6, 5000), torch.float32, 3.0, 9)
    s[:, ::3] = float("-inf")
    s[1] += 20000.0
    s[2, 17] = 1e30
    ref = oracle.log_softmax_rows(s)
    y = binding.bi_log_softmax_lastdim(s.cuda())
    check_log_softmax(y, ref, 5000, "masked / large")
    assert bool(torch.isneginf(y[:, ::3]).all())


def test_rmsnorm_eps_and_zero_rows():
    # an all-zero row gives zeros (1/sqrt(eps) finite); eps shifts the scale
    x = _x((4, 3000), torch.float32, 1.0, 10)
    x[2] = 0.0
    for eps in (0.0, 1e-6, 0.5):
        ref = oracle.rmsnorm_rows(x, None, eps=eps)
        if eps == 0.0:
            ref[2] = 0.0  # 0 * inf in the definition; the kernel returns 0 * (1/sqrt(0)) = NaN
            y = binding.bi_rmsnorm_lastdim(x.cuda(), None, eps)
            assert bool(torch.isnan(y[2]).all())
            check_rmsnorm(y[[0, 1, 3]], ref[[0, 1, 3]], 3000, "eps=0")
            continue
        y = binding.bi_rmsnorm_lastdim(x.cuda(), None, eps)
        check_rmsnorm(y, ref, 3000, f"eps={eps}")
        assert bool((y[2] == 0).all())


def test_full_size_workloads_sampled_rows():
    # the timed shapes: RMSNorm over [8192, 4096] bf16 hidden states with a
    # gain, log-softmax over [64, 128256] fp32 logits, mean over [8192, 4096]
    x, w = inputs.rmsnorm_hidden(8192)
    xg, wg = x.cuda(), w.cuda()
    y = binding.bi_rmsnorm_lastdim(xg, wg, 1e-6)
    m = binding.bi_mean_lastdim(xg)
    rows = [0, 1, 4095, 8191]
    check_rmsnorm(y[rows], oracle.rmsnorm_rows(x[rows], w, eps=1e-6), 4096, "rmsnorm full")
    ref, absmean = oracle.mean_rows(x[rows])
    check_mean(m[rows], ref, absmean, 4096, "mean full")
    assert bits_equal(binding.bi_rmsnorm_lastdim(xg[:1], wg, 1e-6), y[:1])
    s = inputs.vocab_logits(64)
    sg = s.cuda()
    p = binding.bi_log_softmax_lastdim(sg)
    rows = [0, 33, 63]
    check_log_softmax(p[rows], oracle.log_softmax_rows(s[rows]), 128256, "log_softmax full")
    assert bits_equal(binding.bi_log_softmax_lastdim(sg[:1]), p[:1])
