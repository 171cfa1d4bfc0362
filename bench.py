"""Benchmark of the batch-invariant contractions on GB300.

Headline line (one JSON object on stdout, rank 0): the LLM-linear addmm
workload -- x [M,4096] bf16 @ W [4096,14336] bf16 + bias, bf16 output, fp32
accumulation -- over its whole M sweep {1,...,8192}.  One "step" is one
bi_addmm launch per M of the sweep (12 launches).  L2 is flushed (512 MB
written, then read back so no dirty lines remain) before every timed launch, and each launch is timed alone with CUDA
events on the launching stream, so ``value`` = total algorithmic FLOP of the
sweep / total kernel time (TFLOP/s), ``ms_per_step`` = that kernel time.

Also reported: per-M TFLOP/s, GB/s and roofline fraction for this workload
and for the other four workloads (large square mm, patch-embedding conv,
attention bmm+softmax+bmm, tiny mm), the same shapes through cuBLAS / cuDNN
with their own row-0 invariance, the roofline of the dominant kernel, the
end-to-end figure through the public API with host buffers, the SM clocks
sampled during the timed region, and the fp64 CPU oracle timed on the host
cores (a reported baseline).

``--impl reference`` times the fp64 CPU oracle (the only reference this
build has) on bounded samples of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "TFLOP/s and % of roofline vs M (bf16 in, fp32 acc), bitwise batch-invariant"
UNIT = "TFLOP/s"
WORKLOAD = "LLM linear addmm: x[M,4096] bf16 @ W[4096,14336] bf16 + bias[14336], bf16 out, M sweep"
K_DIM, N_DIM = 4096, 14336
FLUSH_BYTES = 512 << 20

KERNEL_SOURCES = ["bi_gemm.cu", "bi_roles.cuh", "bi_ptx.cuh", "bi_common.h"]


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "invariant_gemm_bi_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic() -> float | None:
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_kernel_llm_addmm_M8192.md")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def addmm_flops(M: int) -> float:
    return 2.0 * M * K_DIM * N_DIM + M * N_DIM


def addmm_bytes(M: int) -> float:
    return 2.0 * (M * K_DIM + K_DIM * N_DIM + N_DIM + M * N_DIM)


def roofline_frac(flops: float, nbytes: float, seconds: float, peaks: dict) -> tuple[float, str]:
    t_c = flops / (peaks["bf16_tflops"] * 1e12)
    t_b = nbytes / (peaks["hbm_gbs"] * 1e9)
    return max(t_c, t_b) / seconds, ("tensor" if t_c >= t_b else "hbm")


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_rows_timing(n_rows: int, seed: int = 0) -> tuple[float, int]:
    """Times the fp64 oracle computing n_rows full output rows of the addmm
    workload; returns (seconds, threads)."""
    import oracle
    from invariant_gemm_bi_gb300 import inputs
    x = inputs.normal_bf16((n_rows, K_DIM), 1.0, seed)
    w = inputs.normal_bf16((K_DIM, N_DIM), 0.02, 1)
    bias = inputs.normal_bf16((N_DIM,), 0.01, 2)
    oracle.mm(x[:1], w, bias=bias)  # load + warm
    t0 = time.perf_counter()
    oracle.mm(x, w, bias=bias)
    return time.perf_counter() - t0, oracle.num_threads()


def cpu_baseline(target_s: float = 12.0) -> dict:
    import oracle
    threads = oracle.num_threads()
    probe = max(threads, 8)
    t, _ = oracle_rows_timing(probe)
    rows = int(min(4096, max(probe, probe * target_s / max(t, 1e-3))))
    t, threads = oracle_rows_timing(rows)
    return {"value": round(2.0 * rows * K_DIM * N_DIM / t / 1e12, 6), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"{rows} full output rows of the addmm workload (K=4096, N=14336) in fp64, "
                      f"{t:.1f} s"}


def run_reference(args, rank, world):
    """--impl reference: the fp64 oracle on the host cores, bounded sample per step."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    rows = threads  # one output row per host thread per step
    for _ in range(args.warmup):
        oracle_rows_timing(rows)
    times = []
    for s in range(args.steps):
        t, _ = oracle_rows_timing(rows, seed=s)
        times.append(t)
    total = sum(times)
    value = 2.0 * rows * K_DIM * N_DIM * args.steps / total / 1e12
    line = {"metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": WORKLOAD, "sample_rows_per_step": rows},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{rows} output rows per step of the addmm workload in fp64"},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def flush_l2(flush_buf):
    """Writes a 512 MB buffer (evicting everything from L2), then reads it back so
    that the lines left in L2 are clean: the timed kernel starts with a cold L2
    and pays no write-back of the flush's dirty lines."""
    flush_buf.fill_(1)
    torch.sum(flush_buf.view(torch.int64), dtype=torch.int64)


def time_launch(fn, flush_buf, stream):
    """Flush L2, then bracket one launch with CUDA events on `stream`; returns the events."""
    flush_l2(flush_buf)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fn()
    e1.record(stream)
    return e0, e1


def quantile(ts, q: float) -> float:
    """Linear-interpolated quantile q (0..1) of the samples."""
    ts = sorted(ts)
    if len(ts) == 1:
        return ts[0]
    x = q * (len(ts) - 1)
    i = int(x)
    j = min(i + 1, len(ts) - 1)
    return ts[i] + (ts[j] - ts[i]) * (x - i)


def spread(ts) -> dict:
    """Median and the 10th / 90th percentiles of per-launch times (seconds), in µs."""
    return {"p10_us": round(quantile(ts, 0.1) * 1e6, 2), "p90_us": round(quantile(ts, 0.9) * 1e6, 2),
            "launches": len(ts)}


def measure_all(fn, flush_buf, stream, reps: int) -> list[float]:
    """Per-launch times (seconds) of `reps` launches, each after an L2 flush."""
    evs = [time_launch(fn, flush_buf, stream) for _ in range(reps)]
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in evs]


def measure(fn, flush_buf, stream, reps: int) -> float:
    """Median per-launch time (seconds)."""
    return statistics.median(measure_all(fn, flush_buf, stream, reps))


def bits_equal(x, y) -> bool:
    return x.shape == y.shape and bool(torch.equal(x.contiguous().view(torch.uint8),
                                                  y.contiguous().view(torch.uint8)))


def extra_sweeps(flush_buf, stream, peaks, reps: int, only: str | None = None) -> dict:
    """The other workloads, once each: ours vs cuBLAS / cuDNN, with row-0 flags.
    `only` restricts it to one workload (square, conv, attention, tiny, fp16, rows), or to
    the attention's head-dimension sweep alone (heads)."""
    import torch.nn.functional as F
    from invariant_gemm_bi_gb300 import binding, inputs
    out = {}
    want = (lambda name: only is None or only == name)

    # large square mm, fp32 out; plain weight and packed weight
    if want("square"):
        _square(out, binding, inputs, flush_buf, stream, peaks, reps, point_fn(peaks))
    if want("conv"):
        _conv(out, binding, inputs, F, flush_buf, stream, peaks, reps, point_fn(peaks))
    if want("attention"):
        _attention(out, binding, inputs, flush_buf, stream, peaks, reps, point_fn(peaks))
    if want("attention") or only == "heads":
        _attention_heads(out, binding, inputs, flush_buf, stream, reps, point_fn(peaks))
    if want("tiny"):
        _tiny(out, binding, inputs, flush_buf, stream, 20 * reps)  # >= 1000 launches per point at reps >= 50
    if want("fp16"):
        _fp16(out, binding, inputs, flush_buf, stream, peaks, reps, point_fn(peaks))
    if want("rows"):
        _rows(out, binding, inputs, flush_buf, stream, peaks, reps)
    return out


def point_fn(peaks):
    """point(flops, bytes, t): figures at the median of t (a list of per-launch
    times, or one time), with the 10th / 90th percentiles of a list."""
    def point(flops, nbytes, t):
        ts = t if isinstance(t, list) else [t]
        med = statistics.median(ts)
        frac, bound = roofline_frac(flops, nbytes, med, peaks)
        d = {"us": round(med * 1e6, 2), "tflops": round(flops / med / 1e12, 2),
             "gbs": round(nbytes / med / 1e9, 1), "roofline_frac": round(frac, 3), "bound": bound}
        if len(ts) > 1:
            d.update(spread(ts))
        return d
    return point


def _square(out, binding, inputs, flush_buf, stream, peaks, reps, point):
    a, w = inputs.square_mm(max(inputs.SQUARE_MM_M), device="cuda")
    wp = binding.bi_pack_weight(w)
    rows0 = {}
    res = []
    for M in inputs.SQUARE_MM_M:
        am = a[:M]
        c = torch.empty(M, 8192, dtype=torch.float32, device="cuda")
        cp = torch.empty(M, 8192, dtype=torch.float32, device="cuda")
        t = measure_all(lambda: binding.bi_mm(am, w, out=c), flush_buf, stream, reps)
        tp = measure_all(lambda: binding.bi_addmm_packed(None, am, wp, out=cp), flush_buf, stream, reps)
        rows0[M] = c[:1].clone()
        flops, nb = 2.0 * M * 8192 * 8192, 2.0 * (M * 8192 + 8192 * 8192) + 4.0 * M * 8192
        r = {"M": M, **point(flops, nb, t),
             "packed_weight": {**point(flops, nb, tp), "bits_equal_plain": bits_equal(c, cp)}}
        del cp
        cb = torch.empty(M, 8192, dtype=torch.bfloat16, device="cuda")
        tc = measure(lambda: torch.mm(am, w, out=cb), flush_buf, stream, reps)
        r["cublas_us_bf16_out"] = round(tc * 1e6, 2)
        rows0[("cublas", M)] = torch.mm(am, w)[:1].clone()
        res.append(r)
        del c, cb
    ref0 = rows0[1]
    out["square_mm"] = {"points": res,
                        "row0_bit_equal_all_M": all(bits_equal(rows0[M], ref0) for M in inputs.SQUARE_MM_M),
                        "cublas_row0_bit_equal_all_M": all(bits_equal(rows0[("cublas", M)], rows0[("cublas", 1)])
                                                           for M in inputs.SQUARE_MM_M)}
    del a, w, wp


def _fp16(out, binding, inputs, flush_buf, stream, peaks, reps, point):
    # the LLM-linear layer with fp16 operands and output (packed weight), its
    # own fixed fp16 tile path; cuBLAS fp16 addmm alongside
    x, w, bias = inputs.llm_addmm_f16(max(inputs.LLM_ADDMM_F16_M), device="cuda")
    wp = binding.bi_pack_weight(w)
    res, rows0 = [], {}
    for M in inputs.LLM_ADDMM_F16_M:
        xm = x[:M]
        c = torch.empty(M, N_DIM, dtype=torch.float16, device="cuda")
        t = measure_all(lambda: binding.bi_addmm_packed(bias, xm, wp, out=c), flush_buf, stream, reps)
        rows0[M] = c[:1].clone()
        r = {"M": M, **point(addmm_flops(M), addmm_bytes(M), t)}
        r["cublas_us"] = round(measure(lambda: torch.addmm(bias, xm, w), flush_buf, stream, reps) * 1e6, 2)
        res.append(r)
        del c
    first = inputs.LLM_ADDMM_F16_M[0]
    out["llm_addmm_fp16"] = {"points": res,
                             "row0_bit_equal_all_M": all(bits_equal(rows0[M], rows0[first]) for M in rows0)}
    del x, w, bias, wp


def _conv(out, binding, inputs, F, flush_buf, stream, peaks, reps, point):
    # packed filter (bi_conv2d_patch_packed, packed once like the linear weight),
    # the filter as given (bi_conv2d_patch: the same patch kernel, its filter
    # stages built from w) and cuDNN on the same shapes
    x, wc, bc = inputs.patch_embed(max(inputs.PATCH_EMBED_B), device="cuda")
    wpk = binding.bi_conv_pack_weight(wc)
    res, y0, yp0, yc0 = [], {}, {}, {}
    for B in inputs.PATCH_EMBED_B:
        xb = x[:B]
        y = torch.empty(B, 1152, 16, 16, dtype=torch.bfloat16, device="cuda")
        t = measure_all(lambda: binding.bi_conv2d_patch_packed(xb, wpk, bc, out=y), flush_buf, stream, reps)
        y0[B] = y[:1].clone()
        flops = B * (2.0 * 256 * 588 * 1152 + 256 * 1152)
        nb = 2.0 * (B * 3 * 224 * 224 + 1152 * 588 + 1152 + B * 1152 * 256)
        r = {"B": B, **point(flops, nb, t)}
        tp = measure_all(lambda: binding.bi_conv2d_patch(xb, wc, bc, stride=14, out=y), flush_buf, stream, reps)
        yp0[B] = y[:1].clone()
        r["plain_filter"] = point(flops, nb, tp)
        tc = measure(lambda: F.conv2d(xb, wc, bc, stride=14), flush_buf, stream, reps)
        yc0[B] = F.conv2d(xb, wc, bc, stride=14)[:1].clone()
        r["cudnn_us"] = round(tc * 1e6, 2)
        res.append(r)
    out["patch_embed_conv"] = {"points": res,
                               "entry_point": "bi_conv2d_patch_packed (plain_filter: bi_conv2d_patch)",
                               "sample0_bit_equal_all_B": all(bits_equal(y0[B], y0[1]) for B in y0),
                               "plain_filter_sample0_bit_equal_all_B": all(bits_equal(yp0[B], yp0[1])
                                                                           for B in yp0),
                               "cudnn_sample0_bit_equal_all_B": all(bits_equal(yc0[B], yc0[1]) for B in yc0)}
    del x, wc, bc, wpk


def _attention(out, binding, inputs, flush_buf, stream, peaks, reps, point):
    # S = QK^T/16 (fp32), P = softmax(S) (bf16), O = PV (fp32)
    q, k, v = inputs.attention(max(inputs.ATTENTION_B), device="cuda")
    res, o0, of0, sd0 = [], {}, {}, {}
    for B in inputs.ATTENTION_B:
        L = 8 * B
        qb, kb, vb = q[:L], k[:L].transpose(1, 2), v[:L]
        s = torch.empty(L, 816, 816, dtype=torch.float32, device="cuda")
        p = torch.empty(L, 816, 816, dtype=torch.bfloat16, device="cuda")
        o = torch.empty(L, 816, 256, dtype=torch.float32, device="cuda")
        t1 = measure_all(lambda: binding.bi_bmm(qb, kb, alpha=1.0 / 16, out=s), flush_buf, stream, reps)
        t2s = measure_all(lambda: binding.bi_softmax_lastdim(s.view(-1, 816), out=p.view(-1, 816)),
                          flush_buf, stream, reps)
        t2 = statistics.median(t2s)
        t3 = measure_all(lambda: binding.bi_bmm(p, vb, out=o), flush_buf, stream, reps)
        o0[B] = o[:1].clone()
        f1 = L * 2.0 * 816 * 816 * 256
        b1 = L * (2.0 * 816 * 256 * 2 + 4.0 * 816 * 816)
        b2 = L * 816 * 816 * 6.0
        b3 = L * (2.0 * 816 * 816 + 2.0 * 816 * 256 + 4.0 * 816 * 256)
        tcb = measure(lambda: torch.bmm(qb, kb), flush_buf, stream, reps)
        # the same attention fused in one kernel (fp32 out), and PyTorch's SDPA
        of = torch.empty(L, 816, 256, dtype=torch.float32, device="cuda")
        tf = measure_all(lambda: binding.bi_attention(qb, k[:L], vb, 1.0 / 16, out=of), flush_buf, stream, reps)
        of0[B] = of[:1].clone()
        ff = 2 * f1
        bf = L * (3 * 2.0 * 816 * 256 + 4.0 * 816 * 256)
        tsd = measure(lambda: torch.nn.functional.scaled_dot_product_attention(qb, k[:L], vb, scale=1.0 / 16),
                      flush_buf, stream, reps)
        sd0[B] = torch.nn.functional.scaled_dot_product_attention(qb, k[:L], vb, scale=1.0 / 16)[:1].clone()
        fused = {**point(ff, bf, tf), "sdpa_us_bf16_out": round(tsd * 1e6, 2)}
        del of
        res.append({"B": B, "fused": fused, "qk": point(f1, b1, t1),
                    "softmax": {"us": round(t2 * 1e6, 2), "gbs": round(b2 / t2 / 1e9, 1),
                                "roofline_frac": round(b2 / (peaks["hbm_gbs"] * 1e9) / t2, 3), "bound": "hbm",
                                **spread(t2s)},
                    "pv": point(f1, b3, t3), "cublas_qk_us": round(tcb * 1e6, 2)})
        del s, p, o
    # a long key range: one sample (8 heads), T = 8192 -- fused with four fixed
    # 2048-key splits and a merge, the materialised chain, and PyTorch's SDPA
    ql, kl, vl = inputs.attention(1, t=8192, device="cuda")
    Lh, T = ql.shape[0], ql.shape[1]
    fl = 4.0 * Lh * T * T * 256
    bl = Lh * (3 * 2.0 * T * 256 + 4.0 * T * 256)
    ol = torch.empty(Lh, T, 256, dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.bi_attention_workspace_bytes(Lh, T, T), dtype=torch.uint8, device="cuda")
    tfl = measure_all(lambda: binding.bi_attention_ws(ql, kl, vl, 1.0 / 16, out=ol, workspace=ws), flush_buf,
                      stream, reps)
    sl = torch.empty(Lh, T, T, dtype=torch.float32, device="cuda")
    pl = torch.empty(Lh, T, T, dtype=torch.bfloat16, device="cuda")
    oc = torch.empty(Lh, T, 256, dtype=torch.float32, device="cuda")

    def chain():
        binding.bi_bmm(ql, kl.transpose(1, 2), alpha=1.0 / 16, out=sl)
        binding.bi_softmax_lastdim(sl.view(-1, T), out=pl.view(-1, T))
        binding.bi_bmm(pl, vl, out=oc)
    tch = measure(chain, flush_buf, stream, reps)
    del sl, pl
    tsd = measure(lambda: torch.nn.functional.scaled_dot_product_attention(ql, kl, vl, scale=1.0 / 16),
                  flush_buf, stream, reps)
    long_pt = {"heads": Lh, "T": T, "splits": (T + 2047) // 2048, "fused": point(fl, bl, tfl),
               "chain_us": round(tch * 1e6, 2), "sdpa_us_bf16_out": round(tsd * 1e6, 2),
               "fused_head0_equals_head_alone": bits_equal(
                   binding.bi_attention_ws(ql[:1], kl[:1], vl[:1], 1.0 / 16), ol[:1])}
    del ql, kl, vl, ol, oc, ws
    out["attention_long"] = long_pt
    out["attention"] = {"points": res, "head0_bit_equal_all_B": all(bits_equal(o0[B], o0[1]) for B in o0),
                        "fused_head0_bit_equal_all_B": all(bits_equal(of0[B], of0[1]) for B in of0),
                        "sdpa_head0_bit_equal_all_B": all(bits_equal(sd0[B], sd0[1]) for B in sd0)}
    del q, k, v


def _attention_heads(out, binding, inputs, flush_buf, stream, reps, point):
    # head dimensions 64, 128, 256 at the workload's token count (B = 32: 256
    # heads x 816 queries and keys), scale D^-1/2, bf16 out (as SDPA's)
    dims = []
    for d in (64, 128, 256):
        qd, kd, vd = inputs.attention(32, d=d, device="cuda")
        Ld = qd.shape[0]
        od = torch.empty(Ld, 816, d, dtype=torch.bfloat16, device="cuda")
        td = measure_all(lambda: binding.bi_attention(qd, kd, vd, d ** -0.5, out=od), flush_buf, stream, reps)
        tsd = measure(lambda: torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, scale=d ** -0.5),
                      flush_buf, stream, reps)
        fd = 4.0 * Ld * 816 * 816 * d
        bd = Ld * 4 * 2.0 * 816 * d
        dims.append({"D": d, "heads": Ld, "T": 816, "fused": point(fd, bd, td), "sdpa_us": round(tsd * 1e6, 2)})
        del qd, kd, vd, od
    out["attention_head_dims"] = dims


def _rows(out, binding, inputs, flush_buf, stream, peaks, reps):
    # the row reductions, HBM-bound: RMSNorm of [R, 4096] bf16 hidden states
    # with a gain (bf16 out), log-softmax of [R, 128256] fp32 logits (fp32 out),
    # mean of [R, 4096] bf16 (fp32 out); PyTorch's own kernels alongside
    hbm = peaks["hbm_gbs"] * 1e9

    def pt(nb, ts, t_torch):
        t = statistics.median(ts)
        return {"us": round(t * 1e6, 2), "gbs": round(nb / t / 1e9, 1),
                "roofline_frac": round(nb / hbm / t, 3), "bound": "hbm", "torch_us": round(t_torch * 1e6, 2),
                **spread(ts)}

    x, w = inputs.rmsnorm_hidden(max(inputs.RMSNORM_ROWS), device="cuda")
    s = inputs.vocab_logits(max(inputs.LOGITS_ROWS), device="cuda")
    N, V = x.shape[1], s.shape[1]
    rms, mean, lsm, r0 = [], [], [], {"rms": {}, "mean": {}, "lsm": {}}
    for R in inputs.RMSNORM_ROWS:
        xr = x[:R]
        y = torch.empty(R, N, dtype=torch.bfloat16, device="cuda")
        m = torch.empty(R, dtype=torch.float32, device="cuda")
        t = measure_all(lambda: binding.bi_rmsnorm_lastdim(xr, w, 1e-6, out=y), flush_buf, stream, reps)
        tt = measure(lambda: torch.nn.functional.rms_norm(xr, (N,), w, 1e-6), flush_buf, stream, reps)
        rms.append({"rows": R, **pt(2.0 * (2 * R * N + N), t, tt)})
        tm = measure_all(lambda: binding.bi_mean_lastdim(xr, out=m), flush_buf, stream, reps)
        ttm = measure(lambda: torch.mean(xr, dim=-1, dtype=torch.float32), flush_buf, stream, reps)
        mean.append({"rows": R, **pt(2.0 * R * N + 4.0 * R, tm, ttm)})
        r0["rms"][R], r0["mean"][R] = y[:1].clone(), m[:1].clone()
        del y, m
    for R in inputs.LOGITS_ROWS:
        sr = s[:R]
        y = torch.empty(R, V, dtype=torch.float32, device="cuda")
        t = measure_all(lambda: binding.bi_log_softmax_lastdim(sr, out=y), flush_buf, stream, reps)
        tt = measure(lambda: torch.log_softmax(sr, dim=-1), flush_buf, stream, reps)
        lsm.append({"rows": R, **pt(8.0 * R * V, t, tt)})
        r0["lsm"][R] = y[:1].clone()
        del y
    eq = {k: all(bits_equal(v[R], v[min(v)]) for R in v) for k, v in r0.items()}
    out["rmsnorm_hidden_4096"] = {"points": rms, "row0_bit_equal_all_R": eq["rms"]}
    out["mean_hidden_4096"] = {"points": mean, "row0_bit_equal_all_R": eq["mean"]}
    out["log_softmax_vocab_128256"] = {"points": lsm, "row0_bit_equal_all_R": eq["lsm"]}
    del x, w, s


def _tiny(out, binding, inputs, flush_buf, stream, reps):
    # launch-latency bound: report microseconds (median over `reps` launches,
    # each after an L2 flush), cuBLAS (fp32 out) on the same shapes alongside
    a, w = inputs.tiny_mm(64, device="cuda")
    res, rows0, cub0 = [], {}, {}
    for M in inputs.TINY_MM_M:
        am = a[:M]
        c = torch.empty(M, 128, dtype=torch.float32, device="cuda")
        cb = torch.empty(M, 128, dtype=torch.bfloat16, device="cuda")
        ts = measure_all(lambda: binding.bi_mm(am, w, out=c), flush_buf, stream, reps)
        rows0[M] = c[:1].clone()
        tc = measure_all(lambda: torch.mm(am, w, out=cb), flush_buf, stream, reps)
        cub0[M] = torch.mm(am, w)[:1].clone()
        res.append({"M": M, "us": round(statistics.median(ts) * 1e6, 2), **spread(ts),
                    "cublas_us_bf16_out": round(statistics.median(tc) * 1e6, 2)})
    out["tiny_mm"] = {"points": res,
                      "row0_bit_equal_all_M": all(bits_equal(rows0[M], rows0[1]) for M in rows0),
                      "cublas_row0_bit_equal_all_M": all(bits_equal(cub0[M], cub0[1]) for M in cub0)}


def run_only(args):
    """One workload's points (ours vs the library reference), printed as JSON."""
    from invariant_gemm_bi_gb300 import binding, build
    build.build()
    binding.load()
    torch.cuda.set_device(0)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):  # untimed passes
        extra_sweeps(flush_buf, torch.cuda.current_stream(), load_peaks(), reps=1, only=args.only)
    res = extra_sweeps(flush_buf, torch.cuda.current_stream(), load_peaks(), reps=max(1, args.steps),
                       only=args.only)
    print(json.dumps({"only": args.only, "steps": args.steps, "warmup": args.warmup, "result": res}))


def run_ours(args, rank, local, world):
    from invariant_gemm_bi_gb300 import binding, build, inputs
    build.build()
    binding.load()
    dev = local if torch.cuda.device_count() > local else 0
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    Ms = list(inputs.LLM_ADDMM_M)
    if args.m_list:
        Ms = [int(v) for v in args.m_list.split(",")]
    M_max = max(Ms)

    x, w, bias = inputs.llm_addmm(M_max, device="cuda")
    outs = {M: torch.empty(M, N_DIM, dtype=torch.bfloat16, device="cuda") for M in Ms}
    outs_other = {M: torch.empty(M, N_DIM, dtype=torch.bfloat16, device="cuda") for M in Ms}
    xs = {M: x[:M] for M in Ms}
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    # The weight is constant: its packed form is made once, outside any timed region.
    packed = binding.bi_pack_weight(w)
    torch.cuda.synchronize()

    def launch_packed(M, out):
        binding.bi_addmm_packed(bias, xs[M], packed, out=out)

    def launch_plain(M, out):
        binding.bi_addmm(bias, xs[M], w, out=out)

    main_fn, other_fn = ((launch_packed, launch_plain) if args.weight == "packed"
                         else (launch_plain, launch_packed))

    def launch(M):
        main_fn(M, outs[M])

    # warm-up steps
    for _ in range(args.warmup):
        for M in Ms:
            launch(M)
    for M in Ms:
        other_fn(M, outs_other[M])
    torch.cuda.synchronize()
    # row-0 invariance across the sweep (checked on the warm-up outputs), and
    # the packed and plain weights giving the same bits
    row0_equal = all(bits_equal(outs[M][:1], outs[Ms[0]][:1]) for M in Ms)
    packed_equals_plain = all(bits_equal(outs[M], outs_other[M]) for M in Ms)
    del outs_other

    # timed region: K steps x one launch per M, each after an L2 flush
    events = {M: [] for M in Ms}
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clocks:
        t_wall0 = time.perf_counter()
        for _ in range(args.steps):
            for M in Ms:
                events[M].append(time_launch(lambda: launch(M), flush_buf, stream))
        torch.cuda.synchronize()
        barrier(world)
        t_wall = time.perf_counter() - t_wall0
    per_m = {M: [a.elapsed_time(b) * 1e-3 for a, b in events[M]] for M in Ms}
    kernel_s = sum(sum(v) for v in per_m.values())
    kernel_s = max_over_ranks(kernel_s, world)
    flops_step = sum(addmm_flops(M) for M in Ms)
    total_flops = sum_over_ranks(flops_step * args.steps, world)
    value = total_flops / kernel_s / 1e12
    gpu_launches = len(Ms) * args.steps

    point = point_fn(peaks)
    sweep = [{"M": M, **point(addmm_flops(M), addmm_bytes(M), per_m[M])} for M in Ms]

    # the other weight path, same shapes
    other_out = {M: torch.empty(M, N_DIM, dtype=torch.bfloat16, device="cuda") for M in Ms}
    other_name = "plain_weight_us" if args.weight == "packed" else "packed_weight_us"
    for r in sweep:
        M = r["M"]
        r[other_name] = round(measure(lambda: other_fn(M, other_out[M]), flush_buf, stream, 20) * 1e6, 2)
    del other_out

    # cuBLAS on the same sweep (not invariant in general): time + row-0 flag
    cublas_row0 = None
    if not args.no_compare:
        cub = {}
        for M in Ms:
            tcb = measure(lambda: torch.addmm(bias, xs[M], w), flush_buf, stream, 20)
            cub[M] = (tcb, torch.addmm(bias, xs[M], w)[:1].clone())
        for r in sweep:
            r["cublas_us"] = round(cub[r["M"]][0] * 1e6, 2)
        cublas_row0 = all(bits_equal(cub[M][1], cub[Ms[0]][1]) for M in Ms)

    # dominant kernel: the M=8192 launch of gemm_kernel, at the median launch
    # time (the statistic of every sweep point)
    t_dom = statistics.median(per_m[M_max])
    f_dom = addmm_flops(M_max)
    traffic = load_traffic()
    roof = {"bound": "tensor", "achieved": round(f_dom / t_dom / 1e12, 2),
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(f_dom / t_dom / 1e12 / peaks["bf16_tflops"], 4),
            "traffic": traffic,
            "kernel": f"gemm_kernel<MN-major B, {args.weight} weight> (bi_addmm{'_packed' if args.weight == 'packed' else ''}, M=8192)",
            "peak_source": f"{peaks['source']} bf16 dense (burst)",
            "algorithmic_bytes": addmm_bytes(M_max)}

    # end to end through the public API with host buffers (pinned), per step:
    # H2D of the step's inputs (x for the largest M -- every M reads a prefix
    # of it -- W and the bias) on a copy stream into one of two device input
    # sets, the addmm of every M, and the D2H of each output on a second copy
    # stream; step i + 1's inputs cross while step i computes and its outputs
    # return.  Every copy of every timed step is inside the timed region.
    e2e = None
    if not args.no_compare:
        x_h = x.cpu().pin_memory()
        w_src = packed.buffer if args.weight == "packed" else w
        w_h = w_src.cpu().pin_memory()
        b_h = bias.cpu().pin_memory()
        outs_h = {M: torch.empty(M, N_DIM, dtype=torch.bfloat16).pin_memory() for M in Ms}
        ins = []
        for _ in range(2):
            xd, wd, bd = torch.empty_like(x), torch.empty_like(w_src), torch.empty_like(bias)
            pd = binding.PackedWeight(wd, binding.BiPackedWeightDesc(
                wd.data_ptr(), packed.desc.bytes, packed.desc.K, packed.desc.N, packed.desc.layout,
                packed.desc.tile_n))
            ins.append((xd, wd, bd, pd))
        e2e_steps = max(1, min(args.steps, 5))
        h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
        in_ready = [torch.cuda.Event() for _ in range(2)]
        in_free = [torch.cuda.Event() for _ in range(2)]   # the launches reading a set are done
        done = {M: torch.cuda.Event() for M in Ms}          # the output of M is computed
        out_free = {M: torch.cuda.Event() for M in Ms}      # ... and back on the host

        def e2e_run(n, start):
            h2d_stream.wait_event(start)
            for i in range(n):
                xd, wd, bd, pd = ins[i % 2]
                if i >= 2:
                    h2d_stream.wait_event(in_free[i % 2])
                with torch.cuda.stream(h2d_stream):
                    xd.copy_(x_h, non_blocking=True)
                    wd.copy_(w_h, non_blocking=True)
                    bd.copy_(b_h, non_blocking=True)
                    in_ready[i % 2].record(h2d_stream)
                stream.wait_event(in_ready[i % 2])
                for M in Ms:
                    if i >= 1:
                        stream.wait_event(out_free[M])  # outs[M] is rewritten only once it is home
                    if args.weight == "packed":
                        binding.bi_addmm_packed(bd, xd[:M], pd, out=outs[M])
                    else:
                        binding.bi_addmm(bd, xd[:M], wd, out=outs[M])
                    done[M].record(stream)
                    d2h_stream.wait_event(done[M])
                    with torch.cuda.stream(d2h_stream):
                        outs_h[M].copy_(outs[M], non_blocking=True)
                        out_free[M].record(d2h_stream)
                in_free[i % 2].record(stream)
            stream.wait_stream(d2h_stream)  # the run ends when every output is on the host

        w0 = torch.cuda.Event()
        w0.record(stream)
        e2e_run(1, w0)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(e2e_steps, e0)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world)
        e2e_val = sum_over_ranks(flops_step * e2e_steps, world) / e2e_s / 1e12
        h2d = 2 * (M_max * K_DIM + N_DIM) + w_src.numel() * w_src.element_size()
        d2h = sum(2 * M * N_DIM for M in Ms)
        e2e = {"value": round(e2e_val, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps}

    sweeps = None
    if not args.headline_only and not args.m_list:
        sweeps = extra_sweeps(flush_buf, stream, peaks, reps=args.sweep_reps)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * kernel_s / args.steps, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "M_sweep": Ms, "K": K_DIM, "N": N_DIM,
                           "out_dtype": "bf16", "accumulate": "fp32",
                           "weight": ("packed once with bi_pack_weight before timing (same bits as the "
                                      "plain [4096,14336] weight)" if args.weight == "packed"
                                      else "plain row-major [4096,14336]"),
                           "l2": "flushed before every timed launch: 512 MB written then read back (L2 cold and clean)",
                           "timing": ("CUDA events around each launch on its stream; flush excluded; per point "
                                      "the median launch with p10 / p90; value = all FLOP / all launch time"),
                           "wall_s_timed_region": round(t_wall, 3)},
                "row0_bit_equal_all_M": row0_equal,
                "packed_equals_plain_all_M": packed_equals_plain,
                "cublas_row0_bit_equal_all_M": cublas_row0,
                "sweep": sweep,
                "roofline": roof,
                "gpu_launches": gpu_launches,
                "clocks": clocks.summary(),
                "e2e": e2e,
                "cpu_baseline": cpu,
                "peaks": peaks,
                "sweeps": sweeps}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other workloads and the cuBLAS/cuDNN comparison")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip the cuBLAS comparison and the end-to-end pass (for profiling)")
    ap.add_argument("--only", choices=["square", "conv", "attention", "heads", "tiny", "fp16", "rows"],
                    default=None,
                    help="measure only this workload (no headline line; for profiling)")
    ap.add_argument("--weight", choices=["packed", "plain"], default="plain",
                    help="weight path of the timed step (the other one is measured alongside)")
    ap.add_argument("--sweep-reps", type=int, default=50,
                    help="launches per point of the other workloads (tiny mm: 20x this)")
    ap.add_argument("--m-list", type=str, default=None,
                    help="comma-separated subset of the M sweep (for profiling one launch shape)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    rank, local, world = dist_init()
    if args.only:
        run_only(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
