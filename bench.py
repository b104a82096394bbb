"""Benchmark of the GB300 blocked GEMM library; prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload bf16_8192|bf16_4096|tf32_4096|exact_4096|f16acc_4096|bf16_skinny|
                               ragged_216|softmax_<M>x<N>]
                    [--sustain-s S] [--no-configs]

A step is one C = A @ B over one batch of seeded synthetic inputs already resident
in HBM. Default workload: bf16 M = N = K = 8192, A row-major, B column-major,
values N(0, 1)/sqrt(K), fp32 accumulation, bf16 output. Inputs total 256 MB per
step (larger than the 129 MB L2) and rotate over three buffer sets.

``value`` is whole-job TFLOP/s (2*M*N*K per step, all ranks) over the device-timed
region of K steps; ``roofline`` divides the dominant kernel's algorithmic FLOPs (or bytes,
for the memory-bound skinny shape) by its mean CUDA-event duration (events recorded by the
library around that kernel alone, after any staging copies); ``kernel_ms`` gives its mean,
median, min and p90. ``sustained`` runs the same product back to back for a few seconds
(whatever K is) with a 50 ms clock sampler, against the sustained cuBLAS figure. ``configs``
measures the other workloads of the target in the same run (bf16 4096^3, fp32 4096^3 in
tf32 and in exact mode, the skinny bf16 16384x128x8192, and the 216-product ragged sweep),
each with its own roofline and CPU-oracle baseline. ``e2e`` repeats the headline metric
through host buffers (pinned host -> device copies of A and B, the GEMM, and the copy of C
back, every step); ``cpu_baseline`` times the fp64 CPU oracle on a bounded sample (all
cores, plus one thread on a row slab, extrapolated to the whole product).

``--impl reference`` times the CPU oracle itself (the only reference this method has)
on the same workload, one bounded sample per step.
Under torchrun (N > 1) every rank runs its own replica on its own GPU (the product is
single-GPU; there is no data-path collective), and the timing is the max over ranks.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "GEMM TFLOP/s and % of GB300 dense tensor peak (1 GPU) vs CPU oracle"
DATASHEET_BF16_TFLOPS = 2250.0  # dense bf16, NVIDIA GB300 (nominal)
TF32_OVER_BF16 = 1100.0 / 2250.0  # nominal dense tf32 / bf16 ratio
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "dense_tiled_gemm_05_gb300", "csrc")
# sources of the CTA-pair tensor-core kernel (bf16/fp16/tf32)
TC_SOURCES = [os.path.join(CSRC, f) for f in ("tc2_kernel.cu", "tc_common.cuh", "ptx.cuh",
                                              "sk_schedule.h")]
# sources of the chunked kernel (exact fp32 on split tf32 operands)
CHUNK_SOURCES = [os.path.join(CSRC, f) for f in ("tc_chunk_kernel.cu", "tc_common.cuh",
                                                 "ptx.cuh", "sk_schedule.h")]


def _profile(name):
    return os.path.join(ROOT, "profiles", name)


# committed ncu summaries whose per-launch DRAM bytes the roofline's `traffic` reports,
# with the sources of the kernel each was taken on
PROFILES = {"bf16_8192": (_profile("tc2_gemm_cta_pair_bf16_8192.md"), TC_SOURCES),
            "bf16_skinny": (_profile("tc2_gemm_cta_pair_bf16_skinny_16384x128x8192.md"),
                            TC_SOURCES),
            "bf16_4096": (_profile("tc2_gemm_cta_pair_bf16_4096.md"), TC_SOURCES),
            "tf32_4096": (_profile("tc2_gemm_cta_pair_tf32_4096.md"), TC_SOURCES),
            "exact_4096": (_profile("tc_chunk_exact_fp32_4096.md"), CHUNK_SOURCES)}


def max_over_ranks(value, dist=None, device=None):
    """The largest `value` over all ranks (the slowest replica's time); `value` itself on
    one process. Replicas share nothing else: the product is not sharded."""
    if dist is None:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, elapsed_ms):
    """Whole-job rate: the units every rank processed, over the slowest rank's time."""
    return units_per_rank * world / (elapsed_ms / 1e3)


def workload(name):
    """(problem, description, bound) for a named workload."""
    if name == "bf16_8192":
        return (W.bf16_square(8192, seed=5),
                "bf16 GEMM M=N=K=8192, A row-major, B column-major, N(0,1)/sqrt(K), "
                "fp32 accumulate, bf16 out", "tensor")
    if name == "bf16_4096":
        return (W.bf16_square(4096), "bf16 GEMM M=N=K=4096, A row-major, B column-major, "
                "N(0,1)/sqrt(K), fp32 accumulate, bf16 out", "tensor")
    if name == "tf32_4096":
        return (W.fp32_square(4096, "tf32"), "fp32 GEMM M=N=K=4096 row-major, U[-1,1], tf32 "
                "mode, fp32 out", "tensor")
    if name == "exact_4096":
        return (W.fp32_square(4096, "exact"), "fp32 GEMM M=N=K=4096 row-major, U[-1,1], "
                "exact-fp32 mode (split-tf32, three tensor-core products), fp32 out",
                "tensor_x3")
    if name == "f16acc_4096":
        return (W.f16acc_square(4096), "fp16 GEMM M=N=K=4096, A row-major, B column-major, "
                "N(0,1)*0.1, fp16 accumulator rounded every 16 K (section 13.3), fp16 out",
                "tensor")
    if name == "bf16_skinny":
        return (W.bf16_skinny(), "bf16 GEMM M=16384 N=128 K=8192, A row-major, B column-major, "
                "N(0,1)/sqrt(K), fp32 accumulate, bf16 out (memory-bound)", "hbm")
    raise SystemExit("unknown workload %s" % name)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK, "fallback"


def algorithmic_bytes(p):
    es = p.A.element_size()
    return p.M * p.K * es + p.K * p.N * es + p.M * p.N * W.TORCH_DTYPES[p.out_dtype].itemsize


def sources_hash(sources):
    h = hashlib.sha256()
    for f in sources:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def profile_traffic(workload):
    """dram bytes per launch from the workload's committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    entry = PROFILES.get(workload)
    if entry is None or not os.path.exists(entry[0]):
        return None
    path, sources = entry
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not s:
        return None
    return float(m.group(1)) if s.group(1) == sources_hash(sources) else None


class ClockSampler:
    """nvidia-smi clock/throttle samples every `period_ms` while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    LOADED_W = 300.0  # samples drawing more than this are taken as "under load"

    def __init__(self, device, period_ms=200):
        self.device = device
        self.period_ms = period_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms), "-i", str(self.device)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.samples = parse_clock_samples(out)
        return False

    def summary(self):
        return clock_summary(getattr(self, "samples", []), self.period_ms)


def parse_clock_samples(text):
    """Samples from nvidia-smi's csv lines (fields as ClockSampler.FIELDS)."""
    samples = []
    for line in text.splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            continue
        try:
            samples.append({"sm": float(f[1]), "max": float(f[2]), "power": float(f[3]),
                            "hw_slowdown": f[5] == "Active",
                            "hw_thermal_slowdown": f[6] == "Active",
                            "sw_thermal_slowdown": f[7] == "Active",
                            "sw_power_cap": f[8] == "Active"})
        except ValueError:
            continue
    return samples


def clock_summary(samples, period_ms=200, bin_mhz=50):
    """Median SM clock of the samples under load (all samples when none is), the throttle
    reasons seen under load, and the loaded samples binned by SM clock."""
    if not samples:
        return None
    loaded = [x for x in samples if x["power"] > ClockSampler.LOADED_W]
    use = loaded or samples
    reasons = sorted({k for x in use for k in ("hw_slowdown", "hw_thermal_slowdown",
                                               "sw_thermal_slowdown", "sw_power_cap") if x[k]})
    bins = {}
    for x in use:
        lo = int(x["sm"] // bin_mhz * bin_mhz)
        key = "%d-%d" % (lo, lo + bin_mhz - 1)
        bins[key] = bins.get(key, 0) + 1
    return {"sm_mhz": statistics.median(x["sm"] for x in use),
            "sm_max_mhz": max(x["max"] for x in samples), "reasons": reasons,
            "samples": len(samples), "samples_under_load": len(loaded),
            "loaded_filter": "power > %.0f W%s" % (ClockSampler.LOADED_W,
                                                   "" if loaded else " (none: all samples used)"),
            "sampler_period_ms": period_ms,
            "power_w_median_under_load": statistics.median(x["power"] for x in use),
            "power_w_max": max(x["power"] for x in samples),
            "sm_mhz_bins": dict(sorted(bins.items()))}


def percentiles(ms):
    """mean, median, min and p90 of a list of durations (ms)."""
    v = sorted(ms)
    return {"mean": statistics.fmean(v), "median": statistics.median(v), "min": v[0],
            "p90": v[min(len(v) - 1, int(math.ceil(0.9 * len(v))) - 1)], "n": len(v)}


F16ACC_CHUNK = 16  # the library's default fp16-accumulator chunk


def oracle_block(p):
    """f(rows, c): the oracle's values of C[rows, :c] for the workload's arithmetic (the
    fp64 product, or the fp16 accumulator's chunked definition)."""
    import oracle
    a, al, lda = W.storage_numpy(p.A)
    b, bl, ldb = W.storage_numpy(p.B)
    bdt = W.dtype_name(p.B.dtype)
    if p.precision == "f16acc":
        assert al == "row"

        def f(rows, c):
            sub = np.stack([a[i * lda:i * lda + p.K] for i in rows])
            return oracle.gemm_f16acc(sub, b, len(rows), c, p.K, lda=p.K, ldb=ldb,
                                      a_dtype="f16", b_dtype=bdt, BK=F16ACC_CHUNK,
                                      b_layout=bl)
        return f
    kw = dict(lda=lda, ldb=ldb, a_dtype=p.in_dtype, b_dtype=bdt, a_layout=al, b_layout=bl)
    return lambda rows, c: oracle.gemm_f64(a, b, p.M, c, p.K, rows=rows, **kw)


def cpu_baseline(p, target_s=10.0):
    """The oracle as it stands on a bounded sample of output rows (all columns)."""
    import oracle
    f = oracle_block(p)
    # Calibrate: the per-call cost is a fixed part (decoding B) plus a per-row part.
    times = {}
    for r in (4, 12):
        t0 = time.perf_counter()
        f(np.arange(r), p.N)
        times[r] = time.perf_counter() - t0
    per_row = max((times[12] - times[4]) / 8, 1e-6)
    fixed = max(times[4] - 4 * per_row, 0.0)
    rows = int(max(8, min(p.M, (target_s - fixed) / per_row)))
    sel = np.linspace(0, p.M - 1, rows).astype(np.int64)
    t0 = time.perf_counter()
    f(sel, p.N)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * p.N * p.K
    cores = 1 if p.precision == "f16acc" else oracle.num_threads()
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": "%d of %d output rows (all %d columns, K=%d) in fp64, %.1f s, %s"
                      % (rows, p.M, p.N, p.K, dt,
                         "fp16 accumulator, 1 thread" if p.precision == "f16acc" else "OpenMP")}


def run_reference(args, p, desc):
    """--impl reference: the CPU oracle timed per step on a bounded block of the output."""
    import oracle
    f = oracle_block(p)
    # One step computes an r x c block of C over the full K: rows spread over M, and the
    # first c columns of B (same storage and leading dimension, so only they are decoded).
    budget = 120.0 / max(1, args.steps + args.warmup)

    def block(r, c, i0):
        return f((np.arange(r) * 7919 + i0) % p.M, c)

    r = c = 32
    t0 = time.perf_counter()
    block(r, c, 0)
    t1 = time.perf_counter() - t0
    scale = max(1.0, budget / max(t1, 1e-4))
    r = int(max(1, min(p.M, r * scale ** 0.5)))
    c = int(max(1, min(p.N, c * scale ** 0.5)))
    for i in range(args.warmup):
        block(r, c, i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        block(r, c, 1000 + i)
    dt = time.perf_counter() - t0
    flops = 2.0 * r * c * p.K * args.steps
    value = flops / dt / 1e12
    f16acc = p.precision == "f16acc"
    cores = 1 if f16acc else oracle.num_threads()
    sample = "per step a %d x %d block of C over K=%d, %s" % (
        r, c, p.K, "fp16-accumulator oracle, 1 thread" if f16acc else "fp64 oracle, OpenMP")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc, "M": p.M, "N": p.N, "K": p.K},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


SOFTMAX_METRIC = "row softmax HBM GB/s (M x N fp32 in and out; one read and one write)"


def softmax_workload(name):
    """(M, N, description) of a row-softmax workload name 'softmax_<M>x<N>'."""
    M, N = (int(v) for v in name[len("softmax_"):].split("x"))
    return M, N, ("row softmax of an fp32 %d x %d matrix, N(0,1)*3 entries, fp32 out "
                  "(Lesson 4, homework 4)" % (M, N))


def softmax_input(M, N, seed=7):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(M, N, generator=gen) * 3.0


def softmax_oracle_rate(x, target_s):
    """Oracle GB/s on whole rows, as many as fit about target_s seconds (1 thread)."""
    import oracle
    M, N = x.shape
    flat = x.numpy().reshape(-1)
    r = 1
    while True:
        t0 = time.perf_counter()
        oracle.softmax_rows(flat[:r * N], r, N, ldx=N, x_dtype="f32")
        dt = time.perf_counter() - t0
        if dt >= target_s or r >= M:
            return r, dt, 8.0 * r * N / dt / 1e9
        r = min(M, max(r + 1, int(r * min(8.0, 1.5 * target_s / max(dt, 1e-4)))))


def run_softmax(args):
    """The row-softmax workload: one step = softmax of one M x N matrix, inputs resident,
    rotated over buffer sets larger than L2."""
    M, N, desc = softmax_workload(args.workload)
    x_cpu = softmax_input(M, N)
    byts = 8.0 * M * N  # fp32 read + fp32 write
    if args.impl == "reference":
        r, dt, rate = softmax_oracle_rate(x_cpu, 100.0 / max(1, args.steps + args.warmup))
        sample = "per step %d of %d rows (N=%d), fp64 oracle, 1 thread" % (r, M, N)
        print(json.dumps({
            "impl": "reference", "metric": SOFTMAX_METRIC, "value": rate, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc, "M": M, "N": N},
            "cpu_baseline": {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    import dense_tiled_gemm_05_gb300 as g
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    h = g.Gemm(0)
    stream = torch.cuda.current_stream(dev)
    xs = [x_cpu.to(dev) for _ in range(max(1, args.rotate))]
    ys = [torch.empty_like(xs[0]) for _ in xs]
    for i in range(args.warmup):
        h.softmax_rows(xs[i % len(xs)], out=ys[i % len(xs)])
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = h.launch_count()
    with ClockSampler(0) as clocks:
        t0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            h.softmax_rows(xs[i % len(xs)], out=ys[i % len(xs)])
            ends[i].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    launches = h.launch_count() - launches0
    elapsed_ms = t0.elapsed_time(t1)
    kernel_ms = statistics.fmean(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends))
    value = byts * args.steps / (elapsed_ms / 1e3) / 1e9
    peaks, peak_src = measured_peaks()
    achieved = byts / (kernel_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": None,
            "peak_source": "%s hbm_gbs (copy)" % peak_src}
    e2e = None
    if not args.no_e2e:  # pinned host matrix in, softmax, result back, every step
        hx = x_cpu.pin_memory()
        hy = torch.empty_like(hx).pin_memory()
        dx, dy = xs[0], ys[0]
        for _ in range(3):
            dx.copy_(hx, non_blocking=True)
            h.softmax_rows(dx, out=dy)
            hy.copy_(dy, non_blocking=True)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            dx.copy_(hx, non_blocking=True)
            h.softmax_rows(dx, out=dy)
            hy.copy_(dy, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = e0.elapsed_time(e1)
        e2e = {"value": byts * args.e2e_steps / (e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hx.numel() * 4, "d2h_bytes_per_step": hy.numel() * 4,
               "ms_per_step": e_ms / args.e2e_steps}
    if h.status() != 0:
        raise SystemExit("device status error")
    line = {
        "metric": SOFTMAX_METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": desc, "M": M, "N": N,
                   "l2": "inputs larger than L2, rotated over %d buffer sets" % len(xs),
                   "parallelism": "single GPU"},
        "roofline": roof, "clocks": clocks.summary(), "e2e": e2e, "gpu_launches": launches,
    }
    if not args.no_cpu_baseline:
        r, dt, rate = softmax_oracle_rate(x_cpu, 10.0)
        line["cpu_baseline"] = {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": "%d of %d rows (N=%d) in fp64, %.1f s, 1 thread"
                                          % (r, M, N, dt)}
    print(json.dumps(line), flush=True)
    h.close()


RAGGED_DESC = ("ragged-edge sweep: fp16 A[M,K] @ B[K,N], fp32 out, all 216 combinations of "
               "M, N, K in {1,17,127,1000,1023,1025}, U[-1,1], row-major, tight leading dims")


def ragged_reference(args, probs, flops):
    """--impl reference for the ragged sweep: the oracle over as many products as fit."""
    import oracle
    t0 = time.perf_counter()
    done = 0.0
    budget = 100.0 / max(1, args.steps + args.warmup)
    for p in probs:
        a, al, lda = W.storage_numpy(p.A)
        b, bl, ldb = W.storage_numpy(p.B)
        oracle.gemm_f64(a, b, p.M, p.N, p.K, lda=lda, ldb=ldb, a_dtype="f16", b_dtype="f16",
                        a_layout=al, b_layout=bl)
        done += 2.0 * p.M * p.N * p.K
        if time.perf_counter() - t0 > budget:
            break
    dt = time.perf_counter() - t0
    rate = done / dt / 1e12
    return {"impl": "reference", "metric": METRIC, "value": rate, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": RAGGED_DESC},
            "cpu_baseline": {"value": rate, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": "%.3g of %.3g flops of the sweep"
                                                         % (done, flops)},
            "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def ragged_measure(g, dev, steps, warmup, peaks, peak_src, period_ms=200, cpu_s=0.0):
    """The ragged-edge sweep on the GPU: one step runs all 216 products (inputs resident),
    replayed from one CUDA graph; returns the measurement as a dict."""
    probs = [W.ragged(M, N, K) for (M, N, K) in W.ragged_combos()]
    flops = sum(2.0 * p.M * p.N * p.K for p in probs)
    h = g.Gemm(dev.index)
    stream = torch.cuda.current_stream(dev)
    ops = [(p.A.to(dev), p.B.to(dev), torch.empty((p.M, p.N), device=dev)) for p in probs]

    def step():
        for a, b, c in ops:
            h.matmul(a, b, out=c)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    # The sweep is launch-bound (hundreds of small products): capture one step in a CUDA
    # graph and replay it, so the host's per-call cost is not what is measured.
    graph = torch.cuda.CUDAGraph()
    launches0 = h.launch_count()
    with torch.cuda.graph(graph):
        step()
    per_step = h.launch_count() - launches0
    graph.replay()
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(dev.index, period_ms) as clocks:
        ev[0].record(stream)
        for i in range(steps):
            graph.replay()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    if h.status() != 0:
        raise SystemExit("device status error in the ragged sweep")
    elapsed_ms = ev[0].elapsed_time(ev[-1])
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    value = flops * steps / (elapsed_ms / 1e3) / 1e12
    out = {"workload": RAGGED_DESC, "value": value, "unit": "TFLOP/s", "steps": steps,
           "ms_per_step": elapsed_ms / steps, "step_ms": percentiles(step_ms),
           "products_per_step": len(ops), "cuda_graph": True, "dtype": "f16",
           "l2": "inputs of all 216 products resident (489 MB)",
           "roofline": {"bound": "tensor", "achieved": value, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": value / peaks["bf16_tflops"], "traffic": None,
                        "peak_source": "%s bf16_tflops (fp16 runs at the bf16 rate); the whole "
                                       "sweep per step (most of the 216 products are too "
                                       "small to fill the GPU)" % peak_src},
           "clocks": clocks.summary(), "gpu_launches": per_step * steps}
    if cpu_s > 0:
        import oracle
        t0 = time.perf_counter()
        done = 0.0
        for p in probs:
            a, al, lda = W.storage_numpy(p.A)
            b, bl, ldb = W.storage_numpy(p.B)
            oracle.gemm_f64(a, b, p.M, p.N, p.K, lda=lda, ldb=ldb, a_dtype="f16", b_dtype="f16",
                            a_layout=al, b_layout=bl)
            done += 2.0 * p.M * p.N * p.K
            if time.perf_counter() - t0 > cpu_s:
                break
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": done / dt / 1e12, "unit": "TFLOP/s",
                               "cores": oracle.num_threads(), "kind": "oracle",
                               "sample": "the sweep's products in order until %.0f s: %.3g of "
                                         "%.3g flops, fp64, OpenMP" % (cpu_s, done, flops)}
    h.close()
    return out


def run_ragged(args):
    """--workload ragged_216: the sweep alone, as the one JSON line."""
    probs = [W.ragged(M, N, K) for (M, N, K) in W.ragged_combos()]
    flops = sum(2.0 * p.M * p.N * p.K for p in probs)
    if args.impl == "reference":
        print(json.dumps(ragged_reference(args, probs, flops)), flush=True)
        return
    import dense_tiled_gemm_05_gb300 as g
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_src = measured_peaks()
    r = ragged_measure(g, dev, args.steps, args.warmup, peaks, peak_src)
    line = {
        "metric": METRIC, "value": r["value"], "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": RAGGED_DESC, "products_per_step": r["products_per_step"],
                   "cuda_graph": True, "l2": r["l2"], "parallelism": "single GPU"},
        "roofline": r["roofline"], "clocks": r["clocks"], "e2e": None,
        "gpu_launches": r["gpu_launches"],
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GEMM workloads

def resident_sets(p, dev, rotate):
    """`rotate` device copies of the workload's operands (layouts kept) and outputs."""
    a0 = torch.as_strided(torch.empty(p.A.numel(), dtype=p.A.dtype, device=dev), p.A.shape,
                          p.A.stride())
    b0 = torch.as_strided(torch.empty(p.B.numel(), dtype=p.B.dtype, device=dev), p.B.shape,
                          p.B.stride())
    a0.copy_(p.A)
    b0.copy_(p.B)
    sets = [(a0, b0)]
    for _ in range(1, max(1, rotate)):
        a1 = torch.empty_strided(a0.shape, a0.stride(), dtype=a0.dtype, device=dev)
        b1 = torch.empty_strided(b0.shape, b0.stride(), dtype=b0.dtype, device=dev)
        a1.copy_(a0)
        b1.copy_(b0)
        sets.append((a1, b1))
    out_dt = W.TORCH_DTYPES[p.out_dtype]
    outs = [torch.empty((p.M, p.N), dtype=out_dt, device=dev) for _ in sets]
    return sets, outs


def sets_for_l2(p, dev, at_least=3):
    """Buffer sets to rotate so that the operands of consecutive steps exceed twice L2."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (129 << 20)
    per_set = p.A.numel() * p.A.element_size() + p.B.numel() * p.B.element_size()
    return max(at_least, int(math.ceil(2.0 * l2 / per_set)) + 1)


def timed_steps(h, step, n, stream, dev, period_ms=200, dist=None, events=True):
    """Run `n` steps back to back on `stream` under the clock sampler. With `events`, each
    step is bracketed by events and the library records a second pair around the GEMM
    kernel alone (after any staging copies); without, only the region is timed, so the
    host's per-step event calls cannot hold back short kernels. Returns (elapsed ms of the
    region, per-step ms, per-kernel ms, launches, clock summary)."""
    m = n if events else 0
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(m)] for _ in range(4)]
    for e in ev[2] + ev[3]:
        e.record(stream)  # the library needs the CUDA events to exist already
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    launches0 = h.launch_count()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index, period_ms) as clocks:
        # an NVTX range marks the timed region for a timeline profiler (no-op without one)
        torch.cuda.nvtx.range_push("timed steps (%d%s)" % (n, ", per-step events" if events else ""))
        t0.record(stream)
        if events:
            for i in range(n):
                h.set_kernel_events(ev[2][i], ev[3][i])
                ev[0][i].record(stream)
                step(i)
                ev[1][i].record(stream)
        else:
            for i in range(n):
                step(i)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_pop()
    h.set_kernel_events()
    if dist:
        dist.barrier()
    launches = h.launch_count() - launches0
    step_ms = [a.elapsed_time(b) for a, b in zip(ev[0], ev[1])]
    kernel_ms = [a.elapsed_time(b) for a, b in zip(ev[2], ev[3])]
    return t0.elapsed_time(t1), step_ms, kernel_ms, launches, clocks.summary()


def kernel_duration(region_ms, steps, launches, kernel_ms_mean):
    """The dominant kernel's average duration for the roofline, and how it was taken. When
    every step is that one kernel (no staging copies), the timed region's events divided by
    the launches: back to back, each launch's prologue overlaps the previous launch's tail,
    which events recorded between launches would prevent. Otherwise the mean of the events
    the library records around that kernel alone."""
    if launches == steps:
        return region_ms / steps, "timed region / launches (one kernel per step, back to back)"
    return kernel_ms_mean, "events around the kernel alone (after its staging copies), mean"


def roofline(p, bound, workload_name, kernel_ms, peaks, peak_src, sustained_peak):
    """Roofline of the dominant kernel: algorithmic flops (or bytes) per launch over its
    mean event-timed duration, against the measured peak for its dtype and bound."""
    flops = 2.0 * p.M * p.N * p.K
    if bound == "hbm":
        achieved = algorithmic_bytes(p) / (kernel_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profile_traffic(workload_name),
                "peak_source": "%s hbm_gbs (copy)" % peak_src,
                "algorithmic_bytes_per_launch": algorithmic_bytes(p),
                "tflops": flops / (kernel_ms / 1e3) / 1e12}
    achieved = flops / (kernel_ms / 1e3) / 1e12
    scale, note = 1.0, ""
    if p.in_dtype == "f32":
        scale *= TF32_OVER_BF16
        note += " x nominal tf32/bf16 ratio %.3f" % TF32_OVER_BF16
    if bound == "tensor_x3":  # exact fp32: three tf32 products per useful product
        scale /= 3.0
        note += " / 3 (three tf32 products per fp32 product)"
    burst = peaks["bf16_tflops"] * scale
    sustained = peaks["bf16_tflops_sustained"] * scale
    peak = sustained if sustained_peak else burst
    src = ("%s bf16_tflops_sustained (cuBLAS, seconds-long loop under the power cap)"
           if sustained_peak else "%s bf16_tflops (cuBLAS burst)") % peak_src
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": profile_traffic(workload_name),
            "peak_source": src + note, "frac_of_burst": achieved / burst,
            "frac_of_sustained": achieved / sustained,
            "algorithmic_flops_per_launch": flops}


def datasheet_peak(in_dtype, bound):
    """The datasheet's dense peak for a product's input type, TFLOP/s: bf16/fp16 2250 (at
    the 2070 MHz maximum clock), tf32 1100 for fp32 inputs, and a third of that for exact
    fp32, which runs three tf32 products per fp32 product."""
    ds = DATASHEET_BF16_TFLOPS * (TF32_OVER_BF16 if in_dtype == "f32" else 1.0)
    return ds / 3.0 if bound == "tensor_x3" else ds


def kernel_name(h, a, b, p):
    plan = h.plan(a, b, out_dtype=p.out_dtype, precision=p.precision)
    if plan["path"] == "tcgen05_3xtf32":
        return "tc_chunk_kernel (exact fp32, split tf32, CTA pairs)", plan
    if plan["path"] == "fma":
        return "fma_gemm_kernel", plan
    return ("tc2_gemm_kernel (CTA pair)" if plan["cta_pair"] else "tc_gemm_kernel (single CTA)"), plan


def measure_config(g, dev, name, peaks, peak_src, min_s=0.3, cpu_s=3.0, hot_l2=False):
    """One workload of the target measured in the default run: warm-up, then steps for
    about `min_s` seconds (at least 50), inputs rotated over buffer sets larger than L2
    (with `hot_l2`, also a labelled run on one buffer set, its operands resident in L2)."""
    p, desc, bound = workload(name)
    h = g.Gemm(dev.index)
    stream = torch.cuda.current_stream(dev)
    sets, outs = resident_sets(p, dev, sets_for_l2(p, dev))

    def step(i):
        a, b = sets[i % len(sets)]
        h.matmul(a, b, out=outs[i % len(sets)], precision=p.precision, stream=stream)

    for i in range(10):
        step(i)
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    for i in range(10):
        step(i)
    torch.cuda.synchronize(dev)
    est_ms = (time.perf_counter() - t) * 100.0
    n = int(min(5000, max(50, math.ceil(min_s * 1e3 / max(est_ms, 1e-3)))))
    elapsed_ms, _, _, launches, clocks = timed_steps(h, step, n, stream, dev, period_ms=50,
                                                     events=False)
    _, step_ms, kern_ms, _, _ = timed_steps(h, step, n, stream, dev, period_ms=50)
    if h.status() != 0:
        raise SystemExit("device status error in config %s" % name)
    kname, plan = kernel_name(h, sets[0][0], sets[0][1], p)
    kp = percentiles(kern_ms)
    flops = 2.0 * p.M * p.N * p.K
    k_ms, k_how = kernel_duration(elapsed_ms, n, launches, kp["mean"])
    roof = roofline(p, bound, name, k_ms, peaks, peak_src, False)
    roof["kernel_ms"], roof["kernel_ms_from"] = k_ms, k_how
    roof["frac_event_bracketed"] = roofline(p, bound, name, kp["mean"], peaks, peak_src,
                                            False)["frac"]
    out = {"workload": desc, "value": flops * n / (elapsed_ms / 1e3) / 1e12, "unit": "TFLOP/s",
           "steps": n, "ms_per_step": elapsed_ms / n, "step_ms": percentiles(step_ms),
           "kernel": kname, "kernel_ms": kp,
           "kernel_share_of_step": kp["mean"] / statistics.fmean(step_ms),
           "staging_launches_per_step": (launches - n) / n,
           "plan": {k: plan[k] for k in ("path", "tile_m", "tile_n", "ctas", "split_tiles",
                                         "stage_a", "stage_b")},
           "roofline": roof,
           "clocks": clocks, "gpu_launches": launches,
           "l2": "inputs larger than L2: %d buffer sets rotated" % len(sets),
           "dtype": {"bf16": "bf16", "f32": "tf32" if p.precision == "tf32" else "f32"}[p.in_dtype]}
    if bound == "hbm":
        out["hbm_gbs"] = algorithmic_bytes(p) * n / (elapsed_ms / 1e3) / 1e9
    else:
        ds = datasheet_peak(p.in_dtype, bound)
        out["datasheet_peak_tflops"] = ds
        out["pct_of_datasheet_peak"] = 100.0 * out["value"] / ds
    if hot_l2:
        # the same operands every step (they stay in L2): labelled, not the config's value
        def hot(i):
            h.matmul(sets[0][0], sets[0][1], out=outs[0], precision=p.precision, stream=stream)
        for i in range(10):
            hot(i)
        hot_ms, _, _, _, hot_clocks = timed_steps(h, hot, n, stream, dev, period_ms=50,
                                                  events=False)
        out["hot_l2"] = {"value": flops * n / (hot_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                         "ms_per_step": hot_ms / n, "steps": n,
                         "l2": "one buffer set: operands resident in L2 across steps",
                         "sm_mhz": hot_clocks.get("sm_mhz")}
    if cpu_s > 0:
        out["cpu_baseline"] = cpu_baseline(p, target_s=cpu_s)
    h.close()
    del sets, outs
    torch.cuda.empty_cache()
    return out


CONFIG_WORKLOADS = ("bf16_4096", "tf32_4096", "exact_4096", "bf16_skinny")


def one_thread_slab(p, target_s=3.0):
    """The oracle on ONE thread over a slab of whole output rows, extrapolated (linearly in
    rows) to the whole product; labelled as extrapolated."""
    import oracle
    a, al, lda = W.storage_numpy(p.A)
    b, bl, ldb = W.storage_numpy(p.B)
    kw = dict(lda=lda, ldb=ldb, a_dtype=p.in_dtype, b_dtype=W.dtype_name(p.B.dtype),
              a_layout=al, b_layout=bl, threads=1)
    rows = 1
    while True:
        t0 = time.perf_counter()
        oracle.gemm_f64(a, b, p.M, p.N, p.K, rows=np.arange(rows), **kw)
        dt = time.perf_counter() - t0
        if dt >= target_s or rows >= p.M:
            break
        rows = min(p.M, max(rows + 1, int(rows * min(8.0, 1.3 * target_s / max(dt, 1e-3)))))
    flops = 2.0 * rows * p.N * p.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": "%d of %d output rows (all %d columns, K=%d) in fp64 on 1 thread, %.1f s"
                      % (rows, p.M, p.N, p.K, dt),
            "extrapolated_full_product_s": dt * p.M / rows,
            "extrapolated": True}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="bf16_8192")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--sustain-s", type=float, default=2.5,
                    help="seconds of back-to-back products for the sustained measurement "
                         "(0: skip)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads measured beside the default one")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--rotate", type=int, default=3)
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload == "ragged_216":
        if world > 1:
            raise SystemExit("the ragged sweep runs on one GPU")
        run_ragged(args)
        return
    if args.workload.startswith("softmax_"):
        if world > 1:
            raise SystemExit("the softmax workload runs on one GPU")
        run_softmax(args)
        return
    p, desc, bound = workload(args.workload)

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, p, desc)), flush=True)
        return

    import dense_tiled_gemm_05_gb300 as g
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local_rank)
    h = g.Gemm(local_rank)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = measured_peaks()
    flops = 2.0 * p.M * p.N * p.K

    # Inputs resident in HBM: `rotate` buffer sets so consecutive steps do not hit in L2.
    sets, outs = resident_sets(p, dev, args.rotate)

    def step(i):
        a, b = sets[i % len(sets)]
        h.matmul(a, b, out=outs[i % len(sets)], precision=p.precision, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if h.status() != 0:
        raise SystemExit("device status error during warm-up")

    # The timed region: K steps back to back. Then the same K steps again with per-step
    # events around each step and around its GEMM kernel, for the kernel's own duration.
    elapsed_ms, _, _, launches, clocks = timed_steps(h, step, args.steps, stream, dev,
                                                     dist=dist, events=False)
    _, step_ms, kern_ms, _, _ = timed_steps(h, step, args.steps, stream, dev, dist=dist)
    if h.status() != 0:
        raise SystemExit("device status error in the timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    kp = percentiles(kern_ms)
    value = job_rate(flops * args.steps, world, elapsed_ms) / 1e12
    # A region of a second or more runs under the power cap: the sustained cuBLAS figure
    # is its denominator; shorter regions use the burst figure.
    long_run = elapsed_ms >= 1000.0
    k_ms, k_how = kernel_duration(elapsed_ms, args.steps, launches, kp["mean"])
    roof = roofline(p, bound, args.workload, k_ms, peaks, peak_src, long_run)
    roof["peak_source"] += "; timed region %.3f s" % (elapsed_ms / 1e3)
    roof["kernel_ms"], roof["kernel_ms_from"] = k_ms, k_how
    roof["frac_event_bracketed"] = roofline(p, bound, args.workload, kp["mean"], peaks,
                                            peak_src, long_run)["frac"]

    # The same product back to back for seconds, whatever --steps is: the steady state
    # under the power cap, with a 50 ms clock record.
    sustained = None
    if args.sustain_s > 0:
        n = int(max(args.steps, math.ceil(args.sustain_s * 1e3 / max(kp["median"], 1e-3))))
        s_ms, s_step, s_kern, s_launch, s_clocks = timed_steps(h, step, n, stream, dev,
                                                               period_ms=50, dist=dist)
        if h.status() != 0:
            raise SystemExit("device status error in the sustained region")
        s_ms = max_over_ranks(s_ms, dist, dev)
        skp = percentiles(s_kern)
        s_roof = roofline(p, bound, args.workload, skp["mean"], peaks, peak_src, True)
        s_roof["kernel_ms"] = skp["mean"]
        s_roof["kernel_ms_from"] = "events around each kernel, mean"
        sustained = {"steps": n, "seconds": s_ms / 1e3,
                     "value": job_rate(flops * n, world, s_ms) / 1e12, "unit": "TFLOP/s",
                     "ms_per_step": s_ms / n, "step_ms": percentiles(s_step), "kernel_ms": skp,
                     "roofline": s_roof, "clocks": s_clocks, "gpu_launches": s_launch}
        if s_clocks and s_clocks.get("samples_under_load"):
            # clock-normalised cost of one kernel: ms x median MHz = millions of SM cycles
            sustained["kernel_mcycles_at_median_clock"] = skp["mean"] * s_clocks["sm_mhz"] / 1e3
            sustained["value_at_max_clock"] = (sustained["value"] * s_clocks["sm_max_mhz"]
                                               / s_clocks["sm_mhz"])

    # End to end through host buffers: pinned A, B in, C out, every step.
    e2e = None
    if not args.no_e2e:
        out_dt = W.TORCH_DTYPES[p.out_dtype]
        ha = torch.empty_strided(p.A.shape, p.A.stride(), dtype=p.A.dtype, pin_memory=True)
        hb = torch.empty_strided(p.B.shape, p.B.stride(), dtype=p.B.dtype, pin_memory=True)
        ha.copy_(p.A)
        hb.copy_(p.B)
        hc = torch.empty((p.M, p.N), dtype=out_dt, pin_memory=True)
        for _ in range(10):
            h.matmul_host(ha, hb, out=hc, precision=p.precision)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        e0.record(stream)
        for _ in range(args.e2e_steps):
            h.matmul_host(ha, hb, out=hc, precision=p.precision)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = e0.elapsed_time(e1)
        e_ms = max_over_ranks(e_ms, dist, dev)
        if h.status() != 0:
            raise SystemExit("device status error in the e2e region")
        e2e = {"value": job_rate(flops * args.e2e_steps, world, e_ms) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": ha.numel() * ha.element_size() + hb.numel() * hb.element_size(),
               "d2h_bytes_per_step": hc.numel() * hc.element_size(),
               "ms_per_step": e_ms / args.e2e_steps}

    kname, plan = kernel_name(h, sets[0][0], sets[0][1], p)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "f16": "f16", "f32": "tf32" if p.precision == "tf32" else "f32"}[
            p.in_dtype],
        "data": "synthetic",
        "config": {"workload": desc, "M": p.M, "N": p.N, "K": p.K,
                   "l2": "inputs larger than L2, rotated over %d buffer sets" % len(sets),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_datasheet_bf16_peak": 100.0 * value / world / DATASHEET_BF16_TFLOPS,
        "kernel": kname,
        "kernel_ms": kp,
        "step_ms": percentiles(step_ms),
        "roofline": roof,
        "clocks": clocks,
        "sustained": sustained,
        "e2e": e2e,
        "gpu_launches": launches,
    }
    del sets, outs
    torch.cuda.empty_cache()
    # The target's other workloads, each measured on its own (rank 0 of a single-GPU run).
    if rank == 0 and world == 1 and not args.no_configs and args.workload == "bf16_8192":
        cpu_s = 0.0 if args.no_cpu_baseline else 3.0
        configs = {}
        for name in CONFIG_WORKLOADS:
            configs[name] = measure_config(g, dev, name, peaks, peak_src, cpu_s=cpu_s,
                                           hot_l2=name == "bf16_4096")
        configs["ragged_216"] = ragged_measure(g, dev, 50, 5, peaks, peak_src, period_ms=50,
                                               cpu_s=cpu_s)
        line["configs"] = configs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
        line["cpu_baseline"]["one_thread"] = one_thread_slab(p)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    h.close()


if __name__ == "__main__":
    main()
