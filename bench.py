"""Benchmark of the GB300 blocked GEMM library; prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload bf16_8192|bf16_4096|tf32_4096|exact_4096|f16acc_4096|bf16_skinny|
                               ragged_216|softmax_<M>x<N>]

A step is one C = A @ B over one batch of seeded synthetic inputs already resident
in HBM. Default workload: bf16 M = N = K = 8192, A row-major, B column-major,
values N(0, 1)/sqrt(K), fp32 accumulation, bf16 output. Inputs total 256 MB per
step (larger than the 129 MB L2) and rotate over three buffer sets.

``value`` is whole-job TFLOP/s (2*M*N*K per step, all ranks) over the device-timed
region; ``roofline`` divides the dominant kernel's algorithmic FLOPs (or bytes, for the
memory-bound skinny shape) by its mean CUDA-event duration; ``e2e`` repeats the metric
through host buffers (pinned host -> device copies of A and B, the GEMM, and the copy of
C back, every step); ``cpu_baseline`` times the fp64 CPU oracle on a bounded sample.

``--impl reference`` times the CPU oracle itself (the only reference this method has)
on the same workload, one bounded sample per step.
Under torchrun (N > 1) every rank runs its own replica on its own GPU (the product is
single-GPU; there is no data-path collective), and the timing is the max over ranks.
"""
import argparse
import hashlib
import json
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
# committed ncu summaries whose per-launch DRAM bytes the roofline's `traffic` reports
PROFILES = {"bf16_8192": os.path.join(ROOT, "profiles", "tc2_gemm_cta_pair_bf16_8192.md"),
            "bf16_skinny": os.path.join(ROOT, "profiles",
                                        "tc2_gemm_cta_pair_bf16_skinny_16384x128x8192.md")}
CSRC = os.path.join(ROOT, "dense_tiled_gemm_05_gb300", "csrc")
# sources of the CTA-pair tensor-core kernel both workloads run
TC_SOURCES = [os.path.join(CSRC, f) for f in ("tc2_kernel.cu", "tc_common.cuh", "ptx.cuh",
                                              "sk_schedule.h")]


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


def profile_traffic(workload):
    """dram bytes per launch from the workload's committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = PROFILES.get(workload)
    if path is None or not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not s:
        return None
    h = hashlib.sha256()
    for f in TC_SOURCES:
        h.update(open(f, "rb").read())
    return float(m.group(1)) if s.group(1) == h.hexdigest() else None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.device)],
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
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                self.samples.append({"sm": float(f[1]), "max": float(f[2]), "power": float(f[3]),
                                     "hw_slowdown": f[5] == "Active",
                                     "hw_thermal_slowdown": f[6] == "Active",
                                     "sw_thermal_slowdown": f[7] == "Active",
                                     "sw_power_cap": f[8] == "Active"})
            except ValueError:
                continue
        return False

    def summary(self):
        s = getattr(self, "samples", [])
        if not s:
            return None
        loaded = [x for x in s if x["power"] > 300.0] or s
        reasons = sorted({k for x in loaded for k in ("hw_slowdown", "hw_thermal_slowdown",
                                                      "sw_thermal_slowdown", "sw_power_cap")
                          if x[k]})
        return {"sm_mhz": statistics.median(x["sm"] for x in loaded),
                "sm_max_mhz": max(x["max"] for x in s), "reasons": reasons,
                "samples": len(s), "samples_under_load": len(loaded),
                "power_w_max": max(x["power"] for x in s)}


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


def run_ragged(args):
    """The ragged-edge sweep (fp16 in, fp32 accumulate and out, every M, N, K in
    {1, 17, 127, 1000, 1023, 1025}, row-major, tight leading dimensions): one step runs all
    216 products, inputs resident on the device."""
    combos = W.ragged_combos()
    probs = [W.ragged(M, N, K) for (M, N, K) in combos]
    flops = sum(2.0 * p.M * p.N * p.K for p in probs)
    desc = ("ragged-edge sweep: fp16 A[M,K] @ B[K,N], fp32 out, all 216 combinations of "
            "M, N, K in {1,17,127,1000,1023,1025}, U[-1,1], row-major, tight leading dims")
    if args.impl == "reference":
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
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": rate, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc},
            "cpu_baseline": {"value": rate, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": "%.3g of %.3g flops of the sweep"
                                                         % (done, flops)},
            "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return
    import dense_tiled_gemm_05_gb300 as g
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    h = g.Gemm(0)
    stream = torch.cuda.current_stream(dev)
    ops = [(p.A.to(dev), p.B.to(dev), torch.empty((p.M, p.N), device=dev)) for p in probs]

    def step():
        for a, b, c in ops:
            h.matmul(a, b, out=c)

    for _ in range(args.warmup):
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
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        t0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    launches = per_step * args.steps
    if h.status() != 0:
        raise SystemExit("device status error")
    elapsed_ms = t0.elapsed_time(t1)
    value = flops * args.steps / (elapsed_ms / 1e3) / 1e12
    peaks, peak_src = measured_peaks()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": desc, "products_per_step": len(ops), "cuda_graph": True,
                   "l2": "inputs of all 216 products resident (489 MB)",
                   "parallelism": "single GPU"},
        "roofline": {"bound": "tensor", "achieved": value, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": value / peaks["bf16_tflops"], "traffic": None,
                     "peak_source": "%s bf16_tflops (fp16 runs at the bf16 rate); most of the "
                                    "216 products are too small to fill the GPU" % peak_src},
        "clocks": clocks.summary(), "e2e": None, "gpu_launches": launches,
    }
    print(json.dumps(line), flush=True)
    h.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="bf16_8192")
    ap.add_argument("--e2e-steps", type=int, default=20)
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

    # Inputs resident in HBM: `rotate` buffer sets so consecutive steps do not hit in L2.
    a0 = torch.as_strided(torch.empty(p.A.numel(), dtype=p.A.dtype, device=dev), p.A.shape,
                          p.A.stride())
    b0 = torch.as_strided(torch.empty(p.B.numel(), dtype=p.B.dtype, device=dev), p.B.shape,
                          p.B.stride())
    a0.copy_(p.A)
    b0.copy_(p.B)
    sets = [(a0, b0)]
    for _ in range(1, max(1, args.rotate)):
        a1 = torch.empty_strided(a0.shape, a0.stride(), dtype=a0.dtype, device=dev)
        b1 = torch.empty_strided(b0.shape, b0.stride(), dtype=b0.dtype, device=dev)
        a1.copy_(a0)
        b1.copy_(b0)
        sets.append((a1, b1))
    out_dt = W.TORCH_DTYPES[p.out_dtype]
    outs = [torch.empty((p.M, p.N), dtype=out_dt, device=dev) for _ in sets]

    def step(i):
        a, b = sets[i % len(sets)]
        h.matmul(a, b, out=outs[i % len(sets)], precision=p.precision, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if h.status() != 0:
        raise SystemExit("device status error during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = h.launch_count()
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step(i)
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    launches = h.launch_count() - launches0
    if h.status() != 0:
        raise SystemExit("device status error in the timed region")
    elapsed_ms = t_start.elapsed_time(t_end)
    kernel_ms = statistics.fmean(s.elapsed_time(e) for s, e in zip(starts, ends))
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)

    flops = 2.0 * p.M * p.N * p.K
    value = job_rate(flops * args.steps, world, elapsed_ms) / 1e12
    peaks, peak_src = measured_peaks()
    if bound == "hbm":
        achieved = algorithmic_bytes(p) / (kernel_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": profile_traffic(args.workload),
                "peak_source": "%s hbm_gbs (copy)" % peak_src}
    elif bound == "alu":
        props = torch.cuda.get_device_properties(dev)
        sm_mhz = peaks.get("sm_max_mhz", 2070.0)
        peak = props.multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12
        achieved = flops / (kernel_ms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None,
                "peak_source": "%d SMs x 128 fp32 FMA/clk x 2 x %.0f MHz"
                               % (props.multi_processor_count, sm_mhz)}
    else:
        achieved = flops / (kernel_ms / 1e3) / 1e12
        # The kernel runs back to back for the whole timed region: when that lasts a second
        # or more it runs under the power cap, and the denominator is the sustained cuBLAS
        # figure (measured over a seconds-long loop); shorter regions use the burst figure.
        long_run = elapsed_ms >= 1000.0
        scale = 1.0
        src = ""
        if p.in_dtype == "f32":
            scale *= TF32_OVER_BF16
            src += " x nominal tf32/bf16 ratio %.3f" % TF32_OVER_BF16
        if bound == "tensor_x3":  # exact fp32: three tf32 products per useful product
            scale /= 3.0
            src += " / 3 (three tf32 products per fp32 product)"
        burst = peaks["bf16_tflops"] * scale
        sustained = peaks["bf16_tflops_sustained"] * scale
        peak = sustained if long_run else burst
        src = ("%s bf16_tflops_sustained (cuBLAS, seconds-long loop; this timed region lasted "
               "%.2f s)" % (peak_src, elapsed_ms / 1e3) if long_run else
               "%s bf16_tflops (cuBLAS burst; timed region %.2f s)"
               % (peak_src, elapsed_ms / 1e3)) + src
        traffic = profile_traffic(args.workload)
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "peak_source": src,
                "frac_of_burst": achieved / burst, "frac_of_sustained": achieved / sustained}

    # End to end through host buffers: pinned A, B in, C out, every step.
    e2e = None
    if not args.no_e2e:
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
        "roofline": roof,
        "clocks": clocks.summary(),
        "e2e": e2e,
        "gpu_launches": launches,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    h.close()


if __name__ == "__main__":
    main()
