"""Benchmark of the tovl hot path on GB300.

Headline step: one tovl_gather_gemm call on the tensor-parallel all-gather +
GEMM workload (4 logical shards x 768 rows, M=3072, K=N=4096, bf16), inputs
resident in HBM, L2 flushed before every timed step (the buffers fit in L2).

The JSON line also carries
  acceptance  the platform page's trio: T_comp alone (GEMM-only control, same
              consumer CTA count), T_comm alone (copy-only control, same
              producer CTA count), T_total (fused); overlap efficiency and
              compute interference (consumer span against consumer span, and
              event time against event time)
  roofline    the fused kernel against the measured bf16 dense peak
  e2e         the same metric through the C ABI with host buffers
              (shards in, output out, pinned memory) inside the timed region
  cpu_baseline the CPU oracle as it stands on this host: the whole TP step on
              every core, and per configuration a bounded sample on every core
              and on one thread
  configs     the other workloads: dispatch + grouped GEMM (uniform and Zipf
              routing), combine, GEMM + reduce-scatter and the gated copy
              sweep (GB/s over the configuration's 1000 rounds, signal latency)

Multi-GPU: the path does not shard across GPUs (replicas only); with
--gpus N each rank runs an independent replica and `value` sums the ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused gather+GEMM TFLOP/s & overlap eff. (1 GB300); gated row-copy HBM GB/s"
L2_FLUSH_BYTES = 512 << 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["tovl", "reference"], default="tovl")
    ap.add_argument("--producers", type=int, default=0, help="producer CTAs (0 = library default)")
    ap.add_argument("--k-slices", type=int, default=4, help="K-slices per chunk watermark")
    ap.add_argument("--sweep", action="store_true", help="also sweep the producer CTA count")
    ap.add_argument("--quick", action="store_true", help="skip the extra workloads")
    ap.add_argument("--full", action="store_true", help="extra workloads at their full round counts")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", choices=["fused", "gemm", "copy", "dispatch", "combine", "rs"], default=None,
                    help="run only W + K calls of one kernel on a small case (for ncu captures) and exit")
    ap.add_argument("--dispatch-align", type=int, default=128, choices=[128, 256],
                    help="expert segment alignment of --profile dispatch/combine (256: CTA-pair tiles)")
    ap.add_argument("--no-coop", action="store_true",
                    help="launch fused kernels without the cooperative attribute (profiler replay)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- utilities
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


FUSED_SOURCES = ["ctrl.cuh", "ptx.cuh", "sync.cuh", "common.cuh", "producer.cuh", "consumer.cuh", "fused.cu"]


def kernel_source_sha(files=FUSED_SOURCES) -> str:
    """sha256 over the fused kernel's sources, in a fixed order."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "consumer_movement_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(profile: str):
    """DRAM bytes per launch from an ncu summary under profiles/, if it was
    taken on the current kernel sources (their sha256 is recorded there)."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source-sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram-bytes-per-launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b:
        return None
    return float(m_b.group(1)) if kernel_source_sha() == m_sha.group(1) else None


def dist_init(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle leg
def _with_threads(n, fn):
    """Run fn() with the oracle's OpenMP thread count set to n (restored after)."""
    import oracle
    old = oracle.num_threads()
    oracle.set_num_threads(n)
    try:
        return fn()
    finally:
        oracle.set_num_threads(old)


def cpu_tp_step(cfg, seed: int = 0, rows=None):
    """One TP step of the oracle as it stands: the whole gather, then the fp32
    matmul of `rows` output rows (None: all M rows, the whole step).  Returns
    (seconds, FLOP done)."""
    import numpy as np
    import oracle
    import workloads
    X, W = workloads.gather_inputs(cfg, seed, "cpu")
    shards = [workloads.bf16_bits(X[s]) for s in range(cfg.shards)]
    Wb = workloads.bf16_bits(W)
    t0 = time.perf_counter()
    G = oracle.gather(shards)
    if rows is None:
        oracle.matmul_f32(G, Wb)
        n = cfg.M
    else:
        oracle.matmul_rows_f32(G, Wb, np.asarray(rows, dtype=np.int64))
        n = len(rows)
    return time.perf_counter() - t0, 2.0 * n * cfg.K * cfg.N


def _sample_rows(n_total: int, n: int, seed: int):
    import numpy as np
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(n_total, size=min(n, n_total), replace=False)).astype(np.int64)


def cpu_dispatch_inputs(cfg, seed: int = 0):
    import workloads
    x, topk, W = workloads.dispatch_inputs(cfg, seed, "cpu")
    return workloads.bf16_bits(x), topk, workloads.bf16_bits(W)


def cpu_dispatch_step(cfg, frac: float, inputs):
    """One dispatch round of the oracle on `inputs` (cpu_dispatch_inputs):
    the routing plan, the scatter into padded expert segments, then the
    grouped fp32 matmul of a `frac` share of every expert's rows (1.0: the
    whole round).  Returns (seconds, FLOP done)."""
    import oracle
    xb, topk, Wb = inputs
    t0 = time.perf_counter()
    p = oracle.dispatch_plan(topk, cfg.E)
    D = oracle.dispatch(xb, p.dst, cfg.k, p.m_pad)
    flops = 0.0
    if frac >= 1.0:
        oracle.grouped_matmul_f32(D, Wb, p.off)
        flops = 2.0 * cfg.T * cfg.k * cfg.H * cfg.N
    else:
        for e in range(cfg.E):
            n_e = int(p.counts[e])
            if n_e == 0:
                continue
            rows = _sample_rows(n_e, max(1, int(round(n_e * frac))), e) + int(p.off[e])
            oracle.matmul_rows_f32(D, Wb[e], rows)
            flops += 2.0 * rows.size * cfg.H * cfg.N
    return time.perf_counter() - t0, flops


def cpu_combine_step(cfg, seed: int = 0):
    """The oracle's combine of one dispatch round (staging + gate-weighted
    sums) on seeded expert outputs.  Returns (seconds, interface bytes)."""
    import oracle
    import workloads
    topk = workloads.routing(cfg, seed)
    p = oracle.dispatch_plan(topk, cfg.E)
    Y = workloads.bf16_bits(workloads.bf16_normal((p.m_pad, cfg.N), 1.0, seed + 1, "cpu"))
    w = workloads.gate_weights(cfg.T, cfg.k, seed)
    t0 = time.perf_counter()
    oracle.combine(Y, p.dst, w)
    return time.perf_counter() - t0, 3.0 * cfg.T * cfg.k * cfg.N * 2 + cfg.T * cfg.N * 2


def cpu_copy_step(n_rows: int, row_bytes: int, seed: int = 0):
    """The oracle's permuted copy dst[perm[i]] = src[i].  Returns (seconds, bytes moved)."""
    import numpy as np
    import oracle
    import workloads
    perm = workloads.permutation(n_rows, seed)
    src = np.random.default_rng(seed).integers(0, 256, size=(n_rows, row_bytes), dtype=np.uint8)
    t0 = time.perf_counter()
    oracle.copy_perm(src, perm)
    return time.perf_counter() - t0, 2.0 * n_rows * row_bytes


def cpu_baseline(cfg):
    """The CPU oracle, as it stands, on this host: the whole TP step on every
    core (the headline), then per configuration one bounded sample on every
    core and on one thread.  Each figure is the rate of the work actually
    done; `sample` says what that work was.  The oracle's matmuls are shared
    over output rows with OpenMP; its plan, scatter, combine and copy loops
    are single-threaded whatever the setting."""
    import oracle
    import workloads
    cores = oracle.num_threads()
    t, f = cpu_tp_step(cfg)
    out = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
           "sample": f"one whole TP step (gather + fp32 matmul of all {cfg.M} rows, K=N={cfg.K}) on {cores} "
                     f"threads: {t:.2f} s"}
    per = {}

    rows = _sample_rows(cfg.M, 96, 1)
    t1, f1 = _with_threads(1, lambda: cpu_tp_step(cfg, 1, rows))
    per["tp"] = {"all_cores": {k: out[k] for k in ("value", "unit", "sample")} | {"threads": cores, "seconds": t},
                 "single_thread": {"value": f1 / t1 / 1e12, "unit": "TFLOP/s", "threads": 1, "seconds": t1,
                                   "sample": f"whole gather + fp32 matmul of {rows.size} of {cfg.M} output rows"}}
    for name, dcfg, fr_all, fr_one in (("dispatch_uniform", workloads.DISPATCH, 1 / 4, 1 / 32),
                                       ("dispatch_zipf", workloads.SKEWED, 1 / 16, 1 / 128)):
        legs = {}
        inputs = cpu_dispatch_inputs(dcfg)
        for key, threads, fr in (("all_cores", cores, fr_all), ("single_thread", 1, fr_one)):
            t, f = _with_threads(threads, lambda: cpu_dispatch_step(dcfg, fr, inputs))
            legs[key] = {"value": f / t / 1e12, "unit": "TFLOP/s", "threads": threads, "seconds": t,
                         "sample": f"plan + scatter of the whole round, grouped fp32 matmul of "
                                   f"{'every expert' if fr >= 1 else f'1/{round(1 / fr)} of each expert'}'s rows"}
        per[name] = legs
        del inputs
    for name, dcfg in (("combine_uniform", workloads.DISPATCH), ("combine_zipf", workloads.SKEWED)):
        t, b = cpu_combine_step(dcfg)
        per[name] = {"single_thread": {"value": b / t / 1e9, "unit": "GB/s", "threads": 1, "seconds": t,
                                       "sample": "the whole combine (staging + weighted sums); interface bytes"}}
    n, rb = 1 << 16, 8192
    t, b = cpu_copy_step(n, rb)
    per["gated_copy"] = {"single_thread": {"value": b / t / 1e9, "unit": "GB/s", "threads": 1, "seconds": t,
                                           "sample": f"{n} permuted rows of {rb} B (1/16 of the 2^20-row "
                                                     "sweep's row count, one row size)"}}
    out["configs"] = per
    return out


def run_reference(args):
    """Reference arm: the CPU oracle as it stands, on this host's cores, on
    the TP workload.  Every step is one whole step (gather + fp32 matmul of
    all M rows) when the run fits its time budget; otherwise every step does
    the whole gather and the matmul of a seeded sample of output rows.  Either
    way the reported rate is FLOP actually done / time actually spent, and
    ms_per_step is the measured time of one step as run."""
    import oracle
    import workloads
    rank, world, _ = dist_init(args)
    if rank != 0:
        return
    cfg = workloads.TP
    oracle.build()
    n_steps = args.warmup + args.steps
    budget_s = max(60.0, args.cpu_seconds * 12)        # the whole run, a few minutes at most
    t_full, _ = cpu_tp_step(cfg, 0, _sample_rows(cfg.M, 256, 0))
    est_full = t_full * cfg.M / 256
    rows_per_step = cfg.M if est_full * n_steps <= budget_s else \
        max(8, int(cfg.M * budget_s / (est_full * n_steps)))
    times, flops = [], []
    for i in range(n_steps):
        rows = None if rows_per_step >= cfg.M else _sample_rows(cfg.M, rows_per_step, i)
        t, f = cpu_tp_step(cfg, i, rows)
        if i >= args.warmup:
            times.append(t)
            flops.append(f)
    ms = statistics.mean(times) * 1e3
    value = sum(flops) / sum(times) / 1e12
    sample = (f"every step: the whole TP step (gather + fp32 matmul of all {cfg.M} rows)" if rows_per_step >= cfg.M
              else f"every step: the whole gather + fp32 matmul of {rows_per_step} seeded rows of {cfg.M}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": cfg.name, "parallelism": "replicas only", "l2": "n/a (CPU)",
                   "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU legs
class Timer:
    """CUDA-event timing of single calls on one stream, L2 flushed before each.

    The flush writes a 512 MiB buffer (evicting everything the call used) and
    then reads another 512 MiB buffer, so the L2 is left holding clean lines
    of neither the inputs nor the flush writes: the timed call starts cold
    and does not pay for writing back the flush buffer's dirty lines."""

    def __init__(self, stream):
        import torch
        self.torch = torch
        self.stream = stream
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def do_flush(self):
        self.flush.fill_(1)
        self.flush_read.max()

    def time_calls(self, fn, n: int, flush: bool = True):
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(self.stream):
            for a, b in evs:
                if flush:
                    self.do_flush()
                a.record(self.stream)
                fn()
                b.record(self.stream)
        self.stream.synchronize()
        return [a.elapsed_time(b) for a, b in evs]


def tp_setup(h, cfg, dev):
    import torch
    import workloads
    X, W = workloads.gather_inputs(cfg, 0, dev)
    gathered = torch.empty(cfg.M, cfg.K, dtype=torch.bfloat16, device=dev)
    out = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=dev)
    return X, W, gathered, out


def acceptance(h, timer, cfg, X, W, gathered, out, n: int, producers: int):
    """T_comp alone, T_comm alone and T_total (median ms) plus the consumers'
    span inside the fused kernel, from the kernel's own %globaltimer stamps.
    `producers` is the handle's producer setting (0 = automatic split), put
    back after the controls."""
    from consumer_movement_gemm_gb300 import tovl
    t_total = statistics.median(timer.time_calls(lambda: h.gather_gemm(X, W, gathered, out), n))
    # the controls run with the fused call's split: C consumers alone, P producers alone
    P, C = h.get_option(tovl.OPT_PRODUCERS), h.get_option(tovl.OPT_CONSUMERS)
    h.set_option(tovl.OPT_PRODUCERS, P)
    t_comp = statistics.median(timer.time_calls(lambda: h.gemm_only(gathered, W, out), n))
    t_comm = statistics.median(timer.time_calls(lambda: h.copy_only(X, gathered), n))
    assert h.get_option(tovl.OPT_CONSUMERS) == C
    # the consumer CTAs' span (first consumer start to last consumer end,
    # %globaltimer stamps inside the kernel) of the fused call and of the
    # GEMM-only control, measured the same way
    h.set_option(tovl.OPT_STATS, 1)
    spans, spans_alone = [], []
    for _ in range(min(n, 20)):
        timer.time_calls(lambda: h.gather_gemm(X, W, gathered, out), 1)
        st = h.read_stats()
        spans.append((st[2] - st[1]) / 1e6)
        timer.time_calls(lambda: h.gemm_only(gathered, W, out), 1)
        st = h.read_stats()
        spans_alone.append((st[2] - st[1]) / 1e6)
    h.set_option(tovl.OPT_STATS, 0)
    h.set_option(tovl.OPT_PRODUCERS, producers)
    t_comp_fused = statistics.median(spans)
    t_comp_span = statistics.median(spans_alone)
    overlap = (t_comp + t_comm - t_total) / min(t_comp, t_comm)
    return {
        "T_comp_alone_ms": t_comp, "T_comm_alone_ms": t_comm, "T_total_ms": t_total,
        "T_comp_at_fused_span_ms": t_comp_fused, "T_comp_alone_span_ms": t_comp_span,
        "overlap_efficiency": overlap, "overlap_target": 0.8,
        # like for like: consumer span in the fused call / consumer span of the GEMM-only call
        "compute_interference": t_comp_fused / t_comp_span, "interference_target": 1.1,
        # like for like: CUDA-event time of the fused call / of the GEMM-only call
        "compute_interference_events": t_total / t_comp,
        "interference_note": "compute_interference = consumer span (in-kernel %globaltimer) fused / GEMM-only; "
                             "compute_interference_events = event time fused / GEMM-only (the copy's share "
                             "included)",
        "producer_ctas": P, "consumer_ctas": C,
    }


def unfused_context(timer, cfg, X, W, n: int):
    """For context only, not the product path: the same step without fusion,
    with library kernels on the same GPU -- a torch copy of the shards into
    the gathered buffer (every SM) and a cuBLAS GEMM (torch.matmul), alone
    and back to back (median ms, L2 flushed before each)."""
    import torch
    G = torch.empty(cfg.M, cfg.K, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device="cuda")
    Xf = X.reshape(cfg.M, cfg.K)
    copy = lambda: G.copy_(Xf)  # noqa: E731
    gemm = lambda: torch.matmul(G, W, out=C)  # noqa: E731
    both = lambda: (copy(), gemm())  # noqa: E731
    res = {}
    for name, fn in (("torch_copy_ms", copy), ("cublas_gemm_ms", gemm), ("copy_then_cublas_ms", both)):
        timer.time_calls(fn, 3)
        res[name] = statistics.median(timer.time_calls(fn, n))
    res["note"] = "library kernels on the same GPU for comparison; not part of the timed product path"
    return res


def e2e_tp(h, cfg, W, gathered, out, steps: int, stream):
    """Host shards -> device, fused call, device -> host output, every step.
    Pipelined like a serving loop: two buffer sets and three streams, so the
    upload of step i+1 and the download of step i-1 overlap step i's fused
    call; every step still moves its whole input up and its whole output
    back.  Time = first upload start to last download end, per step."""
    import torch
    import workloads
    X_host = workloads.gather_inputs(cfg, 0, "cpu")[0].pin_memory()
    X_dev = [torch.empty_like(X_host, device="cuda") for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    gath = [gathered, torch.empty_like(gathered)]
    out_host = [torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]      # upload of buffer set b done
    ev_done = [torch.cuda.Event() for _ in range(2)]    # fused call on set b done
    ev_out = [torch.cuda.Event() for _ in range(2)]     # download of set b done

    def step(i):
        b = i % 2
        s_in.wait_event(ev_done[b])                     # set b's last fused call has read X_dev[b]
        with torch.cuda.stream(s_in):
            X_dev[b].copy_(X_host, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])                    # set b's last output has been read back
        h.gather_gemm(X_dev[b], W, gath[b], outs[b], stream=stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            out_host[b].copy_(outs[b], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(i)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    # the last step's downloaded output equals a plain call's on the same input
    with torch.cuda.stream(stream):
        h.gather_gemm(X_dev[0], W, gath[0], outs[0], stream=stream)
    torch.cuda.synchronize()
    verified = bool(torch.equal(out_host[(steps - 1) % 2], outs[0].cpu()))
    return {"value": cfg.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": X_host.numel() * 2, "d2h_bytes_per_step": out_host[0].numel() * 2,
            "pipelined": "upload of step i+1 and download of step i-1 overlap step i (two buffer sets, three streams)",
            "last_output_verified": verified}


def dispatch_bench(cfg, rounds: int, dev, producers: int, k_slices: int, align: int = 128):
    """Dispatch + grouped GEMM: algorithmic TFLOP/s (real rows only).  `align`
    = expert segment alignment (128, the pages' row block; 256 lets CTA pairs
    take 256-row tiles inside one expert)."""
    import numpy as np
    import torch
    import workloads
    from consumer_movement_gemm_gb300 import tovl
    x, topk_np, W = workloads.dispatch_inputs(cfg, 0, dev)
    rows = tovl.dispatch_rows_aligned(cfg.T, cfg.k, cfg.E, align)
    with tovl.Handle(0, max_rows=rows, max_pairs=cfg.T * cfg.k, max_experts=cfg.E, k_slices=k_slices) as h:
        h.set_option(tovl.OPT_DISPATCH_ALIGN, align)
        if producers:
            h.set_option(tovl.OPT_PRODUCERS, producers)
        topk = torch.from_numpy(topk_np).to(dev)
        dispatched = torch.zeros(rows, cfg.H, dtype=torch.bfloat16, device=dev)
        offs = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
        out = torch.empty(rows, cfg.N, dtype=torch.bfloat16, device=dev)
        stream = torch.cuda.current_stream()
        timer = Timer(stream)
        fn = lambda: h.dispatch_grouped_gemm(x, topk, W, dispatched, offs, out)  # noqa: E731
        timer.time_calls(fn, 3)
        ms = statistics.mean(timer.time_calls(fn, rounds))
        assert h.sync_status() == 0
        counts = np.bincount(topk_np.reshape(-1), minlength=cfg.E)
        m_pad = int(offs[-1].item())
        flops = 2.0 * cfg.T * cfg.k * cfg.H * cfg.N
        res = {"workload": cfg.name, "segment_alignment": align, "pair_tiles": bool(h.get_option(tovl.OPT_PAIRS)) and (align == 256 or bool(h.get_option(tovl.OPT_EMBEDDED))),
               "producer_ctas": h.get_option(tovl.OPT_PRODUCERS),
               "embedded_producers": bool(h.get_option(tovl.OPT_EMBEDDED)), "ms_per_round": ms, "TFLOP/s": flops / (ms * 1e-3) / 1e12,
               "algorithmic_GFLOP": flops / 1e9, "padded_rows": m_pad, "max_expert_rows": int(counts.max()),
               "min_expert_rows": int(counts.min()), "rounds": rounds, "l2": "flushed before every round"}
        res["combine"] = combine_bench(h, cfg, out, timer, rounds, dev)
        return res


def combine_bench(h, cfg, y, timer, rounds: int, dev):
    """Combine of the dispatch round just run on `h`: algorithmic bytes =
    expert rows read + staging written + staging read + combined written
    (+ weights), per call, against the measured HBM copy bandwidth."""
    import torch
    import workloads
    T, k, N = cfg.T, cfg.k, cfg.N
    w = torch.from_numpy(workloads.gate_weights(T, k, 0)).to(dev)
    staging = torch.empty(T * k, N, dtype=torch.bfloat16, device=dev)
    combined = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
    fn = lambda: h.combine(y, w, staging, combined)  # noqa: E731
    timer.time_calls(fn, 3)
    ms = statistics.mean(timer.time_calls(fn, rounds))
    assert h.sync_status() == 0
    # every byte at the kernel's interface once: expert rows read, staging
    # written, combined rows written, weights read.  The staging rows are
    # also read back by the reducers, but within the call: that re-read is
    # served by L2 (ncu: the DRAM reads of a call are about the expert rows
    # alone), so it is not counted against HBM
    unique = 2.0 * T * k * N * 2 + T * N * 2 + T * k * 4
    moved = unique + T * k * N * 2
    peaks, _ = measured_peaks()
    gbs = unique / (ms * 1e-3) / 1e9
    return {"ms_per_round": ms, "GB/s": gbs, "unique_MB": unique / 1e6, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "GB/s_incl_L2_reread": moved / (ms * 1e-3) / 1e9, "moved_MB_incl_L2_reread": moved / 1e6,
            "bytes_note": "GB/s and frac_of_hbm count each interface byte once (expert rows read, staging and "
                          "combined rows written); the staging re-read stays in L2 and only appears in "
                          "GB/s_incl_L2_reread",
            "producer_ctas": h.get_option(1), "reducer_ctas": h.get_option(2),
            "copy": "10 copy warps in every CTA, the other 6 reduce" if h.get_option(1) == 0 else "producer CTAs beside reducer CTAs",
            "l2": "flushed before every call (expert outputs start in HBM)"}


def rs_bench(cfg, rounds: int, dev, producers_sweep=(0, 8, 16, 24, 32, 48), role_switch: int = 1):
    """GEMM + reduce-scatter on the TP shape split four ways along K: shard s
    multiplies X_s [M][K/S] by W_s [K/S][N]; the S partials are reduced.
    Algorithmic TFLOP/s = 2*M*N*K / time; reduction GB/s = (S+1)*M*N*2 / time."""
    import torch
    import workloads
    from consumer_movement_gemm_gb300 import tovl
    S, M, K, N = cfg.shards, cfg.M, cfg.K, cfg.N
    Ks = K // S
    X = workloads.bf16_normal((S, M, Ks), 1 / K ** 0.5, 0, dev)
    W = workloads.bf16_normal((S, Ks, N), 1 / K ** 0.5, 1, dev)
    partials = torch.empty(S, M, N, dtype=torch.bfloat16, device=dev)
    out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    res = []
    with tovl.Handle(0, max_rows=1 << 14, k_slices=4) as h:
        timer = Timer(torch.cuda.current_stream())
        for P in producers_sweep:
            h.set_option(tovl.OPT_PRODUCERS, P)
            h.set_option(tovl.OPT_ROLE_SWITCH, role_switch)
            fn = lambda: h.gemm_reduce_scatter(X, W, partials, out)  # noqa: E731
            timer.time_calls(fn, 3)
            ms = statistics.mean(timer.time_calls(fn, rounds))
            assert h.sync_status() == 0
            res.append({"producer_ctas": h.get_option(tovl.OPT_PRODUCERS), "consumer_ctas": h.get_option(tovl.OPT_CONSUMERS),
                        "ms": ms, "TFLOP/s": cfg.flops / (ms * 1e-3) / 1e12,
                        "reduce_GBps": (S + 1) * M * N * 2 / (ms * 1e-3) / 1e9, "auto": P == 0,
                        "role_switch": role_switch})
    best = max(res, key=lambda r: r["TFLOP/s"])
    return {"workload": f"GEMM + reduce-scatter: {S} shards, M={M}, K={K} (K/S={Ks} per shard), N={N}",
            "TFLOP/s": res[0]["TFLOP/s"], "ms_per_round": res[0]["ms"], "producer_ctas": res[0]["producer_ctas"],
            "best_sweep_TFLOP/s": best["TFLOP/s"], "sweep": res, "rounds": rounds,
            "l2": "flushed before every round"}


def copy_sweep(rounds: int, dev, sizes, rounds_other: int = 20):
    """Gated and ungated permuted copies of 2^20 rows at every row size:
    `rounds` timed rounds (sequences advance every gated round) in the default
    automatic mode, `rounds_other` in the vector and bulk modes."""
    import numpy as np
    import torch
    import workloads
    from consumer_movement_gemm_gb300 import tovl
    cfg = workloads.COPY
    n = cfg.n_rows
    perm = torch.from_numpy(workloads.permutation(n, cfg.seed)).to(dev)
    res = []
    big = max(sizes)
    src_all = torch.empty(n * big, dtype=torch.uint8, device=dev)
    dst_all = torch.empty(n * big, dtype=torch.uint8, device=dev)
    src_all.random_(0, 256)
    with tovl.Handle(0, max_rows=n) as h:
        stream = torch.cuda.current_stream()
        timer = Timer(stream)
        for rb in sizes:
            src = src_all[: n * rb].view(n, rb)
            dst = dst_all[: n * rb].view(n, rb)
            for mode in (tovl.TOVL_COPY_AUTO, tovl.TOVL_COPY_VECTOR, tovl.TOVL_COPY_BULK):
                h.set_option(tovl.OPT_COPY_MODE, mode)
                row = {"row_bytes": rb, "copy_mode": {0: "vector", 1: "bulk", 2: "auto"}[mode]}
                nr = rounds if mode == tovl.TOVL_COPY_AUTO else rounds_other
                row["rounds"] = nr
                for gated in (False, True):
                    fn = lambda: h.gated_copy(src, dst, perm, gated=gated)  # noqa: E731
                    timer.time_calls(fn, 2, flush=False)
                    ts = timer.time_calls(fn, nr, flush=False)
                    ms = statistics.median(ts)
                    key = "gated" if gated else "ungated"
                    row[f"{key}_GBps"] = 2.0 * n * rb / (ms * 1e-3) / 1e9
                    row[f"{key}_GBps_mean"] = 2.0 * n * rb / (statistics.mean(ts) * 1e-3) / 1e9
                h.gated_copy(src, dst, perm, gated=True, stamps=True)
                assert h.sync_status() == 0
                pub, obs = h.read_latency((n + 63) // 64)
                lat = (obs - pub).astype(np.float64) / 1e3
                row["signal_wait_us_median"] = float(np.median(lat))
                row["signal_wait_us_p99"] = float(np.percentile(lat, 99))
                res.append(row)
    return {"workload": cfg.name, "rows": n, "rounds": rounds, "rounds_bulk": rounds_other,
            "default_copy_mode": "auto (vector below 8 KB rows, bulk from 8 KB)",
            "l2": "inputs larger than L2 (no flush)", "sweep": res}


def run_tovl(args):
    import torch
    import workloads
    from consumer_movement_gemm_gb300 import build as tovl_build
    from consumer_movement_gemm_gb300 import tovl

    rank, world, local = dist_init(args)
    torch.cuda.set_device(local)
    dev = "cuda"
    if rank == 0 or world > 1:
        tovl_build.build()
    barrier(world)
    cfg = workloads.TP
    peaks, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    h = tovl.Handle(local, max_rows=1 << 14, producer_ctas=args.producers, k_slices=args.k_slices)
    if args.no_coop:
        h.set_option(tovl.OPT_COOPERATIVE, 0)   # for profilers that cannot replay cooperative cluster launches
    X, W, gathered, out = tp_setup(h, cfg, dev)
    timer = Timer(stream)
    step = lambda: h.gather_gemm(X, W, gathered, out, stream=stream)  # noqa: E731
    timer.time_calls(step, args.warmup)
    assert h.sync_status() == 0

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        times = timer.time_calls(step, args.steps)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    assert h.sync_status() == 0
    ms = statistics.mean(times)
    ms_max = max_over_ranks(ms, world)
    value = sum_over_ranks(cfg.flops, world) / (ms_max * 1e-3) / 1e12

    acc = acceptance(h, timer, cfg, X, W, gathered, out, 50, args.producers)
    e2e = e2e_tp(h, cfg, W, gathered, out, 50, stream)
    context = unfused_context(timer, cfg, X, W, 30)

    extra = {}
    if args.sweep:
        sweep = []
        for P in [4, 8, 16, 24, 32]:
            h.set_option(tovl.OPT_PRODUCERS, P)
            a = acceptance(h, timer, cfg, X, W, gathered, out, 30, P)
            a["TFLOP/s"] = cfg.flops / (a["T_total_ms"] * 1e-3) / 1e12
            sweep.append(a)
        h.set_option(tovl.OPT_PRODUCERS, args.producers)
        extra["producer_sweep"] = sweep
        ks = []
        for S in [1, 2, 4, 8]:
            with tovl.Handle(local, max_rows=1 << 14, producer_ctas=acc["producer_ctas"], k_slices=S) as hs:
                a = acceptance(hs, timer, cfg, X, W, gathered, out, 30, acc["producer_ctas"])
                a["k_slices"] = S
                a["TFLOP/s"] = cfg.flops / (a["T_total_ms"] * 1e-3) / 1e12
                ks.append(a)
        extra["k_slices_sweep"] = ks
    h.close()
    if not args.quick:
        extra["dispatch_uniform"] = dispatch_bench(workloads.DISPATCH, 30 if not args.full else workloads.DISPATCH.rounds * 10,
                                                   dev, args.producers, args.k_slices)
        extra["dispatch_zipf"] = dispatch_bench(workloads.SKEWED, 20 if not args.full else workloads.SKEWED.rounds * 10,
                                                dev, args.producers, args.k_slices)
        extra["dispatch_uniform_pairs"] = dispatch_bench(workloads.DISPATCH, 30 if not args.full else workloads.DISPATCH.rounds * 10,
                                                         dev, args.producers, args.k_slices, align=256)
        extra["dispatch_zipf_pairs"] = dispatch_bench(workloads.SKEWED, 20 if not args.full else workloads.SKEWED.rounds * 10,
                                                      dev, args.producers, args.k_slices, align=256)
        extra["gemm_reduce_scatter"] = rs_bench(workloads.TP, 30 if not args.full else 200, dev)
        sizes = list(workloads.COPY.row_sizes)
        extra["gated_copy"] = copy_sweep(workloads.COPY.rounds, dev, sizes, 1000 if args.full else 20)

    if rank != 0:
        return
    tf = cfg.flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    traffic = recorded_traffic("fused_gather_gemm_tp.md")
    cpu = cpu_baseline(cfg)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "shards": cfg.shards, "rows_per_shard": cfg.rows_per_shard, "K": cfg.K,
                   "N": cfg.N, "parallelism": "replicas only" if world > 1 else "single GPU",
                   "l2": "flushed before every timed step: 512 MiB written, then 512 MiB read (cold, clean L2)",
                   "producer_ctas": acc["producer_ctas"], "consumer_ctas": acc["consumer_ctas"],
                   "k_slices": args.k_slices},
        "overlap_efficiency": acc["overlap_efficiency"],
        "gated_copy_GBps": (min(r["gated_GBps"] for r in extra["gated_copy"]["sweep"] if r["copy_mode"] == "auto")
                            if "gated_copy" in extra else None),
        "gated_copy_note": "lowest gated GB/s over the row sizes 256 B - 16 KB, default (auto) mode",
        "acceptance": acc,
        "unfused_context": context,
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                     "traffic": traffic, "peak_kind": f"{peak_kind} bf16 burst (kernel timed alone)",
                     "frac_of_sustained": tf / peaks.get("bf16_tflops_sustained", peak)},
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks.summary(),
        "gpu_launches": args.steps,
        "wall_s_timed_region": t_wall,
        "configs": extra,
    }
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Small, deterministic launch sequences for profiler captures: W + K
    calls of one kernel, nothing else timed.
      fused     tovl_gather_gemm on the TP shape (about 110 MB resident)
      gemm      tovl_gemm_only on the TP shape
      copy      tovl_gated_copy, 2^18 rows x 8 KB, gated, default copy mode (4 GB resident)
      dispatch  tovl_dispatch_grouped_gemm on the uniform top-2 workload
      combine   the dispatch calls, each followed by tovl_combine
      rs        tovl_gemm_reduce_scatter on the TP shape split four ways along K"""
    import torch
    import workloads
    from consumer_movement_gemm_gb300 import build as tovl_build
    from consumer_movement_gemm_gb300 import tovl
    tovl_build.build()
    dev = "cuda"
    n = args.warmup + args.steps
    if args.profile in ("fused", "gemm"):
        cfg = workloads.TP
        with tovl.Handle(0, max_rows=1 << 14, producer_ctas=args.producers, k_slices=args.k_slices) as h:
            if args.no_coop:
                h.set_option(tovl.OPT_COOPERATIVE, 0)
            X, W, gathered, out = tp_setup(h, cfg, dev)
            for _ in range(n):
                if args.profile == "fused":
                    h.gather_gemm(X, W, gathered, out)
                else:
                    h.gemm_only(gathered, W, out)
            assert h.sync_status() == 0
    elif args.profile == "copy":
        rows, rb = 1 << 18, 8192
        perm = torch.from_numpy(workloads.permutation(rows, 0)).to(dev)
        src = workloads.random_bytes(rows, rb, 0, dev)
        dst = torch.empty_like(src)
        with tovl.Handle(0, max_rows=rows) as h:      # the default (automatic) copy mode: bulk at 8 KB rows
            for _ in range(n):
                h.gated_copy(src, dst, perm, gated=True)
            assert h.sync_status() == 0
    elif args.profile == "rs":
        cfg = workloads.TP
        S, M, K, N = cfg.shards, cfg.M, cfg.K, cfg.N
        X = workloads.bf16_normal((S, M, K // S), 1 / K ** 0.5, 0, dev)
        W = workloads.bf16_normal((S, K // S, N), 1 / K ** 0.5, 1, dev)
        partials = torch.empty(S, M, N, dtype=torch.bfloat16, device=dev)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        with tovl.Handle(0, max_rows=1 << 14, k_slices=4) as h:
            if args.no_coop:
                h.set_option(tovl.OPT_COOPERATIVE, 0)
            for _ in range(n):
                h.gemm_reduce_scatter(X, W, partials, out)
            assert h.sync_status() == 0
    else:
        cfg = workloads.DISPATCH
        x, topk_np, W = workloads.dispatch_inputs(cfg, 0, dev)
        rows = tovl.dispatch_rows_aligned(cfg.T, cfg.k, cfg.E, args.dispatch_align)
        with tovl.Handle(0, max_rows=rows, max_pairs=cfg.T * cfg.k, max_experts=cfg.E, k_slices=args.k_slices) as h:
            h.set_option(tovl.OPT_DISPATCH_ALIGN, args.dispatch_align)
            if args.no_coop:
                h.set_option(tovl.OPT_COOPERATIVE, 0)
            topk = torch.from_numpy(topk_np).to(dev)
            dispatched = torch.zeros(rows, cfg.H, dtype=torch.bfloat16, device=dev)
            offs = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
            out = torch.empty(rows, cfg.N, dtype=torch.bfloat16, device=dev)
            w = torch.from_numpy(workloads.gate_weights(cfg.T, cfg.k, 0)).to(dev)
            staging = torch.empty(cfg.T * cfg.k, cfg.N, dtype=torch.bfloat16, device=dev)
            combined = torch.empty(cfg.T, cfg.N, dtype=torch.bfloat16, device=dev)
            for _ in range(n):
                h.dispatch_grouped_gemm(x, topk, W, dispatched, offs, out)
                if args.profile == "combine":
                    h.combine(out, w, staging, combined)
            assert h.sync_status() == 0
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "calls": n}))


def main(argv=None):
    args = parse_args(argv)
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_tovl(args)


if __name__ == "__main__":
    main()
