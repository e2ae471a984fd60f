#!/usr/bin/env python
"""Benchmark: effective TFLOPS (2MNK/t) of lcgemm on the BF16 square sweep.

Workload (one "step"): C = A . B for M = N = K in {2048, 4096, 8192, 16384},
BF16 operands drawn i.i.d. N(0,1) with a seeded generator, A row-major, B
column-major, FP32 accumulation, BF16 output, algorithm chosen per shape by
the library's cost model (``LCGEMM_AUTO``).  ``value`` is sum(2 n^3) over the
sweep divided by the summed device time of the four GEMMs (CUDA events on the
launching stream, L2 flushed by a 256 MB write before every timed launch,
outside the event pair).  Offline timing is per shape: each size gets its W
warm-up launches and then its K timed launches back to back, sizes ascending.
``server`` repeats the launches with seeded random 0-5 ms host sleeps in
between (the randomly spaced launch mode), ``e2e`` times the host-buffer entry
point ``lcgemm_run_host`` with page-locked inputs (host->device copies, the
GEMM and the device->host copy of C inside the timed region), and ``context``
times torch.mm (cuBLAS) on the same operands with the offline protocol, as a
labelled context line outside the library's timed region (``--no-cublas``
skips it).

``--impl reference`` times the CPU oracle (FP64 triple loop, OpenMP) on a
bounded row sample of the same workload instead.

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the sweep (the GEMMs are independent), timing is the max over ranks and
``value`` the flops of all ranks over that time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SIZES = (2048, 4096, 8192, 16384)
WORKLOAD = ("bf16 square sweep M=N=K in {2048,4096,8192,16384}; A row-major, B column-major; "
            "entries N(0,1) seeded; FP32 accumulate, BF16 out; algo=auto")
METRIC = "effective TFLOPS (2MNK/t) FP16/BF16 GEMM, % of GB300 dense peak, offline+server"
UNIT = "TFLOPS"
L2_FLUSH_BYTES = 256 << 20


def _dist():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    return world, rank, local


def _barrier(world):
    import torch
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(x, world, device):
    import torch
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), \
            float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def _kernel_source_hash(name: str) -> str:
    path = os.path.join(ROOT, "complexity_matmul_gb300", "csrc", name)
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "complexity_matmul_gb300", "csrc")
    for p in sorted([path] + [os.path.join(csrc, hdr) for hdr in ("ptx.cuh", "epilogue.cuh", "plain_common.cuh")]):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel_file: str, n: int):
    """DRAM bytes per launch from a committed ncu summary of `kernel_file` at n^3, if that
    summary was taken on the current source of the kernel (else None)."""
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None
    want = _kernel_source_hash(kernel_file)
    for fn in sorted(os.listdir(prof)):
        if not fn.endswith(".md"):
            continue
        text = open(os.path.join(prof, fn)).read()
        for m in re.finditer(r"traffic_per_launch:\s*kernel=(\S+)\s+n=(\d+)\s+bytes=(\d+)\s+source=(\w+)", text):
            if m.group(1) == kernel_file and int(m.group(2)) == n and m.group(4) == want:
                return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        sm, smax, reasons, power = [], None, set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            try:
                power.append(float(f[3]))
            except ValueError:
                pass
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons)}
        loaded = sorted(sm)[len(sm) // 2:] if len(sm) > 4 else sm   # upper half = samples under load
        out = {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
               "samples": len(sm)}
        if power:
            out["power_w"] = statistics.median(sorted(power)[len(power) // 2:])
        return out


# ---------------------------------------------------------------- GPU arm

def run_gpu(args):
    import numpy as np
    import torch

    import complexity_matmul_gb300 as lcg
    import synthetic

    world, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    h = lcg.Handle(local)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    ops = {}
    for n in SIZES:
        A, B = synthetic.operands(n, n, n, "normal", 2, "bf16", str(dev))
        C = torch.empty((n, n), dtype=torch.bfloat16, device=dev)
        ops[n] = (A, B, C)
    chosen = {n: lcg.ALGO_NAMES[h.select(n, n, n, lcg.BF16)] for n in SIZES}
    launches_per_gemm = {"plain": 1, "strassen1": 2, "strassen2": 2}

    def one(n, timed_events=None):
        A, B, C = ops[n]
        flush.fill_(1.0)                               # evict the previous launch's operands from L2
        if timed_events is not None:
            # a device-side wait between the flush and the start event: the host submits the
            # GEMM while the GPU waits, so no host-side gap lands inside the event pair
            torch.cuda._sleep(HOST_COVER_CYCLES)
            timed_events[0].record(stream)
        h.run(A, B, C, algo="auto", stream=stream)
        if timed_events is not None:
            timed_events[1].record(stream)

    evs = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] for n in SIZES}
    # ---- offline, per shape (the offline protocol: warm-up runs of a shape, then its launches back
    # to back): for each size, W untimed launches, then its K timed launches between a barrier and a
    # synchronisation on both sides.  A step is one timed launch of every size, so the K steps are
    # timed exactly, size by size; the sizes run in ascending order.
    t_wall = 0.0
    with ClockSampler(local) as clk:          # runs through warm-up and the timed launches (samples under load)
        for n in SIZES:
            for _ in range(args.warmup):
                one(n)
            torch.cuda.synchronize(dev)
            rc = h.sync_status()
            if rc:
                raise RuntimeError(f"device status {rc} after warm-up")
            _barrier(world)
            torch.cuda.synchronize(dev)
            t_wall0 = time.perf_counter()
            for s in range(args.steps):
                one(n, evs[n][s])
            torch.cuda.synchronize(dev)
            t_wall += time.perf_counter() - t_wall0
            _barrier(world)
    rc = h.sync_status()
    if rc:
        raise RuntimeError(f"device status {rc} in the timed region")
    per_n_ms = {n: [a.elapsed_time(b) for a, b in evs[n]] for n in SIZES}
    step_ms = [sum(per_n_ms[n][s] for n in SIZES) for s in range(args.steps)]
    total_s = _max_over_ranks(sum(step_ms) * 1e-3, world, dev)
    flops_step = sum(2.0 * n ** 3 for n in SIZES)
    value = flops_step * args.steps * world / total_s / 1e12

    # ---- server mode: seeded random 0-5 ms host sleeps before every launch (the GPU idles in
    # between); each launch is event-timed on its own
    rng = np.random.default_rng(1234 + rank)
    srv = {n: [] for n in SIZES}
    for _ in range(args.server_reps):
        for n in SIZES:
            e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            torch.cuda.synchronize(dev)
            time.sleep(float(rng.uniform(0.0, 5e-3)))
            one(n, e)
            torch.cuda.synchronize(dev)
            srv[n].append(e[0].elapsed_time(e[1]))
    srv_total = sum(statistics.median(srv[n]) for n in SIZES) * 1e-3
    server_value = flops_step / srv_total / 1e12
    server_per_size = {str(n): {"median_ms": round(statistics.median(srv[n]), 4),
                                "p10_ms": round(float(np.percentile(srv[n], 10)), 4),
                                "p90_ms": round(float(np.percentile(srv[n], 90)), 4),
                                "tflops": round(2.0 * n ** 3 / (statistics.median(srv[n]) * 1e-3) / 1e12, 1)}
                       for n in SIZES}

    # ---- context only (not on the library's path): cuBLAS through torch.mm on the same operands,
    # with the offline protocol above (per size W warm-up launches, then K launches back to back,
    # each after the same flush and device-side wait, CUDA events), so the two arms meet the same
    # power state; the library's offline per-size medians are the figures to compare with
    context = None
    if not args.no_cublas:
        ctx = {}
        for n in SIZES:
            A, B, C = ops[n]
            for _ in range(args.warmup):
                flush.fill_(1.0)
                torch.mm(A, B.t(), out=C)
            torch.cuda.synchronize(dev)
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(args.steps)]
            for e0, e1 in pairs:
                flush.fill_(1.0)
                torch.cuda._sleep(HOST_COVER_CYCLES)
                e0.record(stream)
                torch.mm(A, B.t(), out=C)
                e1.record(stream)
            torch.cuda.synchronize(dev)
            med = statistics.median(e0.elapsed_time(e1) for e0, e1 in pairs)
            ctx[str(n)] = {"median_ms": round(med, 4), "tflops": round(2.0 * n ** 3 / (med * 1e-3) / 1e12, 1)}
        flops = sum(2.0 * n ** 3 for n in SIZES)
        context = {"torch_mm_cublas": ctx,
                   "value": round(flops / (sum(ctx[str(n)]["median_ms"] for n in SIZES) * 1e-3) / 1e12, 2),
                   "note": "context line, not the library: torch.mm (cuBLAS) on the same BF16 operands with the "
                           "offline protocol (per size W warm-ups, then K launches back to back after the same "
                           "L2 flush and device-side wait, CUDA events); compare with per_size"}

    # ---- roofline of the dominant kernel (largest share of the step)
    peak_burst, peak_sust, hbm, peak_kind = _peaks()
    dom = max(SIZES, key=lambda n: statistics.median(per_n_ms[n]))
    dom_algo = chosen[dom]
    dom_ms = statistics.median(per_n_ms[dom])          # the statistic per_size reports
    mma_frac = {"plain": 1.0, "strassen1": 7 / 8, "strassen2": 49 / 64}[dom_algo]
    achieved = mma_frac * 2.0 * dom ** 3 / (dom_ms * 1e-3) / 1e12
    # square shapes above 128 run the CTA-pair kernels (gemm_pair.cu, lcma_pair.cu)
    kernel_file = {"plain": "gemm_pair.cu", "strassen1": "lcma_pair.cu", "strassen2": "lcma_fused.cu"}[dom_algo]
    traffic = _traffic(kernel_file, dom)
    roofline = {"bound": "tensor", "kernel": f"{dom_algo} GEMM {dom}^3 ({kernel_file})", "achieved": round(achieved, 1),
                "peak": peak_burst, "unit": "TFLOP/s", "frac": round(achieved / peak_burst, 4),
                "peak_source": f"{peak_kind} bf16 burst", "traffic": traffic,
                "duration": "median CUDA-event time of the timed launches",
                # the dominant launches run back to back for the whole timed region (power-capped):
                # the measured sustained figure is the other fair denominator
                "peak_sustained": peak_sust, "frac_sustained": round(achieved / peak_sust, 4)}

    # ---- end to end through the host-buffer entry point (page-locked inputs)
    e2e = run_e2e(h, ops, args, dev, stream, world)

    # ---- CPU baseline: the oracle on a bounded row sample (rank 0, N = 1 only)
    cpu = run_cpu_baseline(ops, args) if (rank == 0 and world == 1 and not args.no_cpu) else None

    clocks = clk.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_s * 1e3 / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sizes": list(SIZES), "algo": "auto",
                       "chosen": {str(n): chosen[n] for n in SIZES}, "parallelism": f"replicas x{world}",
                       "l2": "flushed (256 MB write) before every timed launch; inputs >= 8192^3 exceed L2",
                       "timing": "offline, per size in ascending order: W warm-up launches, then the K timed "
                                 "launches back to back between barrier + synchronize brackets; CUDA events around "
                                 "each launch on the launching stream; a ~0.2 ms device-side wait after the flush "
                                 "covers the host's submission of the GEMM"},
            "pct_of_peak": round(value / world / peak_burst, 4),
            "per_size": {str(n): {"algo": chosen[n], "median_ms": round(statistics.median(per_n_ms[n]), 4),
                                  "tflops": round(2.0 * n ** 3 / (statistics.median(per_n_ms[n]) * 1e-3) / 1e12, 1),
                                  "p10_ms": round(float(np.percentile(per_n_ms[n], 10)), 4),
                                  "p90_ms": round(float(np.percentile(per_n_ms[n], 90)), 4)} for n in SIZES},
            "server": {"value": round(server_value, 2), "unit": UNIT, "reps": args.server_reps,
                       "gaps_ms": "uniform 0-5, seeded", "statistic": "sum of per-size medians",
                       "per_size": server_per_size},
            "roofline": roofline,
            "e2e": e2e,
            "gpu_launches": args.steps * sum(launches_per_gemm[chosen[n]] for n in SIZES),
            "clocks": clocks,
            "wall_s_timed": round(t_wall, 4),
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if context is not None:
            line["context"] = context
        print(json.dumps(line), flush=True)
    h.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def run_e2e(h, ops, args, dev, stream, world):
    import ctypes

    import torch

    host = {}
    for n in SIZES:
        A, B, _ = ops[n]
        host[n] = (A.cpu().pin_memory(), B.cpu().pin_memory(),
                   torch.empty((n, n), dtype=torch.bfloat16).pin_memory())
    sp = ctypes.c_void_p(stream.cuda_stream)

    def one(n, ev=None):
        Ah, Bh, Ch = host[n]
        if ev is not None:
            ev[0].record(stream)
        rc = h.run_host_raw(n, n, n, Ah.data_ptr(), n, Bh.data_ptr(), n, Ch.data_ptr(), n, 1, 3, sp)
        if rc:
            raise RuntimeError(f"lcgemm_run_host failed: {rc}")
        if ev is not None:
            ev[1].record(stream)

    for n in SIZES:
        one(n)
    torch.cuda.synchronize(dev)
    reps = max(1, min(args.steps, 3))
    times = []
    _barrier(world)
    for _ in range(reps):
        tot = 0.0
        for n in SIZES:
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            one(n, ev)
            torch.cuda.synchronize(dev)
            tot += ev[0].elapsed_time(ev[1]) * 1e-3
        times.append(tot)
    t = _max_over_ranks(statistics.median(times), world, dev)
    flops = sum(2.0 * n ** 3 for n in SIZES)
    return {"value": round(flops * world / t / 1e12, 2), "unit": UNIT,
            "h2d_bytes_per_step": sum(2 * 2 * n * n for n in SIZES),
            "d2h_bytes_per_step": sum(2 * n * n for n in SIZES),
            "api": "lcgemm_run_host (page-locked host buffers)"}


def _cpu_sample_rows():
    return 1024


def run_cpu_baseline(ops, args):
    import numpy as np

    import oracle
    import synthetic
    n = max(SIZES)
    A, B, _ = ops[n]
    rows = synthetic.row_sample(n, _cpu_sample_rows())
    Ab = synthetic.bits(A[torch_index(rows, A.device)])
    Bb = synthetic.bits(B)
    t0 = time.perf_counter()
    oracle.gemm(Ab, Bb, oracle.BF16, rows=np.arange(len(rows)))
    t = time.perf_counter() - t0
    flops = 2.0 * len(rows) * n * n
    return {"value": round(flops / t / 1e12, 6), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(rows)} seeded rows of C for the {n}^3 GEMM (FP64 naive triple loop), {t:.1f} s"}


def torch_index(rows, device):
    import torch
    return torch.as_tensor(rows, device=device)


# ---------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args):
    import numpy as np

    import oracle
    import synthetic
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    rows_per = 32                      # >= the host's OpenMP threads on the GPU machine
    data = {}
    for n in SIZES:
        A = synthetic.matrix(rows_per, n, "normal", 1002, "bf16")       # a row sample of A
        B = synthetic.matrix(n, n, "normal", 2002, "bf16")
        data[n] = (synthetic.bits(A), synthetic.bits(B))

    def step():
        for n in SIZES:
            Ab, Bb = data[n]
            oracle.gemm(Ab, Bb, oracle.BF16)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    flops = sum(2.0 * rows_per * n * n for n in SIZES) * args.steps
    value = flops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sizes": list(SIZES), "algo": "oracle (plain definition)",
                   "sample": f"{rows_per} rows of C per size per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{rows_per} rows of C for each n in {list(SIZES)} per step"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_case(args):
    """Run one GEMM shape a few times without timing (a fixed launch sequence for ncu captures)."""
    import torch

    import complexity_matmul_gb300 as lcg
    import synthetic
    dims = [int(x) for x in args.case.split(",")]
    M, N, K = (dims * 3)[:3] if len(dims) == 1 else dims
    dev = torch.device("cuda", 0)
    h = lcg.Handle(0)
    if args.plain_kernel:
        h.set_option(lcg.OPT_PLAIN_KERNEL, args.plain_kernel)
    if args.lcma_kernel:
        h.set_option(lcg.OPT_LCMA_KERNEL, args.lcma_kernel)
    if args.group_order is not None:
        h.set_option(lcg.OPT_GROUP_ORDER, args.group_order)
    A, B = synthetic.operands(M, N, K, "normal", 2, "bf16", str(dev))
    C = torch.empty((M, (N + 7) // 8 * 8), dtype=torch.bfloat16, device=dev)[:, :N]
    if args.torch_mm:
        # context for captures: cuBLAS (torch.mm) on the same operands, not the library
        for _ in range(args.reps):
            torch.mm(A, B.t(), out=C)
        torch.cuda.synchronize(dev)
        print(f"case {M}x{N}x{K} torch.mm reps={args.reps}")
        h.close()
        return
    for _ in range(args.reps):
        h.run(A, B, C, algo=args.algo)
    torch.cuda.synchronize(dev)
    rc = h.sync_status()
    print(f"case {M}x{N}x{K} algo={args.algo} reps={args.reps} last={lcg.ALGO_NAMES[h.last_algo()]} status={rc}")
    h.close()
    if rc:
        sys.exit(1)


# A device-side sleep (~0.2 ms) between the L2 flush and the timed launch: the host enqueues the
# launch while the GPU sleeps, so no host-side gap lands between the two events of a short kernel.
HOST_COVER_CYCLES = 400_000
OFFLINE_REPS = 20                # --grid-mode offline: back-to-back launches per algorithm and shape
OFFLINE_COVER_CYCLES = 4_000_000 # GPU sleep (~2 ms) covering the host's enqueueing of those launches


def _time_launch(h, A, B, C, algo, reps, flush):
    """Median device time (s) of `reps` launches, L2 flushed before each."""
    import torch
    for _ in range(2):
        h.run(A, B, C, algo=algo)
    ts = []
    for _ in range(reps):
        flush.fill_(1.0)
        torch.cuda._sleep(HOST_COVER_CYCLES)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        h.run(A, B, C, algo=algo)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    ts.sort()
    return ts[len(ts) // 2]


def _time_offline(h, A, B, C, algo, reps):
    """Device time (s) per launch of `reps` back-to-back launches (no flush, no host gaps): one event
    pair around all of them, since consecutive launches may overlap (a kernel's prologue runs while
    the one before it finishes) and an event between two launches would serialise them."""
    import torch
    for _ in range(2):
        h.run(A, B, C, algo=algo)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(OFFLINE_COVER_CYCLES)       # the host enqueues all launches before the GPU reaches them
    e0.record()
    for _ in range(reps):
        h.run(A, B, C, algo=algo)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3 / reps


def _time_server(h, A, B, C, algo, reps, rng):
    """Median device time (s) of `reps` launches, each after a host pause drawn uniform in 0-5 ms."""
    import torch
    for _ in range(2):
        h.run(A, B, C, algo=algo)
    ts = []
    for _ in range(reps):
        torch.cuda.synchronize()
        time.sleep(float(rng.uniform(0.0, 5e-3)))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        h.run(A, B, C, algo=algo)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    ts.sort()
    return ts[len(ts) // 2]


def run_grid(args):
    """Cost-model accuracy on the FP16 shape grid: time every eligible algorithm per
    (M, N, K), check that `auto`'s choice is within 2 % of the fastest one.  Timing modes:
    `flushed` (L2 flushed before each launch), `offline` (back-to-back launches), `server`
    (seeded uniform 0-5 ms host pauses before each launch)."""
    import numpy as np
    import torch

    import complexity_matmul_gb300 as lcg
    import synthetic
    triples = synthetic.grid_quick_subset() if args.grid == "quick" else synthetic.grid_triples()
    dev = torch.device("cuda", 0)
    h = lcg.Handle(0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    rng = np.random.default_rng(4321)
    rows, correct = [], 0
    for (M, N, K) in triples:
        A = synthetic.matrix(M, K, "normal", 1003, "f16", str(dev), scale=1.0 / K ** 0.5)
        B = synthetic.matrix(N, K, "normal", 2003, "f16", str(dev))
        C = torch.empty((M, N), dtype=torch.float16, device=dev)
        times = {}
        for algo in ("plain", "strassen1", "strassen2"):
            try:
                h.estimate(M, N, K, lcg.F16, algo)
            except lcg.LcgemmError:
                continue
            if args.grid_mode == "offline":
                times[algo] = _time_offline(h, A, B, C, algo, OFFLINE_REPS)
            elif args.grid_mode == "server":
                times[algo] = _time_server(h, A, B, C, algo, args.grid_reps, rng)
            else:
                times[algo] = _time_launch(h, A, B, C, algo, args.grid_reps, flush)
        chosen = lcg.ALGO_NAMES[h.select(M, N, K, lcg.F16)]
        best = min(times, key=times.get)
        ok = times[chosen] <= 1.02 * times[best]
        correct += ok
        rows.append({"M": M, "N": N, "K": K, "chosen": chosen, "best": best, "ok": bool(ok),
                     "tflops": {a: round(2.0 * M * N * K / t / 1e12, 2) for a, t in times.items()},
                     "pred_ms": {a: round(h.estimate(M, N, K, lcg.F16, a) * 1e3, 4) for a in times},
                     "ms": {a: round(t * 1e3, 4) for a, t in times.items()}})
        del A, B, C
    rc = h.sync_status()
    ratios = {}
    for a in ("plain", "strassen1", "strassen2"):
        r = sorted(row["pred_ms"][a] / row["ms"][a] for row in rows if a in row["ms"] and row["ms"][a] > 0)
        if r:
            ratios[a] = {"geomean": round(float(np.exp(np.mean(np.log(r)))), 3),
                         "p10": round(float(np.percentile(r, 10)), 3), "median": round(float(np.median(r)), 3),
                         "p90": round(float(np.percentile(r, 90)), 3)}
    misses = [{k: row[k] for k in ("M", "N", "K", "chosen", "best", "ms")} for row in rows if not row["ok"]]
    summary = {"grid": args.grid, "mode": args.grid_mode, "shapes": len(triples), "auto_within_2pct": correct,
               "fraction": round(correct / len(triples), 4), "status": rc,
               "fastest_counts": {a: sum(r["best"] == a for r in rows) for a in ("plain", "strassen1", "strassen2")},
               "chosen_counts": {a: sum(r["chosen"] == a for r in rows) for a in ("plain", "strassen1", "strassen2")},
               "predicted_over_measured": ratios, "misses": misses}
    print(json.dumps(summary), flush=True)
    if args.grid_out:
        with open(args.grid_out, "w") as f:
            json.dump({"summary": summary, "rows": rows}, f)


def run_skinny(args):
    """LLM-shaped skinny BF16 GEMMs: time per shape, effective TFLOPS and HBM GB/s."""
    import torch

    import complexity_matmul_gb300 as lcg
    import synthetic
    dev = torch.device("cuda", 0)
    h = lcg.Handle(0)
    if args.plain_kernel:
        h.set_option(lcg.OPT_PLAIN_KERNEL, args.plain_kernel)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    _, _, hbm, kind = _peaks()
    for (M, N, K) in synthetic.SKINNY:
        A = synthetic.matrix(M, K, "normal", 1004, "bf16", str(dev))
        B = synthetic.matrix(N, K, "normal", 2004, "bf16", str(dev), scale=0.02)
        C = torch.empty((M, (N + 7) // 8 * 8), dtype=torch.bfloat16, device=dev)[:, :N]
        t = _time_launch(h, A, B, C, "auto", args.grid_reps, flush)
        byts = 2.0 * (M * K + K * N + M * N)
        print(json.dumps({"M": M, "N": N, "K": K, "us": round(t * 1e6, 2), "tflops": round(2.0 * M * N * K / t / 1e12, 2),
                          "GBps": round(byts / t / 1e9, 1), "hbm_frac": round(byts / t / 1e9 / hbm, 3),
                          "algo": lcg.ALGO_NAMES[h.last_algo()]}), flush=True)


def run_large(args):
    """The large rectangular BF16 shapes: plain, one- and two-level Strassen, and the one-level fused
    kernel with Group ordering off and the tail split off; effective and actual-MMA TFLOP/s, with the
    SM clock sampled during each variant's launches."""
    import torch

    import complexity_matmul_gb300 as lcg
    import synthetic
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    variants = [("plain", "plain", {}), ("strassen1", "strassen1", {}), ("strassen2", "strassen2", {}),
                ("strassen1 order off", "strassen1", {lcg.OPT_GROUP_ORDER: 0}),
                ("strassen1 split off", "strassen1", {lcg.OPT_SPLIT: 0})]
    mma_frac = {"plain": 1.0, "strassen1": 7 / 8, "strassen2": 49 / 64}
    for (M, N, K) in synthetic.LARGE_RECT:
        A, B = synthetic.operands(M, N, K, "normal", 5, "bf16", str(dev))
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        out = {}
        for name, algo, opts in variants:
            h = lcg.Handle(0)
            for k, v in opts.items():
                h.set_option(k, v)
            with ClockSampler(0) as clk:
                t = _time_launch(h, A, B, C, algo, args.grid_reps, flush)
            rc = h.sync_status()
            h.close()
            if rc:
                raise RuntimeError(f"device status {rc} for {name}")
            eff = 2.0 * M * N * K / t / 1e12
            cs = clk.summary()
            out[name] = {"ms": round(t * 1e3, 3), "eff_tflops": round(eff, 1),
                         "mma_tflops": round(eff * mma_frac[algo], 1), "sm_mhz": cs.get("sm_mhz"),
                         "reasons": cs.get("reasons")}
        print(json.dumps({"M": M, "N": N, "K": K, **out}), flush=True)
        del A, B, C


RACE_SHAPES = [(4096, 4096, 4096), (8192, 8192, 8192), (16384, 16384, 16384), (24576, 24576, 24576),
               (32768, 32768, 32768), (16384, 16384, 8192), (8192, 28672, 8192), (32768, 8192, 4096)]


def run_race(args):
    """Plain against one-level Strassen (and two-level) per shape, in two regimes: burst (L2
    flushed before each launch, launches interleaved across algorithms, median of --grid-reps)
    and sustained (--race-seconds of back-to-back launches per algorithm, SM clock and board
    power sampled meanwhile): effective TFLOP/s = 2MNK/t, TFLOP/s per median MHz, and energy per
    GEMM (median power x time)."""
    import torch

    import complexity_matmul_gb300 as lcg
    import synthetic
    dev = torch.device("cuda", 0)
    h = lcg.Handle(0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    algos = args.race_algos.split(",")
    shapes = RACE_SHAPES if not args.race_shapes else \
        [tuple(int(x) for x in s.split("x")) * (3 if "x" not in s else 1) for s in args.race_shapes.split(",")]
    for (M, N, K) in shapes:
        A, B = synthetic.operands(M, N, K, "normal", 2, "bf16", str(dev))
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        flops = 2.0 * M * N * K
        for a in algos:
            for _ in range(2):
                h.run(A, B, C, algo=a)
        torch.cuda.synchronize()
        burst = {a: [] for a in algos}
        with ClockSampler(0) as clk:
            for _ in range(args.grid_reps):
                for a in algos:
                    flush.fill_(1.0)
                    torch.cuda._sleep(HOST_COVER_CYCLES)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    h.run(A, B, C, algo=a)
                    e1.record()
                    torch.cuda.synchronize()
                    burst[a].append(e0.elapsed_time(e1) * 1e-3)
        out = {"M": M, "N": N, "K": K, "burst_clock": clk.summary()}
        mma_frac = {"plain": 1.0, "strassen1": 7 / 8, "strassen2": 49 / 64}
        for a in algos:
            t = statistics.median(burst[a])
            out[a] = {"burst_ms": round(t * 1e3, 3), "burst_tflops": round(flops / t / 1e12, 1),
                      "burst_mma_tflops": round(mma_frac.get(a, 1.0) * flops / t / 1e12, 1)}
        for a in algos:
            n = max(3, int(args.race_seconds / max(min(burst[a]), 1e-6)))
            torch.cuda.synchronize()
            with ClockSampler(0) as clk:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(n):
                    h.run(A, B, C, algo=a)
                e1.record()
                torch.cuda.synchronize()
            t = e0.elapsed_time(e1) * 1e-3 / n
            cs = clk.summary()
            row = out[a]
            row.update({"sustained_ms": round(t * 1e3, 3), "sustained_tflops": round(flops / t / 1e12, 1),
                        "sustained_mma_tflops": round(mma_frac.get(a, 1.0) * flops / t / 1e12, 1),
                        "launches": n, "sm_mhz": cs.get("sm_mhz"), "reasons": cs.get("reasons")})
            if cs.get("sm_mhz"):
                row["tflops_per_mhz"] = round(flops / t / 1e12 / cs["sm_mhz"], 4)
            if cs.get("power_w"):
                row["power_w"] = cs["power_w"]
                row["joules_per_gemm"] = round(cs["power_w"] * t, 3)
        rc = h.sync_status()
        if rc:
            raise RuntimeError(f"device status {rc}")
        print(json.dumps(out), flush=True)
        del A, B, C
        torch.cuda.empty_cache()
    h.close()


PADDED_SHAPES = [((8191, 8193, 8190), (8192, 8192, 8192)), ((16383, 16385, 8191), (16384, 16384, 8192))]


def run_padded(args):
    """Strassen on shapes its block split cannot divide (zero-padded operand copies) against the
    neighbouring divisible shape, and plain on both."""
    import torch

    import complexity_matmul_gb300 as lcg
    import synthetic
    dev = torch.device("cuda", 0)
    h = lcg.Handle(0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for odd, even in PADDED_SHAPES:
        row = {}
        for tag, (M, N, K) in (("odd", odd), ("even", even)):
            A, B = synthetic.operands(M, N, K, "normal", 5, "bf16", str(dev))
            A = torch.zeros((M, (K + 7) // 8 * 8), dtype=A.dtype, device=dev)[:, :K].copy_(A)
            B = torch.zeros((N, (K + 7) // 8 * 8), dtype=B.dtype, device=dev)[:, :K].copy_(B)
            C = torch.empty((M, (N + 7) // 8 * 8), dtype=torch.bfloat16, device=dev)[:, :N]
            for algo in ("plain", "strassen1", "strassen2"):
                t = _time_launch(h, A, B, C, algo, args.grid_reps, flush)
                row[f"{tag} {algo}"] = {"shape": [M, N, K], "ms": round(t * 1e3, 3),
                                        "eff_tflops": round(2.0 * M * N * K / t / 1e12, 1)}
            del A, B, C
        print(json.dumps(row), flush=True)
    rc = h.sync_status()
    h.close()
    if rc:
        sys.exit(1)


EPILOGUE_SHAPES = [(4096, 4096, 4096), (8192, 8192, 8192), (8192, 28672, 8192), (16, 14336, 4096),
                   (128, 14336, 4096)]


def run_epilogue(args):
    """Cost of the fused epilogue C = gelu_tanh(A.B + bias) + residual against the bare GEMM, and
    against the same epilogue as a separate element-wise pass over C (torch ops, for context)."""
    import torch

    import complexity_matmul_gb300 as lcg
    import synthetic
    dev = torch.device("cuda", 0)
    h = lcg.Handle(0)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    _, _, hbm, _ = _peaks()
    for (M, N, K) in EPILOGUE_SHAPES:
        A, B = synthetic.operands(M, N, K, "normal", 5, "bf16", str(dev), scale_a=K ** -0.5)
        bias = synthetic.matrix(1, N, "normal", 3005, "bf16", str(dev))[0]
        R = synthetic.matrix(M, N, "normal", 4005, "bf16", str(dev))
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

        def timed(fn):
            for _ in range(2):
                fn()
            ts = []
            for _ in range(args.grid_reps):
                flush.fill_(1.0)
                torch.cuda._sleep(HOST_COVER_CYCLES)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e-3)
            return sorted(ts)[len(ts) // 2]

        t_gemm = timed(lambda: h.run(A, B, C, algo="plain"))
        t_fused = timed(lambda: h.run(A, B, C, algo="plain", bias=bias, residual=R, act="gelu_tanh"))
        t_sep = timed(lambda: torch.add(torch.nn.functional.gelu(h.run(A, B, C, algo="plain") + bias,
                                                                 approximate="tanh"), R))
        print(json.dumps({"M": M, "N": N, "K": K, "epilogue": "bias+gelu_tanh+residual",
                          "gemm_us": round(t_gemm * 1e6, 1), "fused_us": round(t_fused * 1e6, 1),
                          "separate_pass_us": round(t_sep * 1e6, 1),
                          "fused_overhead": round(t_fused / t_gemm - 1.0, 4),
                          "fused_tflops": round(2.0 * M * N * K / t_fused / 1e12, 1),
                          "extra_bytes_min": 2 * M * N + 2 * N,
                          "extra_bytes_min_at_hbm_us": round((2 * M * N + 2 * N) / (hbm * 1e9) * 1e6, 1)}),
              flush=True)
        del A, B, R, C
    rc = h.sync_status()
    h.close()
    if rc:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["lcgemm", "reference"], default="lcgemm")
    ap.add_argument("--server-reps", type=int, default=50)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--no-cublas", action="store_true", help="skip the torch.mm (cuBLAS) context line")
    ap.add_argument("--case", default=None, help="profiling mode: run one shape 'n' or 'M,N,K' --reps times")
    ap.add_argument("--algo", default="auto", help="algorithm for --case")
    ap.add_argument("--torch-mm", action="store_true", help="--case: run torch.mm (cuBLAS) instead, for context")
    ap.add_argument("--reps", type=int, default=3, help="launches for --case")
    ap.add_argument("--plain-kernel", type=int, default=0,
                    help="--case/--skinny: 1 single-CTA, 2 CTA-pair, 3 skinny plain kernel")
    ap.add_argument("--lcma-kernel", type=int, default=0, help="--case: 1 single-CTA, 2 CTA-pair fused kernel")
    ap.add_argument("--grid", choices=["quick", "full"], default=None,
                    help="cost-model accuracy on the FP16 shape grid (100-triple subset or all 1000)")
    ap.add_argument("--grid-out", default=None, help="--grid: write per-shape results to this JSON file")
    ap.add_argument("--grid-mode", choices=["flushed", "offline", "server"], default="flushed",
                    help="--grid timing: L2 flushed before each launch, back-to-back, or random 0-5 ms gaps")
    ap.add_argument("--grid-reps", type=int, default=5, help="--grid/--skinny: timed launches per algorithm")
    ap.add_argument("--skinny", action="store_true", help="time the LLM-shaped skinny GEMMs")
    ap.add_argument("--large", action="store_true",
                    help="large rectangular shapes: plain, Strassen and its ordering / split ablations")
    ap.add_argument("--group-order", type=int, default=None, help="--case: Strassen Group ordering 0/1")
    ap.add_argument("--race", action="store_true",
                    help="plain vs Strassen per shape: burst (flushed, interleaved) and sustained (back to back)")
    ap.add_argument("--race-shapes", default="", help="--race: comma-separated n or MxNxK (default: built-in list)")
    ap.add_argument("--race-algos", default="plain,strassen1", help="--race: algorithms to compare")
    ap.add_argument("--race-seconds", type=float, default=2.0, help="--race: seconds of back-to-back launches")
    ap.add_argument("--padded", action="store_true",
                    help="Strassen on non-divisible shapes (zero-padded operands) against divisible ones")
    ap.add_argument("--epilogue", action="store_true",
                    help="time the fused bias + GELU + residual epilogue against the bare GEMM")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.case:
        run_case(args)
    elif args.grid:
        run_grid(args)
    elif args.skinny:
        run_skinny(args)
    elif args.epilogue:
        run_epilogue(args)
    elif args.large:
        run_large(args)
    elif args.race:
        run_race(args)
    elif args.padded:
        run_padded(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
