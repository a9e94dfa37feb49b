#!/usr/bin/env python
"""Benchmark of the gradient-compression hot path on GB300.

Headline workload (one "step"): 2-bit compression with error feedback of 8
simulated data-parallel workers' fp32 gradients of 25,557,032 elements each
(ResNet-50-sized, g ~ N(0, 1e-3^2), t = 2e-3), then the dequantise-sum of the
8 packed buffers fused with the SGD update w -= 0.1 * avg on fp32 weights.
Metric: input-gradient GB/s = 8 * n * 4 bytes per step / step time.

The JSON line also carries, for the dominant kernel (gc_2bit_quantize), its
achieved HBM bandwidth against the measured copy peak, the end-to-end number
through the C ABI with host buffers, the clocks seen during the timed region,
the CPU oracle timed on this host, and a per-row table for the other
workloads (QSGD, CD-SGD, SAPS + EASGD, the one-worker 2-bit case).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
Multi-GPU: one process per GPU under torchrun; every rank runs its own
independent instance of the workload (weak scaling, no data-path collective).
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

HEADLINE_METRIC = "input-gradient GB/s (and % of GB300 HBM peak) for 2-bit compress+residual"


# ----------------------------------------------------------------------------- helpers

def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle timings")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", default=None,
                    help="run one kernel on a profiling-sized case three times and exit "
                         f"({', '.join(CASES)})")
    ap.add_argument("--case-n", type=int, default=0, help="elements for --case (0 = default)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "gb300" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg, dev=None):
    if pg is not None:
        if dev is not None:
            pg.barrier(device_ids=[dev.index])
        else:
            pg.barrier()


def max_over_ranks(pg, value: float, dev=None) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=dev if dev is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def code_only(text: str) -> str:
    """C/CUDA source without its comments, every run of whitespace folded to
    one space: the part of a file that decides what the compiler builds."""
    out = []
    i, n = 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_sha(rel: str) -> str:
    """Hash of a kernel source's code (comments and layout excluded), which
    ties a committed ncu capture to the code it was taken on."""
    with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
        return hashlib.sha256(code_only(f.read()).encode()).hexdigest()[:16]


def ncu_entry(kernel: str):
    """The committed ncu summary of a kernel (DRAM bytes and warp instructions
    per launch, scaled to the launch bench.py times), or None when the kernel
    source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kernel]
        if d.get("source_sha") != source_sha(d["source"]):
            return None
        return d
    except Exception:
        return None


def ncu_traffic(kernel: str):
    d = ncu_entry(kernel)
    return float(d["bytes_per_launch"]) if d else None


# Issue roofline for kernels bound by instruction issue rather than HBM:
# 152 SMs x 4 schedulers x 1 warp instruction per clock at the 2070 MHz
# maximum SM clock.
ISSUE_PEAK = 152 * 4 * 2070e6


def dram_roofline(kernel: str, ms_list, peak: float):
    """DRAM bytes the kernel really moves (committed ncu capture, scaled to the
    bench launch) over its measured time: the roofline for kernels whose
    algorithmic bytes are far below their unavoidable traffic (random 4-byte
    gathers and scatters move whole DRAM sectors or lines)."""
    d = ncu_entry(kernel)
    if not d or not ms_list:
        return None
    gbps = float(d["bytes_per_launch"]) / (_median(ms_list) * 1e-3) / 1e9
    return {"bound": "hbm (DRAM bytes moved)", "bytes": int(d["bytes_per_launch"]), "achieved": round(gbps, 1),
            "peak": peak, "unit": "GB/s", "frac": round(gbps / peak, 3)}


def issue_roofline(kernel: str, ms_list, mult: int = 1):
    """Issue rate of a launch doing `mult` times the captured kernel's work
    (e.g. a batched call over `mult` streams)."""
    d = ncu_entry(kernel)
    if not d or "warp_inst_per_launch" not in d or not ms_list:
        return None
    inst = mult * float(d["warp_inst_per_launch"])
    rate = inst / (_median(ms_list) * 1e-3)
    return {"bound": "issue", "achieved": round(rate / 1e12, 4), "peak": round(ISSUE_PEAK / 1e12, 4),
            "unit": "T warp instructions/s", "frac": round(rate / ISSUE_PEAK, 3),
            "warp_inst_per_launch": int(inst)}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        win = [p for (t, p) in self.samples if t0 - 0.06 <= t <= t1 + 0.06]
        if not win and self.samples:
            # the timed region was shorter than the sampling period: nearest sample
            mid = 0.5 * (t0 + t1)
            win = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        smax = [num(p[1]) for p in win if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(win)}


def gpu_id_for(dev):
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


class Timer:
    """CUDA events around individual launches on one stream."""

    def __init__(self, stream):
        self.stream = stream
        self.pairs = {}

    def around(self, key, fn):
        import torch
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        fn()
        b.record(self.stream)
        self.pairs.setdefault(key, []).append((a, b))

    def ms(self, key):
        return [a.elapsed_time(b) for a, b in self.pairs.get(key, [])]


def flush_l2(buf):
    buf.add_(1)   # writes a buffer larger than L2


# ----------------------------------------------------------------------------- headline

def headline(args, dev, rank, world, pg):
    import torch
    import gradient_compression_sgd_gc_gb300 as gc
    from gradient_compression_sgd_gc_gb300 import workloads as wl

    cfg = wl.TWOBIT_DQ_SGD
    n, W, t, lr = cfg.n, cfg.workers, cfg.threshold, cfg.lr
    stream = torch.cuda.current_stream(dev)
    pool = min(20, args.steps + args.warmup)
    grads = [[wl.twobit_grad(cfg, s, w, device=dev) for w in range(W)] for s in range(pool)]
    res = [torch.zeros(n, device=dev) for _ in range(W)]
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=dev) for _ in range(W)]
    weights = wl.twobit_weights(cfg, device=dev)
    # validated launches with their arguments prepared once (host cost per
    # launch ~ a ctypes call), so the GPU queue never runs dry; the 8 workers'
    # buffers are quantised by one batched launch
    quant = [gc.gc_2bit_quantize_batched(grads[s], res, codes, t, stream=stream, prepare=True)
             for s in range(pool)]
    dqsum = gc.gc_2bit_dequant_sum_update(codes, n, t, gc.GC_UPD_SGD, lr=lr, weights=weights,
                                          stream=stream, prepare=True)

    for s in range(args.warmup):
        quant[s % pool]()
        dqsum()
    torch.cuda.synchronize(dev)
    evq = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    evd = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    clocks = ClockSampler(gpu_id_for(dev)) if rank == 0 else None
    time.sleep(0.15)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(pg, dev)
    torch.cuda.synchronize(dev)
    w0 = time.time()
    start.record(stream)
    for s in range(args.steps):
        a, b = evq[s]
        a.record(stream)
        quant[(args.warmup + s) % pool]()
        b.record(stream)
        a, b = evd[s]
        a.record(stream)
        dqsum()
        b.record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    w1 = time.time()
    barrier(pg, dev)
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(pg, total_ms, dev)
    clk = None
    if clocks is not None:
        time.sleep(0.1)
        clocks.stop()
        clk = clocks.summary(w0, w1)
    q_ms = [a.elapsed_time(b) for (a, b) in evq]
    d_ms = [a.elapsed_time(b) for (a, b) in evd]
    del grads, quant
    return {"total_ms": total_ms, "quantize_ms": q_ms, "dqsum_ms": d_ms, "clocks": clk,
            "launches": args.steps * 2, "n": n, "W": W}


def e2e(args, dev, pg=None, world: int = 1):
    """Same metric through the public API with host buffers.  The headline
    path: every step hands the 8 pinned host gradient buffers to
    gc_2bit_quantize_batched, whose kernel reads them in place over the host
    link (the API's host-buffer path), then the dequant-sum + SGD runs and the
    8 packed code buffers are read back.  Beside it, the same step with
    explicit uploads (a copy stream, worker w+1's upload overlapping worker
    w's quantisation).  Every rank runs it (each GPU has its own host link);
    the slowest rank's time sets the whole-job value."""
    import torch
    import gradient_compression_sgd_gc_gb300 as gc
    from gradient_compression_sgd_gc_gb300 import workloads as wl

    cfg = wl.TWOBIT_DQ_SGD
    n, W, t, lr = cfg.n, cfg.workers, cfg.threshold, cfg.lr
    stream = torch.cuda.current_stream(dev)
    # one copy stream: measured fastest here (more streams split the host link)
    copies = [torch.cuda.Stream(dev)]
    host_g = [wl.twobit_grad(cfg, 0, w, device="cpu").pin_memory() for w in range(W)]
    host_c = [torch.empty(gc.code_words(n), dtype=torch.int32).pin_memory() for _ in range(W)]
    dev_g = [torch.empty(n, device=dev) for _ in range(W)]
    res = [torch.zeros(n, device=dev) for _ in range(W)]
    codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=dev) for _ in range(W)]
    weights = wl.twobit_weights(cfg, device=dev)
    quant = [gc.gc_2bit_quantize(dev_g[w], res[w], codes[w], t, stream=stream, prepare=True)
             for w in range(W)]
    dqsum = gc.gc_2bit_dequant_sum_update(codes, n, t, gc.GC_UPD_SGD, lr=lr, weights=weights,
                                          stream=stream, prepare=True)
    up = [[torch.cuda.Event() for _ in copies] for _ in range(W)]
    used = [torch.cuda.Event() for _ in range(W)]

    def step():
        for w in range(W):
            for h, cs in enumerate(copies):
                cs.wait_event(used[w])        # the previous step's kernel has read dev_g[w]
                with torch.cuda.stream(cs):
                    dev_g[w].copy_(host_g[w], non_blocking=True)
                up[w][h].record(cs)
        for w in range(W):
            for h in range(len(copies)):
                stream.wait_event(up[w][h])
            quant[w]()
            used[w].record(stream)
        dqsum()
        for w in range(W):
            host_c[w].copy_(codes[w], non_blocking=True)

    # the API's host-buffer path: the batched quantiser reads the pinned host
    # gradients in place
    quant_host = gc.gc_2bit_quantize_batched(host_g, res, codes, t, stream=stream, prepare=True)

    def step_in_place():
        quant_host()
        dqsum()
        for w in range(W):
            host_c[w].copy_(codes[w], non_blocking=True)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        barrier(pg, dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for cs in copies:
            cs.wait_event(a)                  # no upload of the timed steps starts early
        for _ in range(args.e2e_steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(pg, dev)
        return max_over_ranks(pg, a.elapsed_time(b) / args.e2e_steps, dev)

    for w in range(W):
        used[w].record(stream)
    ms_copy = timed(step)
    ms = timed(step_in_place)
    h2d = W * n * 4
    d2h = W * gc.code_words(n) * 4
    return {"value": round(world * W * n * 4 / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4),
            "h2d_GBps": round(h2d / (ms * 1e-3) / 1e9, 1),
            "path": "gc_2bit_quantize_batched reads the pinned host gradients in place; codes read back",
            "explicit_upload_GBps": round(world * W * n * 4 / (ms_copy * 1e-3) / 1e9, 2)}


# ----------------------------------------------------------------------------- CPU oracle

def _oracle_twobit_chunk(job):
    """One host process of the CPU baseline: the oracle, as it stands, on its
    own chunk of m elements per worker of the headline workload (the 2-bit
    step is elementwise, so chunks are independent).  Runs `warmup` steps,
    then `steps` timed steps, or -- with steps = 0 -- as many as fit in
    `seconds`.  Returns (timed steps, seconds)."""
    chunk, m, warmup, steps, seconds = job
    import numpy as np
    import oracle
    from gradient_compression_sgd_gc_gb300 import workloads as wl

    cfg = wl.TWOBIT_DQ_SGD
    W, t, lr = cfg.workers, cfg.threshold, cfg.lr
    grads = [wl.normal(m, cfg.grad_std, 1000 + 16 * chunk + w).numpy() for w in range(W)]
    res = [np.zeros(m, np.float32) for _ in range(W)]
    w64 = wl.uniform(m, 0.05, 7 + chunk).numpy().astype(np.float64)

    def step():
        codes = [oracle.twobit_quantize(grads[q], res[q], t) for q in range(W)]
        oracle.twobit_dequant_sum_update(codes, m, t, oracle.KIND_SGD, lr=lr, weights=w64)

    for _ in range(warmup):
        step()
    done = 0
    t0 = time.perf_counter()
    while True:
        step()
        done += 1
        el = time.perf_counter() - t0
        if (steps and done >= steps) or (not steps and el >= seconds):
            return done, el


def _host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except Exception:
        return max(1, os.cpu_count() or 1)


def _run_chunks(jobs):
    """The chunk jobs on a process pool of one process per job (started with
    spawn: this process has initialised CUDA)."""
    import multiprocessing as mp
    import oracle
    oracle.build()                      # once, before the children load it
    if len(jobs) == 1:
        return [_oracle_twobit_chunk(jobs[0])]
    with mp.get_context("spawn").Pool(len(jobs)) as pool:
        return pool.map(_oracle_twobit_chunk, jobs)


def cpu_baseline_twobit(seconds: float, m: int | None = None):
    """The oracle as it stands (plain C, one thread per process) on every host
    core at once, each process on its own bounded chunk of the headline
    workload: 8 workers x m elements per step, quantise + dequant-sum + SGD,
    repeated for about `seconds`."""
    cfg_W = 8
    m = m or (1 << 20)
    cores = _host_cores()
    out = _run_chunks([(c, m, 1, 0, seconds) for c in range(cores)])
    rate = sum(cfg_W * m * 4 * st / el for st, el in out)
    steps = sum(st for st, _ in out)
    return {"value": round(rate / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes, each the 8-worker 2-bit step on its own {m} elements per worker "
                      f"({steps} steps in about {seconds:.0f} s, single-threaded C oracle per process)"}


# ----------------------------------------------------------------------------- rows

def _median(xs):
    return float(statistics.median(xs)) if xs else None


def _row(name, kernel, bytes_per_launch, ms_list, peak, unit_elems=None, extra=None):
    ms = _median(ms_list)
    d = {"kernel": kernel, "ms": round(ms, 5), "ms_min": round(min(ms_list), 5), "reps": len(ms_list),
         "bytes": int(bytes_per_launch),
         "GBps": round(bytes_per_launch / (ms * 1e-3) / 1e9, 1),
         "frac": round(bytes_per_launch / (ms * 1e-3) / 1e9 / peak, 3)}
    if unit_elems:
        d["Gelem_per_s"] = round(unit_elems / (ms * 1e-3) / 1e9, 2)
    if extra:
        d.update(extra)
    return d


def rows(args, dev, peak):
    import numpy as np
    import torch
    import gradient_compression_sgd_gc_gb300 as gc
    from gradient_compression_sgd_gc_gb300 import workloads as wl

    stream = torch.cuda.current_stream(dev)
    out = {}
    reps = 20
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)   # 256 MB > L2

    # config 1: one worker, 2^20 elements, fits in L2
    cfg = wl.TWOBIT_W1
    n = cfg.n
    g = wl.twobit_grad(cfg, 0, 0, device=dev)
    r = torch.zeros(n, device=dev)
    c = torch.empty(gc.code_words(n), dtype=torch.int32, device=dev)
    o = torch.empty(n, device=dev)
    tm = Timer(stream)
    pq = gc.gc_2bit_quantize(g, r, c, cfg.threshold, stream=stream, prepare=True)
    pd = gc.gc_2bit_dequant_sum_update([c], n, cfg.threshold, gc.GC_UPD_NONE, out=o, stream=stream,
                                       prepare=True)
    # the launch floor of this timing: the same call on 16 elements (one warp,
    # no work to speak of), timed the same way -- event pair, host submission
    # and kernel launch; the config's single launches sit a few us above it
    g16, r16 = g[:16].clone(), torch.zeros(16, device=dev)
    c16 = torch.empty(gc.code_words(16), dtype=torch.int32, device=dev)
    pf = gc.gc_2bit_quantize(g16, r16, c16, cfg.threshold, stream=stream, prepare=True)
    for i in range(reps + 3):
        flush_l2(flush)
        tm.around("q" if i >= 3 else "w", pq)
        flush_l2(flush)
        tm.around("d" if i >= 3 else "w", pd)
        flush_l2(flush)
        tm.around("f" if i >= 3 else "w", pf)
    for i in range(reps + 3):
        tm.around("qh" if i >= 3 else "w", pq)
    torch.cuda.synchronize(dev)
    floor_ms = _median(tm.ms("f"))

    def above_floor(bytes_, key):
        t = _median(tm.ms(key)) - floor_ms
        return {"launch_floor_ms": round(floor_ms, 5),
                "frac_above_floor": round(bytes_ / (t * 1e-3) / 1e9 / peak, 3) if t > 0 else None}

    out["twobit_w1.launch_floor"] = _row("twobit_w1", "gc_2bit_quantize f32 on 16 elements (L2 flushed): the "
                                         "floor of a single timed launch", 12.25 * 16, tm.ms("f"), peak, 16)
    out["twobit_w1.quantize"] = _row("twobit_w1", "gc_2bit_quantize f32 (L2 flushed)", 12.25 * n,
                                     tm.ms("q"), peak, n, above_floor(12.25 * n, "q"))
    out["twobit_w1.quantize_l2"] = _row("twobit_w1", "gc_2bit_quantize f32 (L2-resident)", 12.25 * n,
                                        tm.ms("qh"), peak, n, above_floor(12.25 * n, "qh"))
    out["twobit_w1.dequant"] = _row("twobit_w1", "gc_2bit_dequant_sum_update NONE W=1", 4.25 * n,
                                    tm.ms("d"), peak, n, above_floor(4.25 * n, "d"))
    # the configuration's ten steps (fresh gradient each step, residual
    # carried, codes dequantised) captured once as a CUDA graph: 20 launches
    # replayed without host launch overhead, against the same calls eagerly
    gs = [wl.twobit_grad(cfg, st, 0, device=dev) for st in range(cfg.steps)]
    cs = [torch.empty(gc.code_words(n), dtype=torch.int32, device=dev) for _ in range(cfg.steps)]
    os_ = [torch.empty(n, device=dev) for _ in range(cfg.steps)]

    def ten_steps():
        for st in range(cfg.steps):
            gc.gc_2bit_quantize(gs[st], r, cs[st], cfg.threshold)
            gc.gc_2bit_dequant_sum_update([cs[st]], n, cfg.threshold, gc.GC_UPD_NONE, out=os_[st])

    def ten_fused():
        # one launch per step: gc_2bit_step with one worker quantises and
        # writes the dequantised values (update kind NONE)
        for st in range(cfg.steps):
            gc.gc_2bit_step([gs[st]], [r], [cs[st]], cfg.threshold, gc.GC_UPD_NONE, out=os_[st])

    graphs = {}
    for key, fn in (("g", ten_steps), ("f", ten_fused)):
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        stream.wait_stream(side)
        graphs[key] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[key]):
            fn()
    # the ten steps in one launch: the residual stays in registers across steps
    r_ms = torch.zeros(n, device=dev)
    pms = gc.gc_2bit_quantize_steps(gs, r_ms, cs, cfg.threshold, out=os_, stream=stream, prepare=True)
    tm = Timer(stream)
    for i in range(reps + 3):
        flush_l2(flush)
        tm.around("g" if i >= 3 else "w", graphs["g"].replay)
        flush_l2(flush)
        tm.around("f" if i >= 3 else "w", graphs["f"].replay)
        flush_l2(flush)
        tm.around("e" if i >= 3 else "w", ten_steps)
        flush_l2(flush)
        tm.around("m" if i >= 3 else "w", pms)
    torch.cuda.synchronize(dev)
    ten_bytes = cfg.steps * (12.25 + 4.25) * n
    one_launch_bytes = (cfg.steps * (4 + 0.25 + 4) + 8) * n
    out["twobit_w1.ten_steps_one_launch"] = _row(
        "twobit_w1", "gc_2bit_quantize_steps: 10 steps (codes + dequantised values) in one launch, residual "
        "read and written once (L2 flushed)", one_launch_bytes, tm.ms("m"), peak, cfg.steps * n,
        {"ten_steps_unfused_bytes_frac": round(ten_bytes / (_median(tm.ms("m")) * 1e-3) / 1e9 / peak, 3)})
    out["twobit_w1.ten_steps_graph"] = _row("twobit_w1", "10 x (gc_2bit_quantize + dequant) as one CUDA graph "
                                            "(L2 flushed before each replay)", ten_bytes, tm.ms("g"), peak,
                                            cfg.steps * n, {"eager_ms": round(_median(tm.ms("e")), 5)})
    out["twobit_w1.ten_fused_steps_graph"] = _row("twobit_w1", "10 x gc_2bit_step (W=1, NONE: quantise + "
                                                  "dequant in one launch) as one CUDA graph (L2 flushed)",
                                                  ten_bytes, tm.ms("f"), peak, cfg.steps * n)
    del g, r, c, o, gs, cs, os_, graphs, r_ms, g16, r16, c16

    # config 2 as one fused launch per step vs the two-launch path of the headline
    cfg2 = wl.TWOBIT_DQ_SGD
    n, W = cfg2.n, cfg2.workers
    g2 = [wl.twobit_grad(cfg2, 0, w, device=dev) for w in range(W)]
    r2 = [torch.zeros(n, device=dev) for _ in range(W)]
    c2 = [torch.empty(gc.code_words(n), dtype=torch.int32, device=dev) for _ in range(W)]
    w2 = wl.twobit_weights(cfg2, device=dev)
    pf = gc.gc_2bit_step(g2, r2, c2, cfg2.threshold, gc.GC_UPD_SGD, lr=cfg2.lr, weights=w2, stream=stream,
                         prepare=True)
    tm = Timer(stream)
    for i in range(reps + 3):
        tm.around("f" if i >= 3 else "w", pf)
    torch.cuda.synchronize(dev)
    out["twobit_dq_sgd.fused_step"] = _row("twobit_dq_sgd", "gc_2bit_step (quantise 8 workers + dequant-sum + SGD)",
                                           (W * 12.25 + 8) * n, tm.ms("f"), peak, W * n,
                                           {"input_gradient_GBps": round(W * n * 4 / (_median(tm.ms("f")) * 1e-3) / 1e9, 1)})
    del g2, r2, c2, w2

    # config 3: QSGD, 4 workers x 61,100,840, bucket 512, s = 7 and s = 127
    for qcfg in (wl.QSGD_S7, wl.QSGD_S127):
        n, W, s = qcfg.n, qcfg.workers, qcfg.s
        vs = [wl.qsgd_grad(qcfg, w, device=dev) for w in range(W)]
        nb = gc.qsgd_num_buckets(n, qcfg.bucket)
        cb = gc.qsgd_code_bytes(n, s)
        norms = [torch.empty(nb, device=dev) for _ in range(W)]
        codes = [torch.empty(cb, dtype=torch.uint8, device=dev) for _ in range(W)]
        outq = torch.empty(n, device=dev)
        tm = Timer(stream)
        pq = [gc.qsgd_quantize(vs[w], qcfg.bucket, s, qcfg.seed, w, norms[w], codes[w], stream=stream,
                               prepare=True) for w in range(W)]
        pd = gc.qsgd_dequant_sum(codes, norms, n, qcfg.bucket, s, 1.0 / W, outq, stream=stream, prepare=True)
        for i in range(22):
            for w in range(W):
                tm.around("q" if i >= 2 else "w", pq[w])
            tm.around("d" if i >= 2 else "w", pd)
        torch.cuda.synchronize(dev)
        out[f"{qcfg.name}.quantize"] = _row(qcfg.name, "qsgd_quantize", n * 4 + cb + 4 * nb, tm.ms("q"),
                                            peak, n, {"issue": issue_roofline(f"qsgd_quantize_s{s}", tm.ms("q"))})
        out[f"{qcfg.name}.dequant_sum"] = _row(qcfg.name, "qsgd_dequant_sum", W * (cb + 4 * nb) + 4 * n,
                                               tm.ms("d"), peak, W * n)
        pm = [gc.qsgd_quantize_maxnorm(vs[w], qcfg.bucket, s, qcfg.seed, w, norms[w], codes[w], stream=stream,
                                       prepare=True) for w in range(W)]
        for i in range(7):
            for w in range(W):
                tm.around("m" if i >= 2 else "w", pm[w])
        torch.cuda.synchronize(dev)
        out[f"{qcfg.name}.quantize_maxnorm"] = _row(qcfg.name, "qsgd_quantize_maxnorm", n * 4 + cb + 4 * nb,
                                                    tm.ms("m"), peak, n,
                                                    {"issue": issue_roofline(f"qsgd_maxnorm_s{s}", tm.ms("m"))})
        # every worker's quantisation + the dequant-sum in one pass
        pst = gc.qsgd_step(vs, qcfg.bucket, s, qcfg.seed, norms, codes, 1.0 / W, outq, stream=stream,
                           prepare=True)
        for i in range(22):
            tm.around("t" if i >= 2 else "w", pst)
        torch.cuda.synchronize(dev)
        sep_ms = W * _median(tm.ms("q")) + _median(tm.ms("d"))
        out[f"{qcfg.name}.step_one_pass"] = _row(qcfg.name, "qsgd_step (4 workers quantised + dequant-sum, one pass)",
                                                 W * (n * 4 + cb + 4 * nb) + 4 * n, tm.ms("t"), peak, W * n,
                                                 {"separate_calls_ms": round(sep_ms, 5),
                                                  "issue": issue_roofline(f"qsgd_step_s{s}", tm.ms("t"))})
        # Elias-omega stream of each worker's (l2-norm) codes, and its decode
        for w in range(W):
            pq[w]()
        cap = gc.qsgd_elias_max_words(n, qcfg.bucket, s)
        words = [torch.empty(cap, dtype=torch.int32, device=dev) for _ in range(W)]
        offs = [torch.empty(nb + 1, dtype=torch.int32, device=dev) for _ in range(W)]
        ews = torch.empty(gc.qsgd_elias_workspace_bytes(n, qcfg.bucket), dtype=torch.uint8, device=dev)
        dcodes = torch.empty(cb, dtype=torch.uint8, device=dev)
        dnorms = torch.empty(nb, device=dev)
        pe = [gc.qsgd_elias_encode(codes[w], norms[w], n, qcfg.bucket, s, words[w], offs[w], ews, stream=stream,
                                   prepare=True) for w in range(W)]
        px = [gc.qsgd_elias_decode(words[w], offs[w], n, qcfg.bucket, s, dcodes, dnorms, stream=stream,
                                   prepare=True) for w in range(W)]
        for i in range(7):
            for w in range(W):
                tm.around("e" if i >= 2 else "w", pe[w])
            for w in range(W):
                tm.around("x" if i >= 2 else "w", px[w])
        torch.cuda.synchronize(dev)
        total = sum(int(o[nb].item()) for o in offs) / W
        bits = {"bits_per_coord": round(32 * total / n, 4),
                "bits_per_coord_with_offsets": round(32 * (total + nb + 1) / n, 4),
                "issue": issue_roofline(f"elias_encode_s{s}", tm.ms("e"))}
        out[f"{qcfg.name}.elias_encode"] = _row(qcfg.name, "qsgd_elias_encode (one pass, look-back)",
                                                cb + 4 * nb + 4 * total + 4 * (nb + 1), tm.ms("e"), peak, n,
                                                bits)
        out[f"{qcfg.name}.elias_decode"] = _row(qcfg.name, "qsgd_elias_decode",
                                                4 * total + 4 * (nb + 1) + cb + 4 * nb, tm.ms("x"), peak, n,
                                                {"issue": issue_roofline(f"elias_decode_s{s}", tm.ms("x"))})
        # the quarter-marked stream of worker 0's codes (the same stream, plus 3
        # marks per bucket) and its decode with one thread per quarter bucket
        marks = torch.empty(3 * nb, dtype=torch.int16, device=dev)
        pme = gc.qsgd_elias_encode_marked(codes[0], norms[0], n, qcfg.bucket, s, words[0], offs[0], marks, ews,
                                          stream=stream, prepare=True)
        pqd = gc.qsgd_elias_decode_quarters(words[0], offs[0], marks, n, qcfg.bucket, s, dcodes, dnorms,
                                            stream=stream, prepare=True)
        for i in range(22):
            tm.around("me" if i >= 2 else "w", pme)
            tm.around("qd" if i >= 2 else "w", pqd)
        torch.cuda.synchronize(dev)
        total0 = int(offs[0][nb].item())
        out[f"{qcfg.name}.elias_encode_marked"] = _row(
            qcfg.name, "qsgd_elias_encode_marked (one pass + quarter marks)",
            cb + 4 * nb + 4 * total0 + 4 * (nb + 1) + 6 * nb, tm.ms("me"), peak, n,
            {"marks_bits_per_coord": round(48 * nb / n, 4)})
        out[f"{qcfg.name}.elias_decode_quarters"] = _row(
            qcfg.name, "qsgd_elias_decode_quarters (a thread per quarter bucket)",
            4 * total0 + 4 * (nb + 1) + 6 * nb + cb + 4 * nb, tm.ms("qd"), peak, n,
            {"issue": issue_roofline(f"elias_quarters_s{s}", tm.ms("qd"))})
        del marks
        # the sparse-regime code (distances between non-zero coordinates) of the
        # same codes, and its decode
        scap = gc.qsgd_elias_sparse_max_words(n, qcfg.bucket)
        swords = torch.empty(scap, dtype=torch.int32, device=dev)
        soffs = torch.empty(nb + 1, dtype=torch.int32, device=dev)
        pse = gc.qsgd_elias_encode_sparse(codes[0], norms[0], n, qcfg.bucket, s, swords, soffs, ews, stream=stream,
                                          prepare=True)
        psd = gc.qsgd_elias_decode_sparse(swords, soffs, n, qcfg.bucket, s, dcodes, dnorms, stream=stream,
                                          prepare=True)
        for i in range(22):
            tm.around("se" if i >= 2 else "w", pse)
            tm.around("sd" if i >= 2 else "w", psd)
        torch.cuda.synchronize(dev)
        stotal = int(soffs[nb].item())
        out[f"{qcfg.name}.elias_sparse_encode"] = _row(
            qcfg.name, "qsgd_elias_encode_sparse (one pass, look-back)", cb + 4 * nb + 4 * stotal + 4 * (nb + 1),
            tm.ms("se"), peak, n, {"bits_per_coord": round(32 * stotal / n, 4)})
        out[f"{qcfg.name}.elias_sparse_decode"] = _row(
            qcfg.name, "qsgd_elias_decode_sparse", 4 * stotal + 4 * (nb + 1) + cb + 4 * nb, tm.ms("sd"), peak, n)
        del swords, soffs
        # the W workers' streams in one launch (the receiver's decode before the sum)
        bcodes = [torch.empty(cb, dtype=torch.uint8, device=dev) for _ in range(W)]
        bnorms = [torch.empty(nb, device=dev) for _ in range(W)]
        pb = gc.qsgd_elias_decode_batched(words, offs, n, qcfg.bucket, s, bcodes, bnorms, stream=stream,
                                          prepare=True)
        for i in range(22):
            tm.around("b" if i >= 2 else "w", pb)
        torch.cuda.synchronize(dev)
        out[f"{qcfg.name}.elias_decode_batched"] = _row(
            qcfg.name, f"qsgd_elias_decode_batched ({W} streams, one launch)",
            W * (4 * total + 4 * (nb + 1) + cb + 4 * nb), tm.ms("b"), peak, W * n,
            {"issue": issue_roofline(f"elias_decode_s{s}", tm.ms("b"), mult=W)})
        del vs, norms, codes, outq, words, offs, ews, dcodes, dnorms, bcodes, bnorms

    # config 5: SAPS + EASGD, 16 workers x 25,557,032, p = 0.01 and 0.001
    for scfg in (wl.SAPS_P01, wl.SAPS_P001):
        n, W = scfg.n, scfg.workers
        models = wl.saps_models(scfg, device=dev)
        center = wl.saps_initial_center(models)
        cap = int(n * scfg.p * 1.2 + 10_000)
        idx = torch.empty(cap, dtype=torch.int32, device=dev)
        vals = [torch.empty(cap, device=dev) for _ in range(W)]
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        ws = torch.empty(gc.saps_workspace_bytes(n), dtype=torch.uint8, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        tm = Timer(stream)
        rounds = 62
        for rd in range(rounds):
            seed_t = gc.saps_round_seed(scfg.base_seed, rd)
            pairs = gc.saps_matching(seed_t, W)
            k = "" if rd >= 2 else "w"
            pm = gc.saps_mask_compact(n, scfg.p, seed_t, models, idx, vals, cnt, ws, st, stream=stream,
                                      prepare=True)
            pa = gc.saps_peer_average(models, vals, idx, cnt, pairs, stream=stream, prepare=True)
            pe = gc.easgd_step(models, scfg.alpha, scfg.beta, center, stream=stream, prepare=True)
            pf = gc.saps_average_easgd_step(models, vals, cnt, pairs, scfg.alpha, scfg.beta, center, ws,
                                            stream=stream, prepare=True)
            pr = gc.saps_round(n, scfg.p, seed_t, models, pairs, scfg.alpha, scfg.beta, center, idx, vals,
                               cnt, ws, st, stream=stream, prepare=True)
            if rd % 3 == 2:
                tm.around("r" + k, pr)
                continue
            tm.around("m" + k, pm)
            if rd % 3 == 0:
                tm.around("a" + k, pa)
                tm.around("e" + k, pe)
            else:
                tm.around("f" + k, pf)
        # the same compaction with this process's L2 fetch granularity at 32
        # bytes (gc_l2_fetch_granularity; the gather's random 4-byte reads then
        # fetch less per value), after the same streaming step as above
        torch.cuda.synchronize(dev)
        prev = gc.gc_l2_fetch_granularity(32)
        for i in range(22):
            pe()
            tm.around("g" if i >= 2 else "w", pm)
        torch.cuda.synchronize(dev)
        gc.gc_l2_fetch_granularity(prev)
        K = int(cnt.item())
        assert int(st.item()) == 0
        rm = tm.ms("m")
        mkey = "saps_mask" if scfg.p >= 0.01 else "saps_mask_p001"
        g_ms = _median(tm.ms("g"))
        out[f"{scfg.name}.mask_compact"] = _row(scfg.name, "saps_mask_compact", 4 * K + W * 8 * K, rm, peak, n,
                                                {"masked": K, "issue": issue_roofline(mkey, rm),
                                                 "dram": dram_roofline(mkey, rm, peak),
                                                 "l2_fetch_32B_ms": round(g_ms, 5),
                                                 "l2_fetch_32B_frac": round((4 * K + W * 8 * K) / (g_ms * 1e-3)
                                                                            / 1e9 / peak, 4)})
        out[f"{scfg.name}.peer_average"] = _row(scfg.name, "saps_peer_average", (W // 2) * 20 * K,
                                                tm.ms("a"), peak, None,
                                                {"dram": dram_roofline("saps_avg", tm.ms("a"), peak)
                                                 if scfg.p >= 0.01 else None})
        out[f"{scfg.name}.easgd"] = _row(scfg.name, "easgd_step", (2 * W + 2) * 4 * n, tm.ms("e"), peak, W * n)
        out[f"{scfg.name}.average_easgd_fused"] = _row(scfg.name, "saps_average_easgd_step",
                                                       (2 * W + 2) * 4 * n + W * 4 * K + n // 4,
                                                       tm.ms("f"), peak, W * n)
        round_bytes = 4 * K + W * 8 * K + W * 4 * K + (2 * W + 2) * 4 * n + n // 4
        round_ms = _median(rm) + _median(tm.ms("f"))
        out[f"{scfg.name}.round"] = {"ms": round(round_ms, 4), "bytes": int(round_bytes),
                                     "kernels": "saps_mask_compact + saps_average_easgd_step",
                                     "frac": round(round_bytes / (round_ms * 1e-3) / 1e9 / peak, 3)}
        one_pass_bytes = 4 * K + W * 4 * K + (2 * W + 2) * 4 * n
        out[f"{scfg.name}.round_one_pass"] = _row(scfg.name, "saps_round (mask + compaction + pair average + "
                                                  "elastic step, one pass)", one_pass_bytes, tm.ms("r"), peak,
                                                  W * n, {"masked": K})
        del models, center, vals, idx

    # config 4: CD-SGD, 4 workers x 1.3e9 bf16
    ccfg = wl.CDSGD
    n, W = ccfg.n, ccfg.workers
    try:
        grads = [wl.twobit_grad(ccfg, 1, w, device=dev) for w in range(W)]
        res = [torch.zeros(n, device=dev) for _ in range(W)]
        codes = [torch.empty(gc.code_words(n), dtype=torch.int32, device=dev) for _ in range(W)]
        wts = wl.twobit_weights(ccfg, device=dev, seed=8)
        tm = Timer(stream)
        pq = [gc.gc_2bit_quantize(grads[w], res[w], codes[w], ccfg.threshold, stream=stream, prepare=True)
              for w in range(W)]
        pd = gc.gc_2bit_dequant_sum_update(codes, n, ccfg.threshold, gc.GC_UPD_SGD, lr=ccfg.lr, weights=wts,
                                           stream=stream, prepare=True)
        pc = gc.gc_compensated_sum_update(grads, res, ccfg.lr, wts, stream=stream, prepare=True)
        local = [torch.empty(n, device=dev) for _ in range(W)]
        pl = gc.gc_2bit_quantize_local(grads, res, codes, wts, local, ccfg.threshold, 0.1, stream=stream,
                                       prepare=True)
        # the compressed step in one pass: all 4 workers quantised + dequant-sum
        # + SGD (gc_2bit_step), and the same with eq. 11 local weights
        ps = gc.gc_2bit_step(grads, res, codes, ccfg.threshold, gc.GC_UPD_SGD, lr=ccfg.lr, weights=wts,
                             stream=stream, prepare=True)
        psl = gc.gc_2bit_step(grads, res, codes, ccfg.threshold, gc.GC_UPD_SGD, lr=ccfg.lr, weights=wts,
                              stream=stream, prepare=True, local_weights=local, local_lr=0.1)
        for i in range(21):
            k = "" if i >= 1 else "w"
            for w in range(W):
                tm.around("q" + k, pq[w])
            tm.around("d" + k, pd)
            tm.around("c" + k, pc)
            tm.around("l" + k, pl)
            tm.around("s" + k, ps)
            tm.around("t" + k, psl)
        torch.cuda.synchronize(dev)
        out["cdsgd.step_one_pass"] = _row("cdsgd", "gc_2bit_step bf16 W=4 (quantise all + dequant-sum + SGD, one pass)",
                                          (W * 10.25 + 8) * n, tm.ms("s"), peak, W * n,
                                          {"separate_calls_ms": round(W * _median(tm.ms("q")) + _median(tm.ms("d")), 5)})
        out["cdsgd.step_one_pass_local"] = _row("cdsgd", "gc_2bit_step_local bf16 W=4 (+ eq. 11 local weights)",
                                                (W * 14.25 + 8) * n, tm.ms("t"), peak, W * n,
                                                {"separate_calls_ms": round(_median(tm.ms("l")) + _median(tm.ms("d")), 5)})
        out["cdsgd.quantize_local_update"] = _row("cdsgd", "gc_2bit_quantize_local bf16 W=4 (eq. 11 local weights)",
                                                  (W * (2 + 8 + 0.25 + 4) + 4) * n, tm.ms("l"), peak, W * n)
        del local
        out["cdsgd.quantize_bf16"] = _row("cdsgd", "gc_2bit_quantize bf16", 10.25 * n, tm.ms("q"), peak, n)
        out["cdsgd.dequant_sum_sgd"] = _row("cdsgd", "gc_2bit_dequant_sum_update SGD W=4", (W * 0.25 + 8) * n,
                                            tm.ms("d"), peak, n)
        out["cdsgd.correction"] = _row("cdsgd", "gc_compensated_sum_update bf16 W=4", (W * 10 + 8) * n,
                                       tm.ms("c"), peak, W * n)
        del grads, res, codes, wts
    except torch.cuda.OutOfMemoryError as e:      # pragma: no cover
        out["cdsgd"] = {"skipped": f"out of memory: {e}"}
    torch.cuda.empty_cache()
    return out


def qsgd_level_mismatches(dev, chunks_per_worker: int = 16, chunk: int = 1 << 20):
    """Part of the oracle leg (outside every timed region): the full-size QSGD
    configurations are quantised on the GPU, and on a bounded sample of each
    worker's vector (``chunks_per_worker`` bucket-aligned chunks of ``chunk``
    elements, the first and last included) the GPU's codes are compared with
    the oracle's.  A level that differs by one where the oracle's deciding
    value x = |v| * (s / norm) + u lies within 1e-6 of an integer is a
    boundary mismatch (counted); any other difference, or a sign difference,
    is a violation (must be 0)."""
    import numpy as np
    import torch
    import gradient_compression_sgd_gc_gb300 as gc
    from gradient_compression_sgd_gc_gb300 import workloads as wl
    import oracle

    def levels(codes, n, s):
        if s <= 7:
            c = np.empty(2 * codes.size, np.uint8)
            c[0::2], c[1::2] = codes >> 4, codes & 0xF
            c = c[:n]
            return c >> 3, c & 7
        return codes[:n] >> 7, codes[:n] & 0x7F

    out = {}
    for qcfg in (wl.QSGD_S7, wl.QSGD_S127):
        n, W, s, d = qcfg.n, qcfg.workers, qcfg.s, qcfg.bucket
        rng = np.random.default_rng(1234 + s)
        starts = {0, (n - 1) // chunk * chunk}
        starts |= {int(x) // d * d for x in rng.integers(0, n, chunks_per_worker - 2)}
        mism = viol = norms_diff = elems = 0
        t0 = time.time()
        for w in range(W):
            v = wl.qsgd_grad(qcfg, w, device=dev)
            nb, cb = gc.qsgd_num_buckets(n, d), gc.qsgd_code_bytes(n, s)
            norms = torch.empty(nb, device=dev)
            codes = torch.empty(cb, dtype=torch.uint8, device=dev)
            gc.qsgd_quantize(v, d, s, qcfg.seed, w, norms, codes)
            torch.cuda.synchronize(dev)
            for lo in sorted(starts):
                hi = min(n, lo + chunk)
                vh = v[lo:hi].cpu().numpy()
                rn, rc = oracle.qsgd_quantize(vh, d, s, qcfg.seed, w, i0=lo)
                gn = norms[lo // d:(hi + d - 1) // d].cpu().numpy()
                norms_diff += int((gn != rn).sum())
                gcodes = (codes[lo // 2:(hi + 1) // 2] if s <= 7 else codes[lo:hi]).cpu().numpy()
                elems += hi - lo
                if np.array_equal(gcodes, rc):
                    continue
                gs, gl = levels(gcodes, hi - lo, s)
                rs, rl = levels(rc, hi - lo, s)
                viol += int((gs != rs).sum())
                bad = gl != rl
                x = oracle.qsgd_scaled_values(vh, d, s, qcfg.seed, w, i0=lo)[bad].astype(np.float64)
                k = np.maximum(gl[bad], rl[bad]).astype(np.float64)
                near = (np.abs(gl[bad].astype(int) - rl[bad].astype(int)) == 1) & (np.abs(x - k) <= 1e-6)
                mism += int(near.sum())
                viol += int((~near).sum())
            del v, norms, codes
        out[f"s{s}"] = {"mismatches": mism, "violations": viol, "norms_differing": norms_diff,
                        "elements_checked": elems,
                        "sample": f"{len(starts)} chunks of {chunk} elements per worker x {W} workers "
                                  f"(n = {n}, bucket {d}), first and last included",
                        "oracle_s": round(time.time() - t0, 1)}
    torch.cuda.empty_cache()
    return out


def row_fracs(rows_: dict) -> dict:
    """Compact per-row fractions, [HBM frac of measured peak, issue frac,
    DRAM-bytes frac] (null where a roofline does not apply)."""
    out = {}
    for k, r in rows_.items():
        if not isinstance(r, dict) or "frac" not in r:
            continue
        iss = r.get("issue")
        dram = r.get("dram")
        out[k] = [r["frac"], iss.get("frac") if isinstance(iss, dict) else None,
                  dram.get("frac") if isinstance(dram, dict) else None]
    return out


def cpu_rows(seconds_each: float = 1.5):
    """The oracle timed on bounded samples of each row's workload (one thread)."""
    import numpy as np
    import oracle
    from gradient_compression_sgd_gc_gb300 import workloads as wl

    def timed(fn, units):
        n_it = 0
        t0 = time.perf_counter()
        while True:
            fn()
            n_it += 1
            el = time.perf_counter() - t0
            if el >= seconds_each:
                return units * n_it / el

    out = {}
    m = 1 << 20
    g = wl.normal(m, 1.0, 0).numpy()
    r = np.zeros(m, np.float32)
    out["twobit_w1"] = {"Gelem_per_s": round(timed(lambda: oracle.twobit_quantize(g, r, 0.5), m) / 1e9, 5)}
    qcfg = wl.scaled(wl.QSGD_S7, m)
    v = wl.qsgd_grad(qcfg, 0).numpy()
    out["qsgd_s7"] = {"Gelem_per_s": round(timed(lambda: oracle.qsgd_quantize(v, 512, 7, 42, 0), m) / 1e9, 5)}
    out["qsgd_s127"] = {"Gelem_per_s": round(timed(lambda: oracle.qsgd_quantize(v, 512, 127, 42, 0), m) / 1e9, 5)}
    gb = wl.normal(m, 5e-4, 1, dtype=__import__("torch").bfloat16).view(__import__("torch").int16).numpy().view(np.uint16)
    rb = np.zeros(m, np.float32)
    out["cdsgd"] = {"Gelem_per_s": round(timed(lambda: oracle.twobit_quantize(gb, rb, 1e-3), m) / 1e9, 5)}
    W = 16
    models = [wl.normal(m, 0.05, 4000 + w).numpy().astype(np.float64) for w in range(W)]
    cen = np.mean(models, axis=0)

    def saps_round():
        K, idx, vals = oracle.saps_mask_compact(m, 0.01, 77, models)
        oracle.saps_peer_average(models, vals, idx, oracle.saps_matching(77, W))
        oracle.easgd_step(models, 0.9, 0.9, cen)
    out["saps_p01"] = {"Gelem_per_s": round(timed(saps_round, W * m) / 1e9, 5)}
    for k in out:
        out[k].update({"cores": 1, "kind": "oracle", "sample": f"{m} elements per worker"})
    return out


# ----------------------------------------------------------------------------- reference arm

def reference_arm(args, rank, world, pg):
    """The CPU oracle as it stands, on the host cores, on bounded samples of
    the headline workload (8 workers, 2-bit quantise + dequant-sum + SGD)."""
    import numpy as np
    import oracle
    from gradient_compression_sgd_gc_gb300 import workloads as wl

    if rank != 0:
        return None
    cfg = wl.TWOBIT_DQ_SGD
    W, t, lr = cfg.workers, cfg.threshold, cfg.lr
    total_steps = args.steps + args.warmup
    budget = 90.0
    per_step = min(1.0, budget / max(1, total_steps))
    cores = _host_cores()
    # calibrate each process's chunk so that one step takes about per_step
    # seconds (one process, then every core running the same size)
    m = 1 << 14
    st, el = _oracle_twobit_chunk((0, m, 1, 3, 0.0))
    one = el / st
    m = int(max(1 << 10, min(cfg.n // cores, m * per_step / max(one, 1e-6)))) // 16 * 16
    out = _run_chunks([(c, m, args.warmup, args.steps, 0.0) for c in range(cores)])
    ms = max(el / st for st, el in out) * 1e3
    value = cores * W * m * 4 / (ms * 1e-3) / 1e9
    sample = (f"{cores} x {m} of {cfg.n} elements per worker per step, one single-threaded C oracle "
              f"process per host core")
    return {"impl": "reference", "metric": HEADLINE_METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "twobit_dq_sgd: 8 workers x 25,557,032 fp32, t=2e-3, lr=0.1 (sampled)",
                       "sample_elements_per_worker": cores * m},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- profiling cases

CASES = ("quantize_f32", "quantize_bf16", "quantize_batched", "step_fused", "dqsum_sgd", "saps_fused", "qsgd_quantize_s7", "qsgd_quantize_s127",
         "qsgd_dequant_s7", "qsgd_dequant_s127", "saps_mask", "saps_avg", "easgd", "compensated",
         "elias_encode_s7", "elias_encode_s127", "elias_decode_s7", "elias_decode_s127",
         "quantize_local", "qsgd_maxnorm_s7", "qsgd_maxnorm_s127", "saps_mask_p001", "saps_round",
         "qsgd_step_s7", "qsgd_step_s127", "step_bf16", "multi_step", "elias_sparse_encode_s7",
         "elias_sparse_encode_s127", "elias_sparse_decode_s7", "elias_sparse_decode_s127", "elias_quarters_s7",
         "elias_quarters_s127")


def run_case(name: str, n: int):
    """One kernel on inputs larger than L2 but a few GB at most, launched three
    times; used as the command under ncu."""
    import torch
    import gradient_compression_sgd_gc_gb300 as gc
    from gradient_compression_sgd_gc_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = n or (1 << 26)
    if name in ("quantize_f32", "quantize_bf16"):
        dt = torch.float32 if name == "quantize_f32" else torch.bfloat16
        g = wl.normal(n, 1e-3, 1, device=dev, dtype=dt)
        r = torch.zeros(n, device=dev)
        c = torch.empty(gc.code_words(n), dtype=torch.int32, device=dev)
        fn = lambda: gc.gc_2bit_quantize(g, r, c, 2e-3)
    elif name == "quantize_batched":
        W = 8
        m = n // W
        gs = [wl.normal(m, 1e-3, 1 + w, device=dev) for w in range(W)]
        rs = [torch.zeros(m, device=dev) for _ in range(W)]
        cs = [torch.empty(gc.code_words(m), dtype=torch.int32, device=dev) for _ in range(W)]
        fn = lambda: gc.gc_2bit_quantize_batched(gs, rs, cs, 2e-3)
    elif name == "step_fused":
        W = 8
        m = n // W
        gs = [wl.normal(m, 1e-3, 1 + w, device=dev) for w in range(W)]
        rs = [torch.zeros(m, device=dev) for _ in range(W)]
        cs = [torch.empty(gc.code_words(m), dtype=torch.int32, device=dev) for _ in range(W)]
        wt = torch.zeros(m, device=dev)
        fn = lambda: gc.gc_2bit_step(gs, rs, cs, 2e-3, gc.GC_UPD_SGD, lr=0.1, weights=wt)
    elif name == "step_bf16":
        W = 4
        m = n // W
        gs = [wl.normal(m, 5e-4, 1 + w, device=dev, dtype=torch.bfloat16) for w in range(W)]
        rs = [torch.zeros(m, device=dev) for _ in range(W)]
        cs = [torch.empty(gc.code_words(m), dtype=torch.int32, device=dev) for _ in range(W)]
        wt = torch.zeros(m, device=dev)
        fn = lambda: gc.gc_2bit_step(gs, rs, cs, 1e-3, gc.GC_UPD_SGD, lr=0.01, weights=wt)
    elif name == "multi_step":
        S = 10
        m = n // S
        gs = [wl.normal(m, 1.0, st, device=dev) for st in range(S)]
        r = torch.zeros(m, device=dev)
        cs = [torch.empty(gc.code_words(m), dtype=torch.int32, device=dev) for _ in range(S)]
        os_ = [torch.empty(m, device=dev) for _ in range(S)]
        fn = lambda: gc.gc_2bit_quantize_steps(gs, r, cs, 0.5, out=os_)
    elif name == "dqsum_sgd":
        W = 8
        cs = [torch.randint(-2 ** 31, 2 ** 31 - 1, (gc.code_words(n),), dtype=torch.int32, device=dev)
              for _ in range(W)]
        w = torch.zeros(n, device=dev)
        fn = lambda: gc.gc_2bit_dequant_sum_update(cs, n, 2e-3, gc.GC_UPD_SGD, lr=0.1, weights=w)
    elif name == "quantize_local":
        W = 4
        m = n // W
        gs = [wl.normal(m, 5e-4, 1 + w, device=dev, dtype=torch.bfloat16) for w in range(W)]
        rs = [torch.zeros(m, device=dev) for _ in range(W)]
        cs = [torch.empty(gc.code_words(m), dtype=torch.int32, device=dev) for _ in range(W)]
        wt = torch.zeros(m, device=dev)
        loc = [torch.empty(m, device=dev) for _ in range(W)]
        fn = lambda: gc.gc_2bit_quantize_local(gs, rs, cs, wt, loc, 1e-3, 0.1)
    elif name.startswith("qsgd_step"):
        s = 7 if name.endswith("s7") else 127
        W = 4
        m = n // W
        vs = [wl.qsgd_grad(wl.scaled(wl.QSGD_S7, m), w, device=dev) for w in range(W)]
        nms = [torch.empty(gc.qsgd_num_buckets(m, 512), device=dev) for _ in range(W)]
        cs = [torch.empty(gc.qsgd_code_bytes(m, s), dtype=torch.uint8, device=dev) for _ in range(W)]
        out = torch.empty(m, device=dev)
        fn = lambda: gc.qsgd_step(vs, 512, s, 42, nms, cs, 0.25, out)
    elif name.startswith("qsgd_maxnorm"):
        s = 7 if name.endswith("s7") else 127
        v = wl.qsgd_grad(wl.scaled(wl.QSGD_S7, n), 0, device=dev)
        nm = torch.empty(gc.qsgd_num_buckets(n, 512), device=dev)
        c = torch.empty(gc.qsgd_code_bytes(n, s), dtype=torch.uint8, device=dev)
        fn = lambda: gc.qsgd_quantize_maxnorm(v, 512, s, 42, 0, nm, c)
    elif name.startswith("qsgd_quantize"):
        s = 7 if name.endswith("s7") else 127
        v = wl.qsgd_grad(wl.scaled(wl.QSGD_S7, n), 0, device=dev)
        nm = torch.empty(gc.qsgd_num_buckets(n, 512), device=dev)
        c = torch.empty(gc.qsgd_code_bytes(n, s), dtype=torch.uint8, device=dev)
        fn = lambda: gc.qsgd_quantize(v, 512, s, 42, 0, nm, c)
    elif name.startswith("qsgd_dequant"):
        s = 7 if name.endswith("s7") else 127
        W = 4
        nb = gc.qsgd_num_buckets(n, 512)
        cs = [torch.randint(0, 255, (gc.qsgd_code_bytes(n, s),), dtype=torch.uint8, device=dev)
              for _ in range(W)]
        nms = [torch.rand(nb, device=dev) for _ in range(W)]
        out = torch.empty(n, device=dev)
        fn = lambda: gc.qsgd_dequant_sum(cs, nms, n, 512, s, 0.25, out)
    elif name.startswith("elias_"):
        s = 7 if name.endswith("s7") else 127
        v = wl.qsgd_grad(wl.scaled(wl.QSGD_S7, n), 0, device=dev)
        nb = gc.qsgd_num_buckets(n, 512)
        nm = torch.empty(nb, device=dev)
        c = torch.empty(gc.qsgd_code_bytes(n, s), dtype=torch.uint8, device=dev)
        gc.qsgd_quantize(v, 512, s, 42, 0, nm, c)
        words = torch.empty(gc.qsgd_elias_max_words(n, 512, s), dtype=torch.int32, device=dev)
        offs = torch.empty(nb + 1, dtype=torch.int32, device=dev)
        ews = torch.empty(gc.qsgd_elias_workspace_bytes(n, 512), dtype=torch.uint8, device=dev)
        gc.qsgd_elias_encode(c, nm, n, 512, s, words, offs, ews)
        # each encoder call starts from an L2 filled with other (clean) data
        # -- a read of a buffer larger than L2, no write-back to come -- so
        # that a capture without cache control sees the codes come from DRAM
        flush = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)
        flush_l2 = lambda buf: buf.sum()
        if name.startswith("elias_sparse"):
            sw = torch.empty(gc.qsgd_elias_sparse_max_words(n, 512), dtype=torch.int32, device=dev)
            gc.qsgd_elias_encode_sparse(c, nm, n, 512, s, sw, offs, ews)
            if name.startswith("elias_sparse_encode"):
                fn = lambda: (flush_l2(flush), gc.qsgd_elias_encode_sparse(c, nm, n, 512, s, sw, offs, ews))
            else:
                dc = torch.empty_like(c)
                dn = torch.empty_like(nm)
                fn = lambda: gc.qsgd_elias_decode_sparse(sw, offs, n, 512, s, dc, dn)
        elif name.startswith("elias_quarters"):
            marks = torch.empty(3 * nb, dtype=torch.int16, device=dev)
            gc.qsgd_elias_encode_marked(c, nm, n, 512, s, words, offs, marks, ews)
            dc = torch.empty_like(c)
            dn = torch.empty_like(nm)
            fn = lambda: gc.qsgd_elias_decode_quarters(words, offs, marks, n, 512, s, dc, dn)
        elif name.startswith("elias_encode"):
            fn = lambda: (flush_l2(flush), gc.qsgd_elias_encode(c, nm, n, 512, s, words, offs, ews))
        else:
            dc = torch.empty_like(c)
            dn = torch.empty_like(nm)
            fn = lambda: gc.qsgd_elias_decode(words, offs, n, 512, s, dc, dn)
    elif name in ("saps_mask", "saps_mask_p001", "saps_avg", "easgd", "saps_fused", "saps_round"):
        base = wl.SAPS_P001 if name == "saps_mask_p001" else wl.SAPS_P01
        cfg = wl.scaled(base, n if name not in ("easgd", "saps_fused", "saps_round") else n // 4)
        models = wl.saps_models(cfg, device=dev)
        cap = int(cfg.n * cfg.p * 1.2 + 10_000)
        idx = torch.empty(cap, dtype=torch.int32, device=dev)
        vals = [torch.empty(cap, device=dev) for _ in range(cfg.workers)]
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        ws = torch.empty(gc.saps_workspace_bytes(cfg.n), dtype=torch.uint8, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        center = wl.saps_initial_center(models)
        seed_t = gc.saps_round_seed(5, 0)
        pairs = gc.saps_matching(seed_t, cfg.workers)
        gc.saps_mask_compact(cfg.n, cfg.p, seed_t, models, idx, vals, cnt, ws, st)
        if name in ("saps_mask", "saps_mask_p001"):
            fn = lambda: gc.saps_mask_compact(cfg.n, cfg.p, seed_t, models, idx, vals, cnt, ws, st)
        elif name == "saps_avg":
            fn = lambda: gc.saps_peer_average(models, vals, idx, cnt, pairs)
        elif name == "saps_fused":
            fn = lambda: gc.saps_average_easgd_step(models, vals, cnt, pairs, 0.9, 0.9, center, ws)
        elif name == "saps_round":
            fn = lambda: gc.saps_round(cfg.n, cfg.p, seed_t, models, pairs, 0.9, 0.9, center, idx, vals, cnt, ws, st)
        else:
            fn = lambda: gc.easgd_step(models, 0.9, 0.9, center)
    elif name == "compensated":
        W = 4
        gs = [wl.normal(n, 5e-4, w, device=dev, dtype=torch.bfloat16) for w in range(W)]
        rs = [torch.zeros(n, device=dev) for _ in range(W)]
        w = torch.zeros(n, device=dev)
        fn = lambda: gc.gc_compensated_sum_update(gs, rs, 0.01, w)
    else:
        raise SystemExit(f"unknown case {name}; one of {CASES}")
    for _ in range(3):
        fn()
    torch.cuda.synchronize(dev)
    print(f"case {name} n={n}: 3 launches done")


# ----------------------------------------------------------------------------- main

def main():
    args = parse_args()
    if args.case:
        run_case(args.case, args.case_n)
        return
    rank, world, local, pg = dist_setup(args)
    if args.impl == "reference":
        line = reference_arm(args, rank, world, pg)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peaks()

    h = headline(args, dev, rank, world, pg)
    n, W = h["n"], h["W"]
    total_s = h["total_ms"] * 1e-3
    units = W * n * args.steps * world
    value = units * 4 / total_s / 1e9
    q_ms = statistics.mean(h["quantize_ms"])
    algo_bytes = 12.25 * n * W            # one batched launch quantises all W buffers
    achieved = algo_bytes / (q_ms * 1e-3) / 1e9
    line = {
        "metric": HEADLINE_METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(h["total_ms"] / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "twobit_dq_sgd: 8 workers x 25,557,032 fp32 gradients (ResNet-50-sized), "
                               "g~N(0,1e-3^2), t=2e-3, 2-bit quantise + residual per worker, then "
                               "dequant-sum + SGD w-=0.1*avg",
                   "workers": W, "elements_per_worker": n, "parallelism": f"replicas x{world} (weak)",
                   "l2": "inputs larger than L2 (818 MB of gradients per step, 20 pre-generated steps cycled)"},
        "elements_per_s": round(units / total_s, 1),
        "hbm_frac_step": round((W * 12.25 + (W * 0.25 + 8)) * n / (h["total_ms"] / args.steps * 1e-3) / 1e9
                               / peak, 4),
        "roofline": {"bound": "hbm", "kernel": "gc_2bit_quantize_batched (fp32, 8 buffers per launch)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": ncu_traffic("gc_2bit_quantize_batched_f32"),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback",
                     "algorithmic_bytes_per_launch": int(algo_bytes),
                     "avg_launch_ms": round(q_ms, 5),
                     "dqsum_avg_launch_ms": round(statistics.mean(h["dqsum_ms"]), 5),
                     "dqsum_frac": round((W * 0.25 + 8) * n / (statistics.mean(h["dqsum_ms"]) * 1e-3) / 1e9
                                         / peak, 4)},
        "gpu_launches": h["launches"],
        "clocks": h["clocks"],
    }
    e2e_line = e2e(args, dev, pg, world)
    if rank == 0:
        line["e2e"] = e2e_line
        if world == 1 and not args.no_rows:
            line["rows"] = rows(args, dev, peak)
        if world == 1 and not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline_twobit(args.cpu_seconds)
            if not args.no_rows:
                line["cpu_rows"] = cpu_rows()
                line["qsgd_level_mismatches"] = qsgd_level_mismatches(dev)
        if "rows" in line:
            # last key: the record of a run keeps only the end of stdout
            line["row_fracs"] = row_fracs(line["rows"])
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
