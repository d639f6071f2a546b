#!/usr/bin/env python3
"""Throughput of the fused attention forward on GB300.

One step = one fused forward (S = Q K^T, online softmax, O = P V, O/l, LSE)
over one batch of the workload, through the C ABI ``fa_fwd``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line.  ``value`` is whole-job TFLOP/s with inputs resident in
device memory, timed with CUDA events on the launching stream; FLOPs per step
are 4 B H N^2 d, halved for causal attention.  ``e2e`` is the same metric with
the pinned-host -> device copies of Q, K, V and the device -> host copies of
O and LSE inside the timed region.  ``--impl reference`` times the fp64 CPU
oracle (three-pass route) on the host cores on a bounded sample of rows.

Multi-GPU (torchrun, one rank per GPU): every rank runs the whole workload on
its own seeded inputs (independent problems, no collective on the data path),
so scaling is weak; timing is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16, 1 GB300) and % of dense BF16 tensor peak"
FALLBACK_BF16_TFLOPS = 1900.0  # used only when MEASURED_PEAKS.json is absent
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
FALLBACK_HBM_GBS = 6800.0
SOFTMAX_METRIC = "row softmax GB/s (fp32, online normaliser, 1 GB300) and % of HBM copy bandwidth"
KERNEL_NAME = "fa_fwd_sm103"
L2_BYTES = 129 * 1024 * 1024


def workload_flops(w) -> float:
    """4 B H N^2 d, halved when causal; under a window or document mask, 4 d per visible (query, key) pair."""
    if w.masked:
        from online_softmax_04_gb300 import workloads as wl

        return 4.0 * w.d * float(wl.visible_pairs(w))
    f = 4.0 * w.B * w.H * float(w.N) ** 2 * w.d
    return f / 2 if w.causal else f


def row_flops(w, rows) -> float:
    """The metric's FLOPs attributable to the given query rows: 4 d per visible key."""
    import numpy as np

    if w.masked:
        from online_softmax_04_gb300 import workloads as wl

        return float(4.0 * w.d * wl.visible_per_row(w, rows).sum())
    i = np.asarray(rows) % w.N
    n_vis = (i + 1) if w.causal else np.full(len(i), w.N)
    return float(4.0 * w.d * n_vis.sum())


def oracle_rows(w, q, k, v, rows, return_threads: bool = False):
    """The oracle's three-pass route for the given rows, under the workload's mask if any."""
    import oracle

    if w.masked:
        from online_softmax_04_gb300 import workloads as wl

        o, lse = oracle.attention_masked(q, k, v, w.scale, w.window_left, w.window_right, wl.make_doc_ids(w),
                                         rows=rows, n_threads=0)
        return (o, lse, os.cpu_count() or 1) if return_threads else (o, lse)
    return oracle.attention_three_pass(q, k, v, w.causal, w.scale, rows=rows, return_threads=return_threads)


def l2_policy(w) -> tuple[bool, str]:
    """Whether timed steps flush L2 first (inputs smaller than ~L2), and the sentence saying so."""
    in_bytes = 3 * w.B * w.H * w.N * w.d * 2
    if in_bytes < 1.25 * L2_BYTES:
        return True, "L2 flushed (512 MB write, then 256 MB read) before each individually timed step"
    return False, (f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB of Q, K, V > 129 MB), "
                   "back-to-back steps, no flush")


def bench_config(w, world: int) -> dict:
    """The workload part of the JSON line, shared by both arms so that their configs compare equal."""
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "scale": "1/sqrt(d)", "flops_per_step_per_gpu": workload_flops(w), "l2": l2_policy(w)[1],
            "parallelism": f"independent problem per GPU x{world}",
            **({"window_left": w.window_left, "window_right": w.window_right, "doc_mean": w.doc_mean,
                "flops": "4 d per visible (query, key) pair"} if w.masked else {})}


def algorithmic_bytes(w) -> float:
    """Q, K, V read and O written once (bf16), LSE written once (fp32)."""
    return 2.0 * 4 * w.B * w.H * w.N * w.d + 4.0 * w.B * w.H * w.N


def hbm_side(w, ms_step: float) -> dict:
    peak, src = measured_peak("hbm_gbs")
    gbs = algorithmic_bytes(w) / (ms_step * 1e-3) / 1e9
    return {"achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "bytes_per_step": algorithmic_bytes(w), "peak_source": src}


def rank_workload(w, rank: int):
    """Every rank solves its own problem: the same shapes, its own seed."""
    return w.with_(seed=w.seed + 1000 * rank)


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time (a no-op for a single process)."""
    if dist is None:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank: float, steps: int, ms_total: float) -> float:
    """Aggregate throughput: all ranks' FLOPs over the slowest rank's time."""
    return world * flops_per_rank * steps / (ms_total * 1e-3) / 1e12


class L2Flush:
    """Evicts L2 between timed steps: writes a 512 MB buffer (more than L2), then
    reads a second, 256 MB one, so that the dirty lines of the write are written
    back before the timed region starts rather than during it."""

    def __init__(self, torch, dev):
        self.write = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.read = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.write.fill_(1)
        self.read.sum()


def measured_peak(key: str = "bf16_tflops"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j[key]), "measured"
    except Exception:
        return ({"bf16_tflops": FALLBACK_BF16_TFLOPS, "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED}
                .get(key, FALLBACK_HBM_GBS)), "fallback"


def strip_c_comments(text: str) -> str:
    """C/C++ source without its comments (string literals kept), for hashing what compiles."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":
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
    return "".join(out)


# the csrc/ files each profiled kernel compiles from (fa_fwd.cu holds every launcher)
KERNEL_SOURCES = {
    KERNEL_NAME: ("fa_fwd.cu", "fa_fwd_kernel.cuh", "fa_fwd_two_kernel.cuh", "sm103_ptx.cuh"),
    "softmax_rows_smem": ("fa_fwd.cu", "softmax_rows.cuh", "sm103_ptx.cuh"),
}


def kernel_source_hash(kernel: str = KERNEL_NAME) -> str:
    """sha256 prefix of the csrc/ files `kernel` compiles from (all of them for a kernel not
    listed), comments removed: a traffic record stays valid across comment edits and lapses
    with any change to what the kernel compiles from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "online_softmax_04_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel)
    for name in sorted(os.listdir(csrc)):
        if names is not None and name not in names:
            continue
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            # lines left blank by the comments are dropped, so adding or removing a
            # comment line does not change the hash either
            lines = (ln.rstrip() for ln in strip_c_comments(f.read()).splitlines())
            h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str = KERNEL_NAME):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 3 and parts[0] == workload and parts[1] == want:
                return float(parts[2])
    return None


def step_stats(ms_list):
    """Min / median / max of the individually timed steps (rank 0's device time, ms)."""
    if not ms_list:
        return None
    xs = sorted(ms_list)
    n = len(xs)
    med = xs[n // 2] if n % 2 else 0.5 * (xs[n // 2 - 1] + xs[n // 2])
    return {"min": xs[0], "median": med, "max": xs[-1], "n": n}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return None
        self.out.flush()
        self.out.seek(0)
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx, power = float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            if power < 200:  # idle sample, before or after the kernels
                continue
            sms.append(sm)
            maxes.append(mx)
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.out.name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


def cpu_baseline(w, q, k, v, target_s: float = 10.0):
    """Time the fp64 oracle on the host cores over a bounded sample of query rows."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(w.seed + 99)
    total = w.B * w.H * w.N
    perm = rng.permutation(total) if total <= 50_000_000 else rng.integers(0, total, size=1_000_000)
    n0 = min(256, total)
    t0 = time.perf_counter()
    oracle_rows(w, q, k, v, perm[:n0])
    t_cal = max(time.perf_counter() - t0, 1e-3)
    n = int(min(len(perm), max(n0, n0 * target_s / t_cal)))
    rows = perm[:n]
    t0 = time.perf_counter()
    _, _, used = oracle_rows(w, q, k, v, rows, return_threads=True)
    dt = time.perf_counter() - t0
    return {"value": row_flops(w, rows) / dt / 1e12, "unit": "TFLOP/s", "cores": int(used), "kind": "oracle",
            "sample": f"{n} seeded query rows of {w.name} (of {total}), fp64 three-pass route, {dt:.1f} s"}


def run_softmax(args, rank, world, local_rank):
    """The standalone row softmax: one step = one fa_softmax_rows call over an
    M x N fp32 matrix (y and lse written).  value = algorithmic bytes (read x,
    write y and lse: 8 M N + 4 M) / time."""
    import numpy as np
    import torch

    import __graft_entry__

    M, N = args.rows, args.cols
    name = f"softmax-M{M}-N{N}-fp32"
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle

        rng = np.random.default_rng(2000)
        sample = max(1, min(M, int(os.environ.get("SOFTMAX_REF_ROWS", "256"))))
        x = rng.standard_normal((sample, N), dtype=np.float32)
        ms = []
        for _ in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            for i in range(sample):
                oracle.softmax_three_pass(x[i].astype(np.float64))
            ms.append((time.perf_counter() - t0) * 1e3)
        ms_step = statistics.mean(ms[args.warmup:])
        value = (8.0 * sample * N + 4.0 * sample) / (ms_step * 1e-3) / 1e9
        cpu = {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{sample} rows of {name} per step, fp64 three-pass route, one core"}
        print(json.dumps({"impl": "reference", "metric": SOFTMAX_METRIC, "value": value, "unit": "GB/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": {"workload": name, "rows_per_step": sample},
                          "cpu_baseline": cpu, "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                                                       "d2h_bytes_per_step": 0}}), flush=True)
        return
    if local_rank == 0:
        __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import online_softmax_04_gb300 as fa

    rng = np.random.default_rng(2000 + rank)
    hx = torch.from_numpy(rng.standard_normal((M, N), dtype=np.float32))
    x = hx.to(dev)
    y = torch.empty_like(x)
    lse = torch.empty(M, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    algo_bytes = 8.0 * M * N + 4.0 * M
    flush_l2 = algo_bytes < 2 * L2_BYTES
    flusher = L2Flush(torch, dev) if flush_l2 else None

    def step():
        fa.fa_softmax_rows(x, y, lse, M, N, stream)

    def timed(fn, n):
        torch.cuda.synchronize()
        if flush_l2:
            ms = 0.0
            for _ in range(n):
                flusher()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                ms += e0.elapsed_time(e1)
            return ms
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    fa.fa_clear_device_status()
    for _ in range(args.warmup):
        step()
    with ClockSampler(local_rank) as clk:
        ms_total = timed(step, args.steps)
    ms_step = ms_total / args.steps
    value = algo_bytes / (ms_step * 1e-3) / 1e9
    hxp = hx.pin_memory()
    hy = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    hl = torch.empty(M, dtype=torch.float32, pin_memory=True)

    def e2e_step():
        x.copy_(hxp, non_blocking=True)
        step()
        hy.copy_(y, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    ms_e2e = timed(e2e_step, args.steps) / args.steps
    if fa.fa_get_device_status() != 0:
        raise SystemExit("a softmax kernel gave up on a barrier")
    if rank != 0:
        return
    peak, src = measured_peak("hbm_gbs")
    if N % 4 == 0 and N <= 2048:
        kernel = "softmax_rows_warp"
    elif N % 4 == 0 and 4 * N <= 100 * 1024:
        kernel = "softmax_rows_smem"
    else:
        kernel = "softmax_rows_stream"
    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        sample = min(M, 512)
        xs = hx[:sample].numpy().astype(np.float64)
        t0 = time.perf_counter()
        for i in range(sample):
            oracle.softmax_three_pass(xs[i])
        dt = time.perf_counter() - t0
        cpu = {"value": (8.0 * sample * N + 4.0 * sample) / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{sample} rows of {name}, fp64 three-pass route, one core, {dt:.2f} s"}
    line = {
        "metric": SOFTMAX_METRIC, "value": value * world, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "M": M, "N": N, "bytes_per_step_per_gpu": algo_bytes,
                   "l2": ("L2 flushed (512 MB write, then 256 MB read) before each individually timed step" if flush_l2 else
                          "x and y larger than L2, back-to-back steps, no flush"),
                   "entry_point": "fa_softmax_rows", "path": kernel},
        "roofline": {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "traffic": recorded_traffic(name, kernel), "peak_source": src, "kernel": kernel},
        "cpu_baseline": cpu,
        "e2e": {"value": algo_bytes * world / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": 4 * M * N, "d2h_bytes_per_step": 4 * M * N + 4 * M, "ms_per_step": ms_e2e},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


BWD_METRIC = "attention backward TFLOP/s (bf16, 1 GB300; 5 products per tile pair counted) and % of dense BF16 peak"


def run_backward(args, w, rank, world, local_rank):
    """One step = one fa_bwd call (D, dQ, dK, dV) on the workload; FLOPs =
    2.5 x the forward's (five N x N x d products instead of two)."""
    import numpy as np
    import torch

    import __graft_entry__

    if w.masked:
        raise SystemExit("the backward pass takes full or causal attention")
    flops = 2.5 * workload_flops(w)
    if args.impl == "reference":
        if rank != 0:
            return
        from online_softmax_04_gb300 import workloads as wl
        import oracle

        q, k, v = wl.make_inputs(w)
        rng = np.random.default_rng(w.seed + 9)
        dout = torch.from_numpy(rng.standard_normal(q.shape, dtype=np.float32)).to(torch.bfloat16)
        o = torch.zeros(q.shape, dtype=torch.float32)   # D_i = 0: the oracle's cost does not depend on O
        lse = torch.zeros(q.shape[:3], dtype=torch.float32)
        total = w.B * w.H * w.N
        n = 64
        secs, fl = 0.0, 0.0
        for step in range(args.warmup + args.steps):
            rows = rng.integers(0, total, n)
            t0 = time.perf_counter()
            oracle.attention_backward(q, k, v, o, dout, lse, w.causal, w.scale, q_rows=rows, k_rows=rows)
            dt = time.perf_counter() - t0
            if step >= args.warmup:
                secs += dt
                fl += 2.5 * row_flops(w, rows)   # the per-row share of the same 10 d per visible pair
        value = fl / secs / 1e12
        print(json.dumps({"impl": "reference", "metric": BWD_METRIC, "value": value, "unit": "TFLOP/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": {"workload": w.name, "op": "backward"},
                          "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count() or 1,
                                           "kind": "oracle", "sample": f"{n} query rows and {n} key rows per step"},
                          "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    if local_rank == 0:
        __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import online_softmax_04_gb300 as fa
    from online_softmax_04_gb300 import workloads as wl

    wr = rank_workload(w, rank)
    q, k, v = wl.make_inputs(wr)
    rng = np.random.default_rng(wr.seed + 9)
    hdo = torch.from_numpy(rng.standard_normal(q.shape, dtype=np.float32)).to(torch.bfloat16)
    dq_, dk_, dv_, ddo = q.to(dev), k.to(dev), v.to(dev), hdo.to(dev)
    o, lse = fa.attention(dq_, dk_, dv_, causal=w.causal)     # the forward the backward belongs to
    gq, gk, gv = torch.empty_like(dq_), torch.empty_like(dk_), torch.empty_like(dv_)
    ws_bytes = fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fa_bwd(dq_, dk_, dv_, o, ddo, lse, gq, gk, gv, w.B, w.H, w.N, w.d, w.causal, w.scale, ws, ws_bytes, stream)

    fa.fa_clear_device_status()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    io = 8 * q.numel() * 2
    flush = L2Flush(torch, dev) if io < 2 * L2_BYTES else None

    def timed(fn, n):
        torch.cuda.synchronize()
        if flush is not None:
            ms = 0.0
            for _ in range(n):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                ms += e0.elapsed_time(e1)
            return ms
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    with ClockSampler(local_rank) as clk:
        ms_total = timed(step, args.steps)
    ms_step = ms_total / args.steps
    value = flops / (ms_step * 1e-3) / 1e12
    host = [t.pin_memory() for t in (q, k, v, o.cpu(), hdo, lse.cpu())]
    outs_h = [torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(3)]
    devs = [dq_, dk_, dv_, o, ddo, lse]

    def e2e_step():
        for hd, dd in zip(host, devs):
            dd.copy_(hd, non_blocking=True)
        step()
        for hd, dd in zip(outs_h, (gq, gk, gv)):
            hd.copy_(dd, non_blocking=True)

    for _ in range(3):
        e2e_step()
    ms_e2e = timed(e2e_step, args.steps) / args.steps
    if fa.fa_get_device_status() != 0:
        raise SystemExit("a backward kernel gave up on a barrier")
    if rank != 0:
        return
    peak, src = measured_peak()
    line = {
        "metric": BWD_METRIC, "value": value * world, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "op": "backward", "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "flops_per_step_per_gpu": flops, "entry_point": "fa_bwd",
                   "l2": "L2 flushed before each step" if flush is not None else "inputs larger than L2"},
        "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s", "frac": value / peak,
                     "traffic": None, "peak_source": src,
                     "kernel": "fa_bwd_delta + fa_bwd_dq_sm103 + fa_bwd_dkdv_sm103"},
        "cpu_baseline": None,
        "e2e": {"value": flops * world / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host),
                "d2h_bytes_per_step": 3 * q.numel() * 2, "ms_per_step": ms_e2e},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_reference(args, w, rank, world):
    """The oracle as the reference arm: K timed steps, each a bounded row sample."""
    if rank != 0:
        return
    from online_softmax_04_gb300 import workloads as wl

    q, k, v = wl.make_inputs(w)
    per_step_s = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    import numpy as np

    import oracle

    rng = np.random.default_rng(w.seed + 5)
    total = w.B * w.H * w.N
    t0 = time.perf_counter()
    oracle_rows(w, q, k, v, rng.integers(0, total, 128))
    t_cal = max(time.perf_counter() - t0, 1e-3)
    n = int(max(128, 128 * per_step_s / t_cal))
    flops, secs, used = 0.0, 0.0, 1
    for step in range(args.warmup + args.steps):
        rows = rng.integers(0, total, n)
        t0 = time.perf_counter()
        _, _, used = oracle_rows(w, q, k, v, rows, return_threads=True)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            flops += row_flops(w, rows)
            secs += dt
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, world),
        "entry_point": "oracle.attention_three_pass (fp64, host cores)",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": int(used), "kind": "oracle",
                         "sample": f"{n} random query rows per step of {w.name}, fp64 three-pass route"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--heads", type=int, default=None, help="override H (smaller profiling captures)")
    ap.add_argument("--splitkv", type=int, default=-1,
                    help="use the split-KV entry point with this many splits (0 = automatic; default: off)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=["attention", "softmax", "backward"], default="attention",
                    help="attention (the headline forward), the standalone row softmax, or the attention backward")
    ap.add_argument("--rows", type=int, default=4096, help="--op softmax: M")
    ap.add_argument("--cols", type=int, default=4096, help="--op softmax: N")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.op == "softmax":
        run_softmax(args, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
                    int(os.environ.get("LOCAL_RANK", "0")))
        return

    from online_softmax_04_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload or wl.HEADLINE]
    if args.heads:
        w = w.with_(H=args.heads, name=f"{w.name}@H{args.heads}")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.op == "backward":
        run_backward(args, w, rank, world, local_rank)
        return
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import numpy as np
    import torch

    import __graft_entry__

    if local_rank == 0:
        __graft_entry__.build()
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
        dist.barrier()
        if local_rank != 0:
            __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import online_softmax_04_gb300 as fa

    wr = rank_workload(w, rank)
    q, k, v = wl.make_inputs(wr)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(dq)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    n_splits = -1
    if args.splitkv >= 0:
        n_splits = args.splitkv or fa.fa_splitkv_auto_splits(w.B, w.H, w.N, w.d, w.causal)
        ws_bytes = fa.fa_splitkv_workspace_bytes(w.B, w.H, w.N, w.d, n_splits)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    doc_dev = None
    if w.masked:
        docs = wl.make_doc_ids(w)
        doc_dev = torch.from_numpy(docs).to(dev) if docs is not None else None

    def run_fwd():
        if w.masked:
            fa.fa_fwd_masked(dq, dk, dv, o, lse, w.B, w.H, w.N, w.d, w.window_left, w.window_right, doc_dev,
                             w.scale, stream)
        elif n_splits > 0:
            fa.fa_fwd_splitkv(dq, dk, dv, o, lse, w.B, w.H, w.N, w.d, w.causal, w.scale, n_splits, workspace,
                              ws_bytes, stream)
        else:
            fa.fa_fwd(dq, dk, dv, o, lse, w.B, w.H, w.N, w.d, w.causal, w.scale, stream)

    launches_per_step = 2 if n_splits > 0 else 1

    def step():
        run_fwd()

    fa.fa_clear_device_status()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # Inputs (Q, K, V) well above L2 make back-to-back steps honest; smaller
    # workloads get L2 flushed (a 512 MB write, then a 256 MB read) before each individually timed step.
    flush_l2 = l2_policy(w)[0]
    flusher = L2Flush(torch, dev) if flush_l2 else None

    per_step = []  # this rank's device time of each timed step (ms)

    def timed(fn, n, record_steps=False):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        if flush_l2:
            ms = 0.0
            for _ in range(n):
                flusher()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                ms += e0.elapsed_time(e1)
                if record_steps:
                    per_step.append(e0.elapsed_time(e1))
        else:
            # an event between consecutive steps gives each step's time as well
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
            ev[0].record(stream)
            for i in range(n):
                fn()
                ev[i + 1].record(stream)
            torch.cuda.synchronize()
            ms = ev[0].elapsed_time(ev[n])
            if record_steps:
                per_step.extend(ev[i].elapsed_time(ev[i + 1]) for i in range(n))
        ms = max_over_ranks(ms, dist, dev)
        if dist is not None:
            dist.barrier()
        return ms

    with ClockSampler(local_rank) as clk:
        ms_total = timed(step, args.steps, record_steps=True)
    clocks = clk.summary()
    ms_step = ms_total / args.steps
    flops = workload_flops(w)
    value = whole_job_tflops(world, flops, args.steps, ms_total)

    # end to end: pinned host buffers, copies inside the timed region
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)

    # the plain forward runs end to end through fa_fwd_host: the library copies
    # chunks of heads in, computes and copies them back on overlapping streams;
    # masked and split-KV workloads copy around their device entry point
    host_entry = n_splits < 0 and not w.masked
    if host_entry:
        hpc = 0  # the library's default chunk: ceil(B*H / 8) heads
        ws_host = torch.empty(fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.N, w.d, hpc), dtype=torch.uint8,
                              device=dev)

    def e2e_step():
        if host_entry:
            fa.fa_fwd_host(hq, hk, hv, ho, hl, w.B, w.H, w.N, w.d, w.causal, w.scale, hpc, ws_host,
                           ws_host.numel(), stream)
            return
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        run_fwd()
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    ms_e2e = timed(e2e_step, args.steps)
    e2e_value = whole_job_tflops(world, flops, args.steps, ms_e2e)
    h2d = 3 * q.numel() * q.element_size()
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()

    status = fa.fa_get_device_status()
    if status != 0:
        raise SystemExit(f"device status word {status:#x}: a kernel gave up on a barrier")

    if rank == 0:
        peak, peak_src = measured_peak()
        achieved = flops / (ms_step * 1e-3) / 1e12
        # which forward kernel ran: masked, split-KV, or fa_fwd's choice (one query tile
        # per CTA, CTA pairs at d = 128, or two tiles per CTA at d = 64)
        fwd_kind = (fa.FA_KERNEL_FWD_MASKED if w.masked else fa.FA_KERNEL_FWD_SPLITKV if n_splits > 0
                    else fa.fa_fwd_kernel_for(w.B, w.H, w.N, w.d, w.causal))
        kernel_label = (KERNEL_NAME + " (CTA pairs, cta_group::2)" if fwd_kind == fa.FA_KERNEL_FWD_PAIR else
                        "fa_fwd2_sm103 (two query tiles per CTA)" if fwd_kind == fa.FA_KERNEL_FWD_TWO else
                        KERNEL_NAME + (" + merge" if n_splits > 0 else ""))
        # the burst peak is the denominator (the kernel is timed on its own); the sustained,
        # power-capped figure is given beside it: over long runs the power cap lowers the clock
        peak_sus, _ = measured_peak("bf16_tflops_sustained")
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": recorded_traffic(w.name) if n_splits < 0 else None,
                    "peak_source": peak_src, "peak_sustained": peak_sus, "frac_of_sustained": achieved / peak_sus,
                    "kernel": kernel_label,
                    # the HBM side of the same launch: algorithmic bytes (Q, K, V read, O and LSE
                    # written once) over the step time, against the measured copy bandwidth
                    "hbm": hbm_side(w, ms_step),
                    # registers, shared memory, CTAs per SM and TMEM columns, from the runtime
                    "resources": fa.fa_kernel_resources(w.d, fwd_kind)}
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(w, q, k, v)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": bench_config(w, world),
            "entry_point": ("fa_fwd_masked" if w.masked else "fa_fwd") if n_splits < 0
            else f"fa_fwd_splitkv (n_splits={n_splits})",
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": ms_e2e / args.steps,
                    "entry_point": ("fa_fwd_host (pinned host tensors, heads streamed in chunks of "
                                    f"{-(-w.B * w.H // 8)})") if host_entry else
                    "host->device copies, the device entry point, device->host copies on one stream"},
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clocks,
            "step_ms": step_stats(per_step),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
