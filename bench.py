#!/usr/bin/env python3
"""Benchmark of the NF4 decode projection on GB300.

Workload (one "step"): one nf4_gemv_residual call of the Qwen2.5-3B-shaped
down projection, NF4 W 2048 x 11008 (N(0, 0.02) before quantization, 64-weight
blocks, fp32 scales), x bf16 = silu(z1) * z2, fp32 residual, fp32 out.
Metric: effective weight GB/s = (code + scale bytes) / time per call, and the
same time as microseconds per call.

Timing: the weights rotate over R device copies whose total is more than three
times the L2, so every call streams its weights from HBM; calls are replayed
from CUDA graphs on one stream and timed with CUDA events on that stream,
after W warm-up calls, bracketed by a barrier and a device synchronize.
``e2e`` repeats the measurement through the public Python API with the step's
activation and residual copied from pinned host memory and its output copied
back inside the timed region (weights stay resident, as in decode), issued
from Python as a user writes it, with the step recorded as a CUDA graph and
replayed reported beside it.

``cpu_baseline`` times the oracle on the host: one thread, and one spawned
process per core over disjoint row ranges (the all-core figure).
``--impl reference`` times the CPU oracle instead (the reference arm of this
repository; it is deliberately slow, plain C, single-threaded).

Other workloads (SwiGLU, interleaved gate/up SwiGLU, lm_head + argmax, 14B N=1,
14B chunk, fused 3B q/k/v, embedding-row gather of a 4096-token prompt,
RMSNorm of a decode step and of a prefill chunk) are reported compactly under
"workloads" with the same method and fewer calls; ``--describe`` prints their
launch configurations.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NF4 GEMV effective weight GB/s (N=1, 3B down_proj 2048x11008 + residual)"
UNIT = "GB/s"
MAIN = "down_residual"
# reported beside the main workload, in this order
WORKLOADS = ("swiglu", "glu3b", "lm_head_argmax", "gemv14b", "chunk14b", "qkv3b", "embed_prefill", "rmsnorm3b",
             "rmsnorm_chunk14b")
WORKLOAD_NAME = "3B down_proj 2048x11008 NF4 (block 64, fp32 scales) + fp32 residual, x bf16, N=1"


# ------------------------------------------------------------------ helpers

def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its // and /* */ comments (string and
    character literals kept as they are), trailing blanks and blank lines, so
    that editing a comment does not count as a change of the kernels."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    # lines left empty by a removed comment, and trailing blanks, do not count
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def kernel_source_hash() -> str:
    """First 16 hex digits of sha256 over the kernel sources (file names and
    their code, comments removed)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nf4_weight_quantized_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def bytes_of(kind: str, M: int, K: int, N: int = 1, M_kv: int = 0) -> dict:
    """Algorithmic bytes per call: weight (codes + scales) and total."""
    if kind == "rmsnorm":  # M rows of K: read fp32 rows and the bf16 gain, write bf16 rows
        return {"weight": K * 2, "total": M * K * 4 + K * 2 + M * K * 2}
    if kind == "embed":  # N gathered rows of an M-row table: read N rows, write N bf16 rows
        w = N * (K // 2 + (K // 64) * 4)
        return {"weight": w, "total": w + N * 8 + N * K * 2, "table": M * K // 2 + M * (K // 64) * 4}
    if kind == "qkv":
        M = M + 2 * M_kv
    w = M * K // 2 + M * (K // 64) * 4
    if kind == "qkv":
        tot = w + K * 2 + M * 4 + M * 4  # + biases + outputs
    elif kind == "residual":
        tot = w + K * 2 + M * 4 + M * 4
    elif kind in ("swiglu", "glu"):  # glu: M outputs of a 2 M-row matrix
        w *= 2
        tot = w + K * 2 + M * 2
    elif kind == "argmax":
        tot = w + K * 2 + M * 4 + 8
    elif kind == "chunk":
        tot = w + N * K * 2 + N * M * 4
    else:
        tot = w + K * 2 + M * 4
    return {"weight": w, "total": tot}


def describe(nf4, w) -> str:
    """The library's description of the launch a workload makes."""
    if w.kind == "embed":
        return (f"nf4_dequant_rows: {w.N} rows of a {w.M}x{w.K} NF4 table, bf16 out, one thread per 32 weights, "
                "256-thread blocks")
    if w.kind == "rmsnorm":
        return f"nf4_rmsnorm: {w.M} row(s) of {w.K}, one block per row, bf16 out"
    rows = 2 * w.M if w.kind == "glu" else w.M + 2 * w.M_kv
    return nf4.nf4_describe_launch(w.kind, rows, w.K, w.N)


def build_calls(name: str, torch, nf4, synth, device, copies=None):
    """Inputs for one workload, quantized on the device, with enough rotating
    weight copies to exceed 3x L2 (or `copies`).  Returns (call(i), n_copies,
    bytes, tensors)."""
    w = synth.WORKLOADS[name]
    M, K = w.M, w.K
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 128 << 20)
    b = bytes_of(w.kind, M, K, w.N, w.M_kv)
    fixed_copies = copies
    copies = copies or max(2, int(np.ceil(3 * l2 / b.get("table", b["weight"]))))
    d = synth.workload_inputs(w)

    def quant(Wnp):
        Wt = torch.from_numpy(Wnp).to(device)
        q = nf4.nf4_quantize(Wt)
        del Wt
        return q

    def replicate(q):
        out = [q]
        for _ in range(copies - 1):
            out.append(nf4.NF4Weight(q.codes.clone(), q.scales.clone()))
        return out

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)

    if w.kind == "rmsnorm":  # no weights: inputs are tiny and stay in L2, as in a decode step
        copies = 1
        x = torch.from_numpy(d["x"]).to(device)
        g = bf16(d["w"])
        out = torch.empty((M, K), dtype=torch.bfloat16, device=device)
        call = lambda i, s: nf4.nf4_rmsnorm(x, g, 1e-6, out, stream=s)
        return call, copies, b, {"x": x, "w": g, "out": out}
    if w.kind == "residual":
        Ws = replicate(quant(d["W"]))
        x = bf16(d["x"])
        r = torch.from_numpy(d["r"]).to(device)
        y = torch.empty(M, device=device)
        call = lambda i, s: nf4.nf4_gemv_residual(Ws[i % copies], x, r, y, stream=s)
        ctx = {"W": Ws, "x": x, "r": r, "y": y}
    elif w.kind == "swiglu":
        copies = fixed_copies or max(2, int(np.ceil(3 * l2 / b["weight"])))
        Wg = replicate(quant(d["W"]))
        Wu = replicate(quant(d["Wu"]))
        x = bf16(d["x"])
        out = torch.empty(M, dtype=torch.bfloat16, device=device)
        call = lambda i, s: nf4.nf4_gemv_swiglu(Wg[i % copies], Wu[i % copies], x, out, stream=s)
        ctx = {"Wg": Wg, "Wu": Wu, "x": x, "out": out}
    elif w.kind == "glu":
        Ws = replicate(quant(d["W"]))
        x = bf16(d["x"])
        out = torch.empty(M, dtype=torch.bfloat16, device=device)
        call = lambda i, s: nf4.nf4_gemv_glu_interleaved(Ws[i % copies], x, out, stream=s)
        ctx = {"W": Ws, "x": x, "out": out}
    elif w.kind == "argmax":
        Ws = replicate(quant(d["W"]))
        x = bf16(d["x"])
        logits = torch.empty(M, device=device)
        index = torch.empty(1, dtype=torch.int64, device=device)
        ws = nf4.new_workspace(M, K, 1, device)
        call = lambda i, s: nf4.nf4_gemv_argmax(Ws[i % copies], x, logits, index, ws, stream=s)
        ctx = {"W": Ws, "x": x, "logits": logits, "index": index}
    elif w.kind == "embed":
        Es = replicate(quant(d["W"]))
        ids = torch.from_numpy(d["ids"]).to(device)
        out = torch.empty((w.N, K), dtype=torch.bfloat16, device=device)
        call = lambda i, s: nf4.nf4_dequant_rows(Es[i % copies], ids, out, stream=s)
        ctx = {"E": Es, "ids": ids, "out": out}
    elif w.kind == "qkv":
        Wq, Wk, Wv = replicate(quant(d["W"])), replicate(quant(d["Wk"])), replicate(quant(d["Wv"]))
        x = bf16(d["x"])
        bq, bk, bv = (torch.from_numpy(d[k]).to(device) for k in ("bq", "bk", "bv"))
        out = torch.empty(M + 2 * w.M_kv, device=device)
        qo, ko, vo = out[:M], out[M:M + w.M_kv], out[M + w.M_kv:]
        call = lambda i, s: nf4.nf4_gemv_qkv(Wq[i % copies], Wk[i % copies], Wv[i % copies], x, bq, bk, bv,
                                             qo, ko, vo, stream=s)
        ctx = {"W": (Wq, Wk, Wv), "x": x, "b": (bq, bk, bv), "out": out}
    elif w.kind == "chunk":
        Ws = replicate(quant(d["W"]))
        X = bf16(d["X"])
        Y = torch.empty((w.N, M), device=device)
        ws = nf4.new_workspace(M, K, w.N, device)
        call = lambda i, s: nf4.nf4_gemm_chunk(Ws[i % copies], X, Y, ws, stream=s)
        ctx = {"W": Ws, "X": X, "Y": Y}
    else:
        Ws = replicate(quant(d["W"]))
        x = bf16(d["x"]) if w.x_dtype == "bf16" else torch.from_numpy(d["x"]).to(device)
        y = torch.empty(M, device=device)
        call = lambda i, s: nf4.nf4_gemv(Ws[i % copies], x, y, stream=s)
        ctx = {"W": Ws, "x": x, "y": y}
    return call, copies, b, ctx


def capture(torch, call, n: int, start: int, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                call(start + i, stream)
    return g


def time_calls(torch, call, copies: int, steps: int, warmup: int, stream, dist=None, clock_window_s=0.0,
               sampler=None):
    """Time exactly `steps` calls replayed from CUDA graphs; returns seconds."""
    chunk = min(steps, max(copies, 500))
    chunk = (chunk // copies) * copies if chunk >= copies else chunk
    full, rem = divmod(steps, chunk)
    g = capture(torch, call, chunk, 0, stream)
    g_rem = capture(torch, call, rem, 0, stream) if rem else None
    with torch.cuda.stream(stream):
        for i in range(warmup):
            call(i, stream)
        g.replay()
    stream.synchronize()
    if sampler is not None:
        sampler.start()
    if clock_window_s > 0:
        t0 = time.time()
        while time.time() - t0 < clock_window_s:
            with torch.cuda.stream(stream):
                g.replay()
            stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        # an untimed lead-in replay keeps the GPU busy while the timed replays
        # are queued behind it, so the host's graph-launch latency does not
        # land inside the timed region (it would add ~10 us to a 20-call one)
        g.replay()
        e0.record(stream)
        for _ in range(full):
            g.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop() if sampler is not None else None
    return e0.elapsed_time(e1) / 1e3, clocks


def time_windows(torch, call, copies: int, stream, windows: int = 5, calls: int = 500):
    """Per-call microseconds of `windows` separately timed replays of one graph
    of `calls` calls (after the main timing, outside `value`): the spread
    between windows."""
    n = max(copies, (calls // copies) * copies)
    g = capture(torch, call, n, 0, stream)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    out = []
    for _ in range(windows):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3 / n)
    srt = sorted(out)
    return {"calls_per_window": n, "us_per_call": [round(v, 4) for v in out], "median": round(srt[len(srt) // 2], 4),
            "min": round(srt[0], 4), "max": round(srt[-1], 4)}


# ------------------------------------------------------------- CPU baseline

def _oracle_rows_worker(task):
    """One host process of the all-core oracle timing: the oracle as it stands
    (single-threaded C) on its own contiguous range of the workload's rows,
    repeated until the deadline; returns (calls, seconds)."""
    codes, scales, x, r, r0, r1, target_s = task
    import oracle

    rows = np.arange(r0, r1)
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.gemv_residual(codes, scales, x, r, rows=rows)
        n += 1
        if time.perf_counter() - t0 >= target_s:
            break
    return n, time.perf_counter() - t0


def cpu_oracle_run(target_s: float):
    """The oracle on the host's cores, on the main workload.

    Single thread: full down_proj + residual calls repeated for target_s.
    All cores: one spawned process per core, each running the same oracle on
    its own contiguous share of the rows for target_s; a full call takes as
    long as the slowest share, so the value is weight bytes x calls of the
    slowest process / its time."""
    import multiprocessing as mp

    import oracle
    from nf4_weight_quantized_gb300 import synth

    w = synth.WORKLOADS[MAIN]
    d = synth.workload_inputs(w)
    codes, scales = oracle.quantize(d["W"])
    b = bytes_of(w.kind, w.M, w.K)
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.gemv_residual(codes, scales, d["x"], d["r"])
        n += 1
        if time.perf_counter() - t0 >= target_s:
            break
    dt = time.perf_counter() - t0
    single = {"value": b["weight"] * n / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
              "sample": f"full down_proj 2048x11008 + residual, {n} call(s), {dt:.1f} s, 1 thread",
              "us_per_call": dt / n * 1e6}
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    if cores < 2:
        return single
    bounds = [w.M * i // cores for i in range(cores + 1)]
    tasks = [(codes, scales, d["x"], d["r"], bounds[i], bounds[i + 1], target_s) for i in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_rows_worker, tasks)
    per_call = max(t / c for c, t in res)
    return {"value": b["weight"] / per_call / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"full down_proj 2048x11008 + residual, rows split over {cores} spawned processes "
                       f"(one per core), {min(c for c, _ in res)}+ call(s) each in {target_s:.0f} s"),
            "us_per_call": per_call * 1e6, "single_thread": single}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, timed on the host (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    from nf4_weight_quantized_gb300 import synth

    w = synth.WORKLOADS[MAIN]
    d = synth.workload_inputs(w)
    codes, scales = oracle.quantize(d["W"])
    # one step: a bounded sample of the workload, 8 rows (rotating) of the
    # 2048 with the full K, so that the default run ends within minutes
    rows_per_step = 8
    row_bytes = w.K // 2 + (w.K // 64) * 4

    def step(i):
        r0 = (i * rows_per_step) % w.M
        rows = np.arange(r0, r0 + rows_per_step) % w.M
        oracle.gemv_residual(codes, scales, d["x"], d["r"], rows=rows)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = row_bytes * rows_per_step * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD_NAME, "parallelism": "single",
                                        "sample": f"{rows_per_step} rows per step (rotating), full K",
                                        "rows_per_step": rows_per_step, "l2": "host"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{rows_per_step} rows x K=11008 per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm

def reduce_max(dist, v: float, device=None) -> float:
    """Max over ranks of a per-rank value (the slowest replica's time); the
    value itself without a process group.  NCCL needs a device tensor, gloo a
    CPU one."""
    if dist is None:
        return v
    import torch

    t = torch.tensor([v], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(world: int, bytes_per_call: int, calls: int, max_secs: float) -> float:
    """Whole-job throughput in GB/s: every replica moved `bytes_per_call` per
    call, timed by the slowest replica."""
    return world * bytes_per_call * calls / max_secs / 1e9


def run_gpu(args, rank, world, dist):
    import torch

    from nf4_weight_quantized_gb300 import nf4, synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.Stream(device)
    peaks = measured_peaks()

    call, copies, b, ctx = build_calls(MAIN, torch, nf4, synth, device)
    sampler = ClockSampler(local)
    secs, clocks = time_calls(torch, call, copies, args.steps, args.warmup, stream, dist,
                              clock_window_s=args.clock_window, sampler=sampler)
    secs = reduce_max(dist, secs, device)
    windows = time_windows(torch, call, copies, stream)
    per_call = secs / args.steps
    value = replica_value(world, b["weight"], args.steps, secs)
    achieved = b["total"] / per_call / 1e9

    # e2e through the public API with host buffers
    w = synth.WORKLOADS[MAIN]
    # the step's inputs (x, then the residual) in one pinned host buffer and one
    # device buffer, so each step makes one host-to-device copy
    xb, rb = ctx["x"].numel() * 2, ctx["r"].numel() * 4
    in_host = torch.empty(xb + rb, dtype=torch.uint8).pin_memory()
    in_host[:xb].view(torch.bfloat16).copy_(ctx["x"].cpu())
    in_host[xb:].view(torch.float32).copy_(ctx["r"].cpu())
    in_dev = torch.empty(xb + rb, dtype=torch.uint8, device=device)
    x_dev, r_dev = in_dev[:xb].view(torch.bfloat16), in_dev[xb:].view(torch.float32)
    y_host = torch.empty(w.M, dtype=torch.float32).pin_memory()
    y_dev = torch.empty_like(ctx["y"])
    n_e2e = min(args.steps, args.e2e_steps)
    Ws = ctx["W"]
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            in_dev.copy_(in_host, non_blocking=True)
            nf4.nf4_gemv_residual(Ws[i % copies], x_dev, r_dev, y_dev, stream=stream)
            y_host.copy_(y_dev, non_blocking=True)
    stream.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(n_e2e):
            in_dev.copy_(in_host, non_blocking=True)
            nf4.nf4_gemv_residual(Ws[i % copies], x_dev, r_dev, y_dev, stream=stream)
            y_host.copy_(y_dev, non_blocking=True)
        e1.record(stream)
    stream.synchronize()
    e2e_secs = e0.elapsed_time(e1) / 1e3
    e2e_secs = reduce_max(dist, e2e_secs, device)
    # headline: the step as a user writes it with the public API (copy in,
    # call, copy out, from Python); the graph-replayed form is kept beside it
    e2e = {"value": replica_value(world, b["weight"], n_e2e, e2e_secs), "unit": UNIT,
           "h2d_bytes_per_step": in_host.numel(), "d2h_bytes_per_step": y_host.numel() * 4, "steps": n_e2e,
           "us_per_step": e2e_secs / n_e2e * 1e6,
           "form": "1 pinned H2D copy of x and the residual, nf4_gemv_residual, 1 D2H copy of y, issued from Python"}
    # the same step recorded once per weight copy as a CUDA graph (host -> device
    # copy, the call, device -> host copy) and replayed: how a decode loop
    # issues it, without the per-call Python work
    graphs = []
    for i in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            in_dev.copy_(in_host, non_blocking=True)
            nf4.nf4_gemv_residual(Ws[i], x_dev, r_dev, y_dev)
            y_host.copy_(y_dev, non_blocking=True)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % copies].replay()
    stream.synchronize()
    if dist is not None:
        dist.barrier()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(n_e2e):
            graphs[i % copies].replay()
        e1.record(stream)
    stream.synchronize()
    g_secs = reduce_max(dist, e0.elapsed_time(e1) / 1e3, device)
    e2e["graph"] = {"value": replica_value(world, b["weight"], n_e2e, g_secs), "unit": UNIT,
                    "us_per_step": g_secs / n_e2e * 1e6, "steps": n_e2e,
                    "form": "the same step recorded as a CUDA graph per weight copy, replayed"}
    del graphs
    del ctx, Ws
    torch.cuda.empty_cache()

    # other workloads, compact (us per call, algorithmic GB/s, fraction of the
    # measured HBM peak) so the whole line stays short; their launch
    # configurations are printed by `python bench.py --describe`
    workloads = {}
    if args.all_workloads:
        for name in WORKLOADS:
            try:
                c2, cp2, b2, ctx2 = build_calls(name, torch, nf4, synth, device)
                n2 = args.workload_steps
                s2, _ = time_calls(torch, c2, cp2, n2, args.warmup, stream, dist)
                pc = s2 / n2
                workloads[name] = {"us": round(pc * 1e6, 3), "gbs": round(b2["total"] / pc / 1e9, 1),
                                   "frac": round(b2["total"] / pc / 1e9 / peaks["hbm_gbs"], 4)}
                del ctx2, c2
                torch.cuda.empty_cache()
            except Exception as e:  # report, keep the main line
                workloads[name] = {"error": f"{type(e).__name__}: {e}"[:200]}

    if rank != 0:
        return
    cpu = cpu_oracle_run(args.cpu_seconds) if (world == 1 and args.cpu_seconds > 0) else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_call * 1e3, "us_per_call": per_call * 1e6,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME,
                   "l2": f"rotating {copies} weight copies ({copies * b['weight'] / 1e6:.0f} MB, >3x L2)",
                   "parallelism": "replicas" if world > 1 else "single",
                   "kernel": nf4.nf4_describe_launch("residual", 2048, 11008, 1)},
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "windows": windows,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic("down_residual"),
                     "peak_source": peaks["source"], "algorithmic_bytes_per_launch": b["total"]},
        "cpu_baseline": cpu,
    }
    if workloads:
        line["workloads"] = workloads
    print(json.dumps(line), flush=True)


def run_profile_target(name: str, calls: int):
    """Three (or `calls`) untimed calls of one workload, for ncu captures:
    `ncu ... python bench.py --ncu down_residual`."""
    import torch

    from nf4_weight_quantized_gb300 import nf4, synth

    device = torch.device("cuda", 0)
    call, _, b, ctx = build_calls(name, torch, nf4, synth, device, copies=1)
    s = torch.cuda.current_stream()
    for i in range(calls):
        call(0, s)
    torch.cuda.synchronize()
    w = synth.WORKLOADS[name]
    print(json.dumps({"workload": name, "calls": calls, "algorithmic_bytes": b["total"],
                      "config": describe(nf4, w)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="nf4", choices=["nf4", "reference"])
    ap.add_argument("--clock-window", type=float, default=1.0, help="seconds of replay sampled for clocks")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload-steps", type=int, default=2000)
    ap.add_argument("--no-workloads", dest="all_workloads", action="store_false")
    ap.add_argument("--ncu", default=None, help="run a few untimed calls of one workload (for ncu) and exit")
    ap.add_argument("--ncu-calls", type=int, default=3)
    ap.add_argument("--describe", action="store_true", help="print each workload's launch configuration and exit")
    args = ap.parse_args()
    if args.ncu:
        run_profile_target(args.ncu, args.ncu_calls)
        return
    if args.describe:
        from nf4_weight_quantized_gb300 import nf4, synth

        for name in (MAIN,) + WORKLOADS:
            w = synth.WORKLOADS[name]
            b = bytes_of(w.kind, w.M, w.K, w.N, w.M_kv)
            print(json.dumps({"workload": name, "description": w.description, "algorithmic_bytes": b["total"],
                              "config": describe(nf4, w)}))
        return
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1 and args.impl != "reference":
        import torch
        import torch.distributed as tdist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
