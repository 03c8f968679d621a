"""Benchmark of the 3.25-bit codebook-quantised decode matmul on GB300.

Workload (one "step"): the dense decode batch K=4096, N=12288 (a fused
gate+up projection) called once at each of M = 1, 2, 4, 8 token rows, every
call on a different copy of the packed weights (32 rotating copies, 657 MB,
more than 4x the 129 MB L2, so weight bytes come from HBM).  Activations,
a_scale and codebooks are seeded synthetic data of the pages' distributions.

Metric: effective weight GB/s = packed weight bytes (3KN/8 + KN/32 + 8N per
call) / time.  The timed region replays one CUDA graph of S back-to-back
calls per M, K/S rounds (K steps in all), timed with CUDA events on the
launching stream; the events around each graph replay give every kernel's
mean duration inside the same region.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain C implementation under
oracle/) on a bounded row sample of the same workload on the host cores.
Under torchrun every rank runs its own replica (the matmul needs no
exchange); value is the sum over ranks of the bytes processed divided by the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_codebook_quantized_gb300 import ops, synth  # noqa: E402

K_DIM, N_DIM = 4096, 12288
MS = (1, 2, 4, 8)
ROTATE = 32
FALLBACK_HBM_GBS = 6800.0
METRIC = "effective weight GB/s and % of GB300 HBM roofline per cbq_gemm call (M=1..64)"
WORKLOAD = "decode_4096x12288: cbq_gemm at M=1,2,4,8, K=4096, N=12288 (fused gate+up)"


KERNEL_NAMES = {ops.PATH_GEMV: "gemv_kernel", ops.PATH_MMA: "umma_kernel", ops.PATH_STREAMK: "sk_kernel"}


def kernel_of(M: int) -> str:
    """Kernel the library's automatic choice runs at M rows on the step's matrix."""
    return KERNEL_NAMES[ops.auto_path(M, N_DIM, K_DIM)]


def weight_bytes(N=N_DIM, K=K_DIM) -> int:
    return 3 * K * N // 8 + K * N // 32 + 8 * N


def call_bytes(M, N=N_DIM, K=K_DIM) -> int:
    """Algorithmic bytes of one call: packed weights, activations, a_scale, y."""
    return weight_bytes(N, K) + M * K + 4 * M + 4 * M * N


# ---------------------------------------------------------------- helpers --

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def reduce_max_sum(ws, t_max: float, units: float, device):
    """(max over ranks of t_max, sum over ranks of units)."""
    if ws == 1:
        return t_max, units
    t = torch.tensor([t_max], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for key in ("hbm_gbs", "hbm_GBps", "hbm"):
                if key in d:
                    v = d[key]
                    v = v.get("value", v) if isinstance(v, dict) else v
                    return float(v), "measured (MEASURED_PEAKS.json hbm_gbs)"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"cbq_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1].split()[0]))
                maxs.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxs) if maxs else None,
                "reasons": sorted(reasons), "samples": len(sms)}


# the sources each kernel is compiled from (its translation unit and the
# headers it includes)
KERNEL_SOURCES = {
    "gemv_kernel": ["cbq_gemv.cu", "cbq_device.cuh", "cbq_internal.h"],
    "umma_kernel": ["cbq_umma.cu", "cbq_device.cuh", "cbq_internal.h"],
    "sk_kernel": ["cbq_sk.cu", "cbq_device.cuh", "cbq_internal.h"],
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the kernel's code: its sources with // comments and blank lines
    removed, so a comment-only edit keeps the recorded counters."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_codebook_quantized_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        for line in open(os.path.join(csrc, f), encoding="utf-8"):
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary of this workload,
    or None when the summary is missing or the kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", "cbq_gemm_decode_4096x12288.md")
    if not os.path.exists(p):
        return None
    src, per_m = None, {}
    for line in open(p):
        if line.startswith(f"kernel_source_sha256[{kernel}]:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith(f"dram_bytes_per_launch[{kernel}]"):
            k, v = line.split(":", 1)
            per_m[k.split("M=")[1].rstrip("]").strip()] = float(v)
    if kernel not in KERNEL_SOURCES or src != kernel_source_hash(kernel) or not per_m:
        return None
    return per_m


# --------------------------------------------------------------- our arm --

def run_ours(args):
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(ws, "nccl")
    dev = torch.device("cuda", local)
    from bit_codebook_quantized_gb300 import build as _b
    if rank == 0 or ws == 1:
        _b.build()
    barrier(ws)
    _b.build()
    ops.lib()

    # ---- inputs, resident in HBM before the timed region --------------------
    pw = synth.gen_weights(N_DIM, K_DIM, seed=1)
    w0 = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, N_DIM, K_DIM, device=dev)
    copies = [w0] + [ops.PackedWeights(w0.codes.clone(), w0.scales.clone(), w0.codebooks.clone(),
                                       N_DIM, K_DIM) for _ in range(ROTATE - 1)]
    acts = {M: torch.from_numpy(synth.gen_activations(M, K_DIM, seed=10 + M)).to(dev) for M in MS}
    scs = {M: torch.from_numpy(synth.gen_a_scale(M, seed=20 + M, mode="uniform")).to(dev)
           for M in MS}
    ys = {M: torch.empty((M, N_DIM), dtype=torch.float32, device=dev) for M in MS}
    stream = torch.cuda.Stream(device=dev)

    call = [0]

    def step():
        for M in MS:
            w = copies[call[0] % ROTATE]
            call[0] += 1
            ops.gemm(acts[M], scs[M], w, out=ys[M], stream=stream)

    # ---- warm-up (untimed, eager) --------------------------------------------
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    stream.synchronize()
    if ops.device_status(stream) != ops.OK:
        raise RuntimeError("device status not ok after warm-up")

    # ---- one CUDA graph per M: S back-to-back calls on rotating weight copies --
    S = min(args.steps, 250)
    while args.steps % S:
        S -= 1
    reps = args.steps // S
    graphs = {}
    launches_before = ops.launch_count()
    for M in MS:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(S):
                w = copies[call[0] % ROTATE]
                call[0] += 1
                ops.gemm(acts[M], scs[M], w, out=ys[M], stream=stream)
        graphs[M] = g
    launches_per_step = (ops.launch_count() - launches_before) // S
    for M in MS:
        graphs[M].replay()
    stream.synchronize()

    # ---- timed region: K steps = reps x (S calls at each M), events between
    # the graph replays give every kernel's duration inside the same region
    ev = {M: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)] for M in MS}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            # untimed primer: keeps the GPU busy while the host enqueues the
            # timed replays, so the first one does not include host launch
            # latency (its weight copies are not the first timed graph's)
            graphs[MS[-1]].replay()
            t0.record(stream)
            for rep in range(reps):
                for M in MS:
                    ev[M][rep][0].record(stream)
                    graphs[M].replay()
                    ev[M][rep][1].record(stream)
            t1.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    elapsed_s = t0.elapsed_time(t1) / 1e3
    st = ops.device_status(stream)
    if st != ops.OK:
        raise RuntimeError(f"device status {st} after timed region")
    per_m_us = {M: 1e3 * sum(a.elapsed_time(b) for a, b in ev[M]) / (reps * S) for M in MS}
    kernel_timing = (f"CUDA events around each of the {reps} replays of every per-M graph of {S} "
                     f"back-to-back calls, inside the timed region")

    units = args.steps * len(MS) * weight_bytes()
    t_max, units_all = reduce_max_sum(ws, elapsed_s, units, dev)
    value = units_all / t_max / 1e9

    # ---- e2e through the public API with host buffers --------------------------
    e2e = run_e2e(dev, stream, copies, args)
    e2e["eager"] = run_e2e_eager(dev, stream, copies, steps=max(20, min(args.steps, 1000)))

    peak, peak_src = measured_peak()
    per_call = []
    for M in MS:
        us = per_m_us[M]
        per_call.append({"M": M, "kernel": kernel_of(M), "us": round(us, 3),
                         "weight_GBps": round(weight_bytes() / us / 1e3, 1),
                         "roofline_frac": round(call_bytes(M) / us / 1e3 / peak, 4),
                         "tokens_per_s": round(M / us * 1e6, 1)})
    # dominant kernel: the one with the largest share of the step's time
    fam = {}
    for M in MS:
        fam.setdefault(kernel_of(M), []).append(M)
    dom = max(fam, key=lambda k: sum(per_m_us[M] for M in fam[k]))
    dom_bytes = float(np.mean([call_bytes(M) for M in fam[dom]]))
    dom_us = float(np.mean([per_m_us[M] for M in fam[dom]]))
    traffic = profiled_traffic(dom)
    roof = {"bound": "hbm", "kernel": f"{dom} (M={','.join(map(str, fam[dom]))})",
            "achieved": round(dom_bytes / dom_us / 1e3, 1), "peak": peak, "unit": "GB/s",
            "frac": round(dom_bytes / dom_us / 1e3 / peak, 4),
            "traffic": (round(float(np.mean([traffic[str(M)] for M in fam[dom] if str(M) in traffic])))
                        if traffic and any(str(M) in traffic for M in fam[dom]) else None),
            "algorithmic_bytes_per_launch": int(dom_bytes), "peak_source": peak_src,
            "share_of_step": round(sum(per_m_us[M] for M in fam[dom]) / sum(per_m_us.values()), 3)}

    # ---- the floor of one launch that only reads the same bytes ----------------
    floor = run_read_floor(stream, copies, peak, calls=min(250, max(20, args.steps)))

    # ---- every workload of the specification, >= 200 graphed calls each ------
    per_config = None
    if args.per_config_calls > 0:
        del copies, graphs
        torch.cuda.empty_cache()
        with ClockSampler(local) as clk_pc:
            per_config = run_per_config(dev, stream, peak, calls=args.per_config_calls)
        per_config = {"points": per_config, "clocks": clk_pc.summary(),
                      "timing": f"per point: one CUDA graph of {args.per_config_calls} back-to-back "
                                f"calls on rotating weight copies (>= 4x L2 in all), replayed "
                                f"{PC_REPS} times after one untimed replay; CUDA events on the "
                                f"launching stream"}

    cpu = None
    if rank == 0 and ws == 1 and args.cpu_seconds > 0:
        cpu = cpu_baseline(seconds=args.cpu_seconds)

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_max * 1e3 / args.steps, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3", "data": "synthetic (seeded; packed 3-bit codes, E4M3 codebooks "
                                    "and activations, E8M0 scales)",
            "config": {"workload": WORKLOAD, "M": list(MS), "K": K_DIM, "N": N_DIM,
                       "weight_bytes_per_call": weight_bytes(),
                       "l2": f"inputs larger than L2: {ROTATE} rotating weight copies "
                             f"({ROTATE * weight_bytes() / 1e6:.0f} MB) vs 129 MB L2",
                       "timing": f"per-M CUDA graphs of {S} calls, {reps} rounds; {kernel_timing}",
                       "parallelism": f"replicas x{ws}"},
            "roofline": roof, "per_call": per_call, "read_floor": floor,
            "e2e": e2e, "cpu_baseline": cpu, "per_config": per_config,
            "gpu_launches": int(launches_per_step * args.steps),
            "clocks": clk.summary(),
        }
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_e2e(dev, stream, copies, args):
    """Same metric through the public API with host buffers: every step copies
    the activations and a_scale from pinned host memory, runs cbq_gemm for
    M = 1, 2, 4, 8 and reads every y back to pinned host memory, then the host
    waits for the step.  A step is captured once as a CUDA graph (copies and
    calls, as a serving loop would) -- one graph per group of 4 weight copies,
    cycled, so consecutive steps read different weights."""
    # the step's inputs (activations and a_scale of every M) travel in one
    # host-to-device copy, its outputs (every y) in one device-to-host copy
    a_bytes = {M: M * K_DIM for M in MS}
    pad = lambda n: (n + 255) // 256 * 256             # every piece 256-byte aligned
    in_bytes = sum(pad(a_bytes[M]) + pad(4 * M) for M in MS)
    host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    dev_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    host_y = torch.empty(sum(M * N_DIM for M in MS), dtype=torch.float32).pin_memory()
    dev_y = torch.empty_like(host_y, device=dev)
    views_a, views_s, views_y = {}, {}, {}
    off, yoff = 0, 0
    for M in MS:
        host_in[off:off + a_bytes[M]].copy_(torch.from_numpy(synth.gen_activations(M, K_DIM, seed=10 + M)).view(-1))
        views_a[M] = dev_in[off:off + a_bytes[M]].view(M, K_DIM)
        off += pad(a_bytes[M])
        host_in[off:off + 4 * M].copy_(torch.from_numpy(synth.gen_a_scale(M, seed=20 + M, mode="uniform")).view(torch.uint8))
        views_s[M] = dev_in[off:off + 4 * M].view(torch.float32)
        off += pad(4 * M)
        views_y[M] = dev_y[yoff:yoff + M * N_DIM].view(M, N_DIM)
        yoff += M * N_DIM
    steps = max(20, min(args.steps, 1000))

    def record(first_copy):
        dev_in.copy_(host_in, non_blocking=True)
        for idx, M in enumerate(MS):
            ops.gemm(views_a[M], views_s[M], copies[(first_copy + idx) % ROTATE], out=views_y[M], stream=stream)
        host_y.copy_(dev_y, non_blocking=True)

    graphs = []
    with torch.cuda.stream(stream):
        record(0)                                 # eager once (scratch, warm-up)
    stream.synchronize()
    for gi in range(ROTATE // len(MS)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            record(gi * len(MS))
        graphs.append(g)
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()
    stream.synchronize()
    t = time.perf_counter()
    for i in range(steps):
        with torch.cuda.stream(stream):
            graphs[i % len(graphs)].replay()
        stream.synchronize()
    dt = time.perf_counter() - t
    h2d = sum(a_bytes[M] + 4 * M for M in MS)            # payload (the copy also moves the padding)
    d2h = host_y.numel() * 4
    return {"value": round(steps * len(MS) * weight_bytes() / dt / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(dt * 1e3 / steps, 4),
            "mode": "one CUDA graph per step (one H2D copy of all inputs, 4 cbq_gemm calls, one D2H "
                    "copy of all outputs), host waits every step"}


PC_REPS = 4
L2_FALLBACK = 129 * 10**6


def workload_bytes(wl) -> tuple[int, int]:
    """(packed weight bytes read, algorithmic bytes) of one call of a workload.
    A grouped call reads only the budgeted experts; its output holds one row
    per (token, chosen expert) and it also reads the routing indices."""
    wb = weight_bytes(wl.N, wl.K)
    if wl.experts:
        w_read = wl.budget * wb
        return w_read, w_read + wl.M * wl.K + 4 * wl.M + 4 * wl.M * wl.topk * wl.N + 4 * wl.M * wl.topk
    return wb, wb + wl.M * wl.K + 4 * wl.M + 4 * wl.M * wl.N


def run_per_config(dev, stream, peak, calls=250):
    """Every workload of the specification timed the same way: one CUDA graph
    of `calls` back-to-back calls through the public API, each call on the next
    of R weight copies (R chosen so the copies fill at least 4x L2), one
    untimed replay, then PC_REPS timed replays between CUDA events on the
    launching stream."""
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", L2_FALLBACK) or L2_FALLBACK
    points = []
    for name, wl in synth.workloads().items():
        rows = wl.experts * wl.N if wl.experts else wl.N
        pw = synth.gen_weights(rows, wl.K, seed=1)
        w0 = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, wl.N, wl.K, device=dev)
        copy_bytes = w0.nbytes
        R = int(min(512, max(2, -(-4 * l2 // copy_bytes))))
        copies = [w0] + [ops.PackedWeights(w0.codes.clone(), w0.scales.clone(), w0.codebooks.clone(),
                                           wl.N, wl.K) for _ in range(R - 1)]
        a = torch.from_numpy(synth.gen_activations(wl.M, wl.K, seed=2, half_normal=wl.half_normal)).to(dev)
        s = torch.from_numpy(synth.gen_a_scale(wl.M, seed=3, mode=wl.a_scale)).to(dev)
        if wl.experts:
            idx = torch.from_numpy(synth.gen_moe_routing(wl.M, wl.experts, wl.budget, wl.topk, seed=4)).to(dev)
            y = torch.empty((wl.M, wl.topk, wl.N), dtype=torch.float32, device=dev)
            run = lambda w: ops.grouped_gemm(a, s, w, wl.experts, idx, out=y, stream=stream)  # noqa: E731
            kernel = KERNEL_NAMES[ops.PATH_GEMV if wl.M <= 4 else ops.PATH_MMA]
        else:
            y = torch.empty((wl.M, wl.N), dtype=torch.float32, device=dev)
            run = lambda w: ops.gemm(a, s, w, out=y, stream=stream)  # noqa: E731
            kernel = KERNEL_NAMES[ops.auto_path(wl.M, wl.N, wl.K)]
        with torch.cuda.stream(stream):
            for i in range(3):
                run(copies[i % R])
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(calls):
                run(copies[i % R])
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(PC_REPS + 1)]
        with torch.cuda.stream(stream):
            g.replay()
            ev[0].record(stream)
            for r in range(PC_REPS):
                g.replay()
                ev[r + 1].record(stream)
        stream.synchronize()
        if ops.device_status(stream) != ops.OK:
            raise RuntimeError(f"device status not ok after {name}")
        us = ev[0].elapsed_time(ev[-1]) * 1e3 / (PC_REPS * calls)
        w_read, alg = workload_bytes(wl)
        points.append({"workload": name, "M": wl.M, "N": wl.N, "K": wl.K,
                       **({"experts": wl.experts, "budget": wl.budget, "topk": wl.topk} if wl.experts else {}),
                       "kernel": kernel, "us": round(us, 3),
                       "weight_GBps": round(w_read / us / 1e3, 1),
                       "roofline_frac": round(alg / us / 1e3 / peak, 4),
                       "tokens_per_s": round(wl.M / us * 1e6, 1),
                       "weight_copies": R})
        del g, copies, w0, y
        torch.cuda.empty_cache()
    points += run_gate_up_points(dev, stream, peak, calls, l2)
    points += run_draft_head_points(dev, stream, peak, calls, l2)
    points += run_budget_points(dev, stream, calls)
    return points


def run_budget_points(dev, stream, calls):
    """cbq_select_budget (the verify round's shared expert budget and each
    token's top-k inside it) on seeded N(0,1) router logits, timed like the
    other points.  Its input is a few KB to 1 MB of logits, so the time is
    latency, not bandwidth: no roofline fraction."""
    points = []
    for name, (T, E, k, B) in synth.budget_workloads().items():
        logits = torch.from_numpy(synth.gen_router_logits(T, E, seed=5)).to(dev)
        run = lambda: ops.select_budget(logits, k, B, stream=stream)  # noqa: E731
        with torch.cuda.stream(stream):
            for _ in range(3):
                run()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(calls):
                run()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(PC_REPS + 1)]
        with torch.cuda.stream(stream):
            g.replay()
            ev[0].record(stream)
            for r in range(PC_REPS):
                g.replay()
                ev[r + 1].record(stream)
        stream.synchronize()
        if ops.device_status(stream) != ops.OK:
            raise RuntimeError(f"device status not ok after {name}")
        us = ev[0].elapsed_time(ev[-1]) * 1e3 / (PC_REPS * calls)
        points.append({"workload": name, "T": T, "E": E, "k": k, "B": B,
                       "kernel": "budget_own_kernel + budget_sort_kernel + budget_pick_kernel",
                       "us": round(us, 3), "roofline_frac": None})
        del g
    return points


def run_draft_head_points(dev, stream, peak, calls, l2):
    """cbq_draft_head on the vocabulary-head shape, timed like the other
    points (the 2-bit head rotated over copies >= 4x L2; one FP8 head, of
    which a call reads 16 rows per token).  Algorithmic bytes: the 2-bit head
    (KN/4 + KN/32 + 4N), the FP8 rows and row scales read, the activations
    and their scales, the shortlist, logits and picks written."""
    points = []
    for name, wl in synth.draft_head_workloads().items():
        M, N, K = wl.M, wl.N, wl.K
        h2 = synth.gen_head2(N, K, seed=1)
        w0 = ops.PackedWeights.from_host(h2.codes, h2.scales, h2.codebooks, N, K, device=dev)
        R = int(min(512, max(2, -(-4 * l2 // w0.nbytes))))
        copies = [w0] + [ops.PackedWeights(w0.codes.clone(), w0.scales.clone(), w0.codebooks.clone(), N, K)
                         for _ in range(R - 1)]
        h8, rs = synth.gen_head8(N, K, seed=2)
        h8, rs = torch.from_numpy(h8).to(dev), torch.from_numpy(rs).to(dev)
        a = torch.from_numpy(synth.gen_activations(M, K, seed=3)).to(dev)
        s = torch.from_numpy(synth.gen_a_scale(M, seed=4, mode="uniform")).to(dev)
        run = lambda w: ops.draft_head(a, s, w, h8, rs, stream=stream)  # noqa: E731
        with torch.cuda.stream(stream):
            for i in range(3):
                run(copies[i % R])
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(calls):
                run(copies[i % R])
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(PC_REPS + 1)]
        with torch.cuda.stream(stream):
            g.replay()
            ev[0].record(stream)
            for r in range(PC_REPS):
                g.replay()
                ev[r + 1].record(stream)
        stream.synchronize()
        if ops.device_status(stream) != ops.OK:
            raise RuntimeError(f"device status not ok after {name}")
        us = ev[0].elapsed_time(ev[-1]) * 1e3 / (PC_REPS * calls)
        wb = K * N // 4 + K * N // 32 + 4 * N
        alg = wb + M * 16 * (K + 4) + M * K + 4 * M + M * 16 * 8 + 4 * M
        points.append({"workload": name, "M": M, "N": N, "K": K,
                       "kernel": "sk_kernel (2-bit) + head_topk_chunk_kernel + head_select_kernel",
                       "us": round(us, 3), "weight_GBps": round(wb / us / 1e3, 1),
                       "roofline_frac": round(alg / us / 1e3 / peak, 4),
                       "tokens_per_s": round(M / us * 1e6, 1), "weight_copies": R})
        del g, copies, w0, h8
        torch.cuda.empty_cache()
    return points


# the fused gate-up step on the two gate+up shapes of the specification:
# (name, M, F, K); the packed weight holds N = 2F rows
GATE_UP_POINTS = [("gate_up_4096x6144_m1", 1, 6144, 4096), ("gate_up_4096x6144_m8", 8, 6144, 4096),
                  ("gate_up_5120x12800_m16", 16, 12800, 5120)]


def run_gate_up_points(dev, stream, peak, calls, l2):
    """cbq_gemm_gate_up timed like the other points: the matmul against the
    2F-row gate+up weight, SiLU(gate) * up, and the per-token E4M3
    quantisation of the products.  Algorithmic bytes: the packed weight, the
    activations and their scales in, the E4M3 products and their per-token
    scales out."""
    points = []
    for name, M, F, K in GATE_UP_POINTS:
        N = 2 * F
        pw = synth.gen_weights(N, K, seed=1)
        w0 = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, N, K, device=dev)
        R = int(min(512, max(2, -(-4 * l2 // w0.nbytes))))
        copies = [w0] + [ops.PackedWeights(w0.codes.clone(), w0.scales.clone(), w0.codebooks.clone(), N, K)
                         for _ in range(R - 1)]
        a = torch.from_numpy(synth.gen_activations(M, K, seed=2)).to(dev)
        s = torch.from_numpy(synth.gen_a_scale(M, seed=3, mode="uniform")).to(dev)
        q = torch.empty((M, F), dtype=torch.uint8, device=dev)
        qs = torch.empty((M,), dtype=torch.float32, device=dev)
        run = lambda w: ops.gate_up(a, s, w, out=q, out_scale=qs, stream=stream)  # noqa: E731
        with torch.cuda.stream(stream):
            for i in range(3):
                run(copies[i % R])
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(calls):
                run(copies[i % R])
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(PC_REPS + 1)]
        with torch.cuda.stream(stream):
            g.replay()
            ev[0].record(stream)
            for r in range(PC_REPS):
                g.replay()
                ev[r + 1].record(stream)
        stream.synchronize()
        if ops.device_status(stream) != ops.OK:
            raise RuntimeError(f"device status not ok after {name}")
        us = ev[0].elapsed_time(ev[-1]) * 1e3 / (PC_REPS * calls)
        wb = weight_bytes(N, K)
        alg = wb + M * K + 4 * M + M * F + 4 * M
        points.append({"workload": name, "M": M, "F": F, "N": N, "K": K,
                       "kernel": "sk_kernel (gate-up epilogue) + gate_up_quant_kernel", "us": round(us, 3),
                       "weight_GBps": round(wb / us / 1e3, 1), "roofline_frac": round(alg / us / 1e3 / peak, 4),
                       "tokens_per_s": round(M / us * 1e6, 1), "weight_copies": R})
        del g, copies, w0
        torch.cuda.empty_cache()
    return points


def run_read_floor(stream, copies, peak, calls=250):
    """Where one launch's floor is on this workload: a device-to-device copy
    (Tensor.copy_, one library launch per call) of the code bytes of one call,
    from the same rotating copies, timed the same way as the calls (a CUDA
    graph of back-to-back launches, CUDA events around PC_REPS replays).  It
    moves twice the code bytes (read + write), as the measured copy peak does;
    `read_us` is the time a launch that only reads the call's code bytes
    would take at the copy's rate (half the copy's time)."""
    src = [w.codes for w in copies]
    dst = torch.empty_like(src[0])
    with torch.cuda.stream(stream):
        for i in range(3):
            dst.copy_(src[i % len(src)])
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(calls):
            dst.copy_(src[i % len(src)])
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(PC_REPS + 1)]
    with torch.cuda.stream(stream):
        g.replay()
        ev[0].record(stream)
        for r in range(PC_REPS):
            g.replay()
            ev[r + 1].record(stream)
    stream.synchronize()
    us = ev[0].elapsed_time(ev[-1]) * 1e3 / (PC_REPS * calls)
    nbytes = src[0].numel()
    moved = 2 * nbytes
    return {"op": "Tensor.copy_ of one call's code bytes, device to device (one launch per call)",
            "bytes": nbytes, "bytes_moved": moved, "us": round(us, 3), "read_us": round(us / 2, 3),
            "GBps": round(moved / us / 1e3, 1), "frac": round(moved / us / 1e3 / peak, 4), "calls": calls,
            "copies": len(copies)}


def run_e2e_eager(dev, stream, copies, steps):
    """The e2e step without CUDA graphs: every step copies the inputs from
    pinned host memory, calls cbq_gemm for M = 1, 2, 4, 8 from the host (one
    library call per matmul, as an eager caller would), reads every y back
    and waits."""
    a_host = {M: torch.from_numpy(synth.gen_activations(M, K_DIM, seed=10 + M)).pin_memory() for M in MS}
    s_host = {M: torch.from_numpy(synth.gen_a_scale(M, seed=20 + M, mode="uniform")).pin_memory() for M in MS}
    a_dev = {M: torch.empty_like(a_host[M], device=dev) for M in MS}
    s_dev = {M: torch.empty_like(s_host[M], device=dev) for M in MS}
    y_dev = {M: torch.empty((M, N_DIM), dtype=torch.float32, device=dev) for M in MS}
    y_host = {M: torch.empty((M, N_DIM), dtype=torch.float32).pin_memory() for M in MS}
    call = [0]

    def step():
        with torch.cuda.stream(stream):
            for M in MS:
                a_dev[M].copy_(a_host[M], non_blocking=True)
                s_dev[M].copy_(s_host[M], non_blocking=True)
            for M in MS:
                ops.gemm(a_dev[M], s_dev[M], copies[call[0] % len(copies)], out=y_dev[M], stream=stream)
                call[0] += 1
            for M in MS:
                y_host[M].copy_(y_dev[M], non_blocking=True)
        stream.synchronize()

    for _ in range(5):
        step()
    t = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t
    return {"value": round(steps * len(MS) * weight_bytes() / dt / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": sum(M * K_DIM + 4 * M for M in MS),
            "d2h_bytes_per_step": sum(4 * M * N_DIM for M in MS), "steps": steps,
            "ms_per_step": round(dt * 1e3 / steps, 4),
            "mode": "eager: per step 8 H2D copies, 4 cbq_gemm calls from the host, 4 D2H copies, "
                    "host waits every step"}


# ------------------------------------------------------- oracle (CPU) arm --

def _oracle_step(o, pw, acts, scs, rows):
    sel = np.arange(rows)
    for M in MS:
        o.gemm_rows(acts[M], scs[M], pw.codes, pw.scales, pw.codebooks, M, N_DIM, K_DIM, sel)


def cpu_baseline(seconds: float):
    """The oracle as it stands, on the host cores, on a row sample of the step."""
    import oracle as o
    pw = synth.gen_weights(N_DIM, K_DIM, seed=1)
    acts = {M: synth.gen_activations(M, K_DIM, seed=10 + M) for M in MS}
    scs = {M: synth.gen_a_scale(M, seed=20 + M, mode="uniform") for M in MS}
    rows = 64
    t = time.perf_counter()
    _oracle_step(o, pw, acts, scs, rows)
    probe = time.perf_counter() - t
    rows = int(min(N_DIM, max(64, rows * seconds / max(probe, 1e-3))))
    passes, t = 0, time.perf_counter()
    while True:                      # whole passes until the budget is spent
        _oracle_step(o, pw, acts, scs, rows)
        passes += 1
        dt = time.perf_counter() - t
        if dt >= seconds or passes >= 100:
            break
    units = passes * len(MS) * weight_bytes() * rows / N_DIM
    return {"value": round(units / dt / 1e9, 4), "unit": "GB/s", "cores": o.num_threads(),
            "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of N={N_DIM} at each M in {list(MS)}, {passes} "
                      f"pass(es) in {dt:.1f} s; plain C, fp64, OpenMP over rows",
            "seconds": round(dt, 2)}


def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1:
        dist_init(ws, "gloo")
    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    import oracle as o
    o.build()
    pw = synth.gen_weights(N_DIM, K_DIM, seed=1)
    acts = {M: synth.gen_activations(M, K_DIM, seed=10 + M) for M in MS}
    scs = {M: synth.gen_a_scale(M, seed=20 + M, mode="uniform") for M in MS}
    # size each step's row sample so warm-up + timed steps take about a minute
    t = time.perf_counter()
    _oracle_step(o, pw, acts, scs, 16)
    per_row = (time.perf_counter() - t) / 16
    total_steps = max(1, args.steps + args.warmup)
    rows = int(min(N_DIM, max(1, args.ref_seconds / total_steps / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        _oracle_step(o, pw, acts, scs, rows)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(o, pw, acts, scs, rows)
    dt = time.perf_counter() - t
    units = args.steps * len(MS) * weight_bytes() * rows / N_DIM
    value = units / dt / 1e9
    out = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": WORKLOAD, "M": list(MS), "K": K_DIM, "N": N_DIM},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": o.num_threads(),
                            "kind": "oracle",
                            "sample": f"each step: rows 0..{rows - 1} of N={N_DIM} at every M"},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_single(args):
    """A few back-to-back calls of one named workload on one kernel, for
    profiler captures (cold cache per profiler pass)."""
    from bit_codebook_quantized_gb300 import build as _b
    _b.build()
    dev = torch.device("cuda", 0)
    gu = {name: (M, F, K) for name, M, F, K in GATE_UP_POINTS}
    if args.single in gu:
        # the fused gate-up step: matmul with the SiLU-product epilogue, then
        # the per-token E4M3 quantisation
        M, F, K = gu[args.single]
        pw = synth.gen_weights(2 * F, K, seed=1)
        w = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, 2 * F, K, device=dev)
        a = torch.from_numpy(synth.gen_activations(M, K, seed=2)).to(dev)
        s = torch.from_numpy(synth.gen_a_scale(M, seed=3, mode="uniform")).to(dev)
        for _ in range(args.calls):
            ops.gate_up(a, s, w)
        torch.cuda.synchronize()
        st = ops.device_status()
        print(json.dumps({"single": args.single, "calls": args.calls, "status": st}))
        if st != ops.OK:
            sys.exit(1)
        return
    if args.single in synth.budget_workloads():
        # the verify round's expert budget on seeded router logits
        T, E, k, B = synth.budget_workloads()[args.single]
        logits = torch.from_numpy(synth.gen_router_logits(T, E, seed=5)).to(dev)
        for _ in range(args.calls):
            ops.select_budget(logits, k, B)
        torch.cuda.synchronize()
        st = ops.device_status()
        print(json.dumps({"single": args.single, "calls": args.calls, "status": st}))
        if st != ops.OK:
            sys.exit(1)
        return
    if args.single in synth.draft_head_workloads():
        # the draft head: 2-bit scores, shortlist, FP8 rescoring and pick
        wl = synth.draft_head_workloads()[args.single]
        h2 = synth.gen_head2(wl.N, wl.K, seed=1)
        h8, rs = synth.gen_head8(wl.N, wl.K, seed=2)
        w = ops.PackedWeights.from_host(h2.codes, h2.scales, h2.codebooks, wl.N, wl.K, device=dev)
        h8, rs = torch.from_numpy(h8).to(dev), torch.from_numpy(rs).to(dev)
        a = torch.from_numpy(synth.gen_activations(wl.M, wl.K, seed=3)).to(dev)
        s = torch.from_numpy(synth.gen_a_scale(wl.M, seed=4, mode="uniform")).to(dev)
        for _ in range(args.calls):
            ops.draft_head(a, s, w, h8, rs)
        torch.cuda.synchronize()
        st = ops.device_status()
        print(json.dumps({"single": args.single, "calls": args.calls, "status": st}))
        if st != ops.OK:
            sys.exit(1)
        return
    wl = synth.workloads()[args.single]
    if wl.experts:
        pw = synth.gen_weights(wl.experts * wl.N, wl.K, seed=1)
        idx = torch.from_numpy(synth.gen_moe_routing(wl.M, wl.experts, wl.budget, wl.topk, seed=4)).to(dev)
        y = torch.empty((wl.M, wl.topk, wl.N), device=dev)
    else:
        pw = synth.gen_weights(wl.N, wl.K, seed=1)
        y = torch.empty((wl.M, wl.N), device=dev)
    w = ops.PackedWeights.from_host(pw.codes, pw.scales, pw.codebooks, wl.N, wl.K, device=dev)
    a = torch.from_numpy(synth.gen_activations(wl.M, wl.K, seed=2, half_normal=wl.half_normal)).to(dev)
    s = torch.from_numpy(synth.gen_a_scale(wl.M, seed=3, mode=wl.a_scale)).to(dev)
    for _ in range(args.calls):
        if wl.experts:
            ops.grouped_gemm(a, s, w, wl.experts, idx, out=y, path=args.path)
        else:
            ops.gemm(a, s, w, out=y, path=args.path)
    torch.cuda.synchronize()
    st = ops.device_status()
    print(json.dumps({"single": args.single, "path": args.path, "calls": args.calls, "status": st}))
    if st != ops.OK:
        sys.exit(1)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU-baseline budget on rank 0 (0 disables)")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: CPU seconds the whole run should take")
    ap.add_argument("--single", default=None,
                    help="run --calls calls of one workload (see synth.workloads(), "
                         "synth.draft_head_workloads(), synth.budget_workloads() and the gate-up "
                         "points, e.g. gate_up_4096x6144_m8) and exit")
    ap.add_argument("--path", type=int, default=0, help="kernel for --single: 0 auto, 1 gemv, 2 mma, 3 stream-K")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--per-config-calls", type=int, default=250,
                    help="graphed calls per point of the all-workload leg (0 disables)")
    args = ap.parse_args(argv)
    if args.single:
        run_single(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
