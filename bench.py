#!/usr/bin/env python
"""Throughput of the KDA chunked forward pass on GB300 (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one full forward pass (every kernel of kda_fwd) over one batch of
seeded synthetic inputs shaped like the workload (gated_delta_rule_51_gb300/
inputs.py).  `value` is whole-job tokens/s with the inputs already resident in
HBM; `e2e` repeats the measurement through the public API with pinned host
buffers, the host->device input copies and the device->host result copies
inside the timed region.  The roofline object reports the forward kernel's
compulsory HBM bytes (1282 B per token-head plus states and gate parameters)
over its CUDA-event duration against the measured copy bandwidth.

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload (no runnable FlashKDA code is available).
Under torchrun every rank runs its own replica of the workload (weak scaling,
no data-path collective); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA fwd tokens/s and % of roofline (TFLOP/s, HBM GB/s) on 1xGB300"
DEFAULT_CONFIG = "varlen_T32768_N8_H32"
BYTES_PER_TOKEN_HEAD = 4 * 128 * 2 + 2 + 128 * 2      # q, k, v, g + beta + out (bf16)
FLOPS_PER_TOKEN_HEAD = 6 * 128 * 128 + 6 * 16 * 128 + 4 * 16 * 128   # 16-token chunked form
L2_BYTES = 126 * 1024 * 1024
ALIASES = {"tiny": "tiny_B1_T64_H1", "fixed": "fixed_B2_T4096_H16",
           "varlen": "varlen_T32768_N8_H32", "long": "long_T1048576_H8", "decode": "decode_B256_T1_H32"}
DECODE_METRIC = "KDA decode tokens/s and % of HBM roofline on 1xGB300"
BWD_METRIC = "KDA bwd tokens/s and % of HBM roofline on 1xGB300"
# the backward's compulsory traffic per token-head: q, k, v, g, dout (bf16) and beta read;
# dq, dk, dv, dg (fp32) and dbeta written
BWD_BYTES_PER_TOKEN_HEAD = 5 * 128 * 2 + 2 + 4 * 128 * 4 + 4


def workload(name):
    from gated_delta_rule_51_gb300 import inputs as I

    ws = I.named_workloads()
    name = ALIASES.get(name, name)
    if name not in ws:
        raise SystemExit(f"unknown config {name}; choose from {sorted(ws)}")
    return ws[name]


def compulsory_bytes(w) -> int:
    """Bytes the method must move: inputs, outputs, states, gate parameters."""
    import torch

    sb = 0
    if w.state_dtype is not None:
        per = 128 * 128 * (4 if w.state_dtype == torch.float32 else 2)
        sb = w.N * w.H * per * (int(w.has_initial_state) + int(w.has_final_state))
    params = w.H * 4 + w.H * 128 * 4
    cu = 8 * (w.N + 1) if w.seq_lens is not None else 0
    return w.token_heads * BYTES_PER_TOKEN_HEAD + sb + params + cu


def config_dict(w, extra=None):
    d = {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "K": 128, "V": 128, "N": w.N,
         "state": str(w.state_dtype).replace("torch.", "") if w.state_dtype is not None else None,
         "initial_state": w.has_initial_state, "lower_bound": w.lower_bound, "seed": w.seed,
         "token_heads": w.token_heads}
    if w.seq_lens is not None:
        d["seq_lens"] = w.seq_lens if len(w.seq_lens) <= 16 else f"{len(w.seq_lens)} lengths"
    if extra:
        d.update(extra)
    return d


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# the source files each measured kernel is built from (its own file, the device helpers and
# the parameter structs): a committed DRAM count stands while none of them has changed
KERNEL_FILES = {"chain": ("kda_chain.cuh", "kda_chain.cu", "kda_device.cuh", "kda_internal.h"),
                "decode": ("kda_decode.cu", "kda_device.cuh", "kda_internal.h"),
                "bwd": ("kda_bwd.cu", "kda_device.cuh", "kda_internal.h"),
                "chain_bwd": ("kda_chain.cuh", "kda_chain_bwd.cu", "kda_device.cuh", "kda_internal.h")}


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines, each line's trailing spaces
    dropped: the code a compiler sees, so that editing a comment leaves it unchanged."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":                                    # string or character literal
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash(files=None) -> str:
    """sha256 (first 16 hex digits) over the given csrc files in order (default all of
    them), comments and blank lines removed."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_51_gb300", "csrc")
    for f in (files if files is not None else sorted(os.listdir(csrc))):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload_name: str):
    """DRAM bytes per launch of the workload's dominant kernel from the committed ncu
    summary, if it was taken on that kernel's current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload_name)
    if not e or e.get("kernel_files") not in KERNEL_FILES:
        return None
    if e.get("kernel_source_hash") != kernel_source_hash(KERNEL_FILES[e["kernel_files"]]):
        return None
    return e.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_sample(w, x_cpu, budget_s: float = 15.0):
    """Time the fp64 oracle, as it stands, on a bounded sample of the workload.

    The sample is the first sequences (whole, or a prefix of the first one) of
    the first heads, sized to about `budget_s` of CPU time; tokens/s is scaled
    by the fraction of the workload's token-heads covered."""
    import torch

    import oracle

    threads = os.cpu_count() or 1
    lens = w.seq_lens if w.seq_lens is not None else [w.T] * w.B
    budget_th = int(budget_s * 20000 * threads)    # ~20k token-heads/s per thread
    heads = min(w.H, max(1, threads))
    nseq, tok = 0, 0
    for L in lens:
        if (tok + L) * heads > budget_th and nseq > 0:
            break
        nseq += 1
        tok += L
    if tok * heads > budget_th:                    # one sequence too long: take a prefix
        tok = max(16, budget_th // heads)
    if w.seq_lens is not None:
        q, k, v, g, beta = (x_cpu[n][:, :tok, :heads].contiguous() for n in ("q", "k", "v", "g", "beta"))
        bounds = [0]
        for L in lens[:nseq]:
            bounds.append(min(tok, bounds[-1] + L))
        cu = torch.tensor(bounds, dtype=torch.int64)
        init = x_cpu["initial_state"][:nseq, :heads].contiguous() if x_cpu["initial_state"] is not None else None
    else:
        rows = max(1, min(nseq, w.B))
        t_len = min(tok, w.T)
        q, k, v, g, beta = (x_cpu[n][:rows, :t_len, :heads].contiguous() for n in ("q", "k", "v", "g", "beta"))
        cu = None
        init = x_cpu["initial_state"][:rows, :heads].contiguous() if x_cpu["initial_state"] is not None else None
    th = q.shape[0] * q.shape[1] * heads
    t0 = time.perf_counter()
    oracle.kda_forward(q, k, v, g, beta, x_cpu["scale"], x_cpu["A_log"][:heads].contiguous(),
                       x_cpu["dt_bias"][:heads].contiguous(), x_cpu["lower_bound"], init, cu,
                       nthreads=threads)
    dt = time.perf_counter() - t0
    tokens_per_s = (th / w.H) / dt
    desc = (f"{th} token-heads ({q.shape[0]}x{q.shape[1]} tokens x {heads} of {w.H} heads"
            f"{', ' + str(len(cu) - 1) + ' sequences' if cu is not None else ''}); tokens/s scaled by "
            f"covered token-heads / H")
    return tokens_per_s, threads, desc, dt


def bwd_oracle_sample(w, x_cpu, dout, dfinal, tokens: int = 512, heads: int = 8):
    """Time the fp64 gradient oracle, as it stands, on the first `tokens` tokens of every
    sequence (each batch row) and the first `heads` heads (one thread per (sequence, head)
    pair); tokens/s is scaled by the fraction of the workload's token-heads covered."""
    import oracle

    tt, hs = min(tokens, w.T), list(range(min(heads, w.H)))
    cut = lambda t: t[:, :tt][:, :, hs].double().numpy()
    cu = None
    if x_cpu["cu_seqlens"] is not None:
        # the first sequences that fit in tt tokens
        import numpy as np

        c = x_cpu["cu_seqlens"].numpy()
        keep = [0] + [int(e) for e in c[1:] if e <= tt]
        cu = np.array(keep if keep[-1] == tt else keep + [tt], dtype=np.int64)
    nseq = (len(cu) - 1) if cu is not None else w.B
    init = x_cpu["initial_state"]
    init = init[:nseq][:, hs].double().numpy() if init is not None else None
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.kda_backward(cut(x_cpu["q"]), cut(x_cpu["k"]), cut(x_cpu["v"]), cut(x_cpu["g"]), cut(x_cpu["beta"]),
                        float(x_cpu["scale"]), x_cpu["A_log"][hs].double().numpy(),
                        x_cpu["dt_bias"][hs].double().numpy(), float(x_cpu["lower_bound"]), cut(dout), init,
                        dfinal[:nseq][:, hs].double().numpy(), cu, nthreads=threads)
    dt = time.perf_counter() - t0
    th = w.B * tt * len(hs)
    desc = (f"{th} token-heads ({w.B}x{tt} tokens x {len(hs)} of {w.H} heads); tokens/s scaled by "
            "covered token-heads / H")
    return th / dt / w.H, min(threads, nseq * len(hs)), desc, dt


def bwd_upstream_grads(w, device, generator):
    """dout (bf16 N(0, 1), the shape of out) and dfinal (fp32 0.1 N(0, 1)) for the backward."""
    import torch

    dout = torch.randn((w.B, w.T, w.H, 128), generator=generator, device=device).to(torch.bfloat16)
    dfinal = 0.1 * torch.randn((w.N, w.H, 128, 128), generator=generator, device=device)
    return dout, dfinal


def capture_steps(torch, dev, stream, kda, step, ev, steps):
    """One CUDA graph per timed step, each recording that step's profile events (ev[i][1:]).
    Returns (graphs, launch mode); without graph capture, ([], the reason) and the caller
    times direct calls."""
    graphs = []
    try:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for i in range(steps):
                g = torch.cuda.CUDAGraph()
                kda.set_profile_events(ev[i][1:])
                with torch.cuda.graph(g, stream=cap):
                    step()
                graphs.append(g)
        kda.set_profile_events(None)
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        return graphs, "cuda graph per step"
    except Exception as exc:        # capture not available: time direct calls instead
        kda.set_profile_events(None)
        return [], f"direct calls ({type(exc).__name__} in graph capture)"


def run_bwd_reference(args, w):
    """--impl reference for the backward: the fp64 gradient oracle on the host cores, timed
    per step on a bounded sample of the workload (rank 0 only)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import torch

    from gated_delta_rule_51_gb300 import inputs as I
    import oracle

    oracle.build()
    x = I.make_inputs(w, device="cpu")
    dout, dfinal = bwd_upstream_grads(w, "cpu", torch.Generator().manual_seed(w.seed + 100))
    for _ in range(args.warmup):
        bwd_oracle_sample(w, x, dout, dfinal)
    vals, times = [], []
    desc, threads = "", 1
    for _ in range(args.steps):
        v, threads, desc, dt = bwd_oracle_sample(w, x, dout, dfinal)
        vals.append(v)
        times.append(dt)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": BWD_METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * statistics.mean(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, {"pass": "backward", "parallelism": "cpu threads"}),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's value (timings: the job ends with its slowest rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: int, world: int, steps: int, max_ms: float) -> float:
    """Units per second of the whole job: every rank runs its own replica of the workload
    (weak scaling), so the job processes world x steps x units in the slowest rank's time."""
    return units_per_rank_step * world * steps / (max_ms / 1000.0)


def run_reference(args, w):
    """--impl reference: the fp64 oracle on the host cores, timed per step on a bounded sample."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from gated_delta_rule_51_gb300 import inputs as I
    import oracle

    oracle.build()
    x = I.make_inputs(w, device="cpu")
    budget = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_sample(w, x, budget)
    vals, times = [], []
    desc, threads = "", 1
    for _ in range(args.steps):
        v, threads, desc, dt = cpu_oracle_sample(w, x, budget)
        vals.append(v)
        times.append(dt)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * statistics.mean(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, {"parallelism": "cpu threads"}),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    from gated_delta_rule_51_gb300 import inputs as I
    from gated_delta_rule_51_gb300 import kda

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    kda.load_library()
    x = I.make_inputs(w, device=dev)          # replicas: every rank runs its own copy
    out = torch.empty((w.B, w.T, w.H, 128), dtype=torch.bfloat16, device=dev)
    fin = (torch.empty((w.N, w.H, 128, 128), dtype=w.state_dtype, device=dev)
           if w.has_final_state else None)
    ws = torch.empty(kda.workspace_size(kda.make_shape(w.B, w.T, w.H, w.N)), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], out, x["A_log"], x["dt_bias"],
                x["lower_bound"], initial_state=x["initial_state"], final_state=fin,
                cu_seqlens=x["cu_seqlens"], workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if kda.check_device_error(ws, dev):
        raise SystemExit("device error flags set during warm-up")
    launches_per_step = kda.last_launch_count()

    # timed region: per step an L2 flush, then start event, kernels (phase events).
    # Each step is one kda_fwd captured in a CUDA graph (as a serving loop would run it),
    # so the host-side argument checks do not sit between the GPU's steps; e2e below
    # times direct calls.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for e in ev:
        for t in e:
            t.record(stream)        # creates the events before their handles are handed out
    torch.cuda.synchronize(dev)
    graphs, launch_mode = capture_steps(torch, dev, stream, kda, step, ev, args.steps)
    barrier()
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            if graphs:
                graphs[i].replay()
            else:
                kda.set_profile_events(ev[i][1:])
                step()
        kda.set_profile_events(None)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    barrier()
    # launch phases: schedule, forward runs (every segment's forward, overlapping the
    # transition runs), carry composition with the corrections of the split segments (the
    # correction launch starts beside the composition); the fourth mark closes an empty phase
    step_ms = [e[0].elapsed_time(e[4]) for e in ev]
    sch_ms = [e[0].elapsed_time(e[1]) for e in ev]
    fwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    cmp_ms = [e[2].elapsed_time(e[3]) for e in ev]   # composition and corrections (one phase)
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    tokens = w.B * w.T
    value = whole_job_rate(tokens, world, args.steps, total_ms)
    ms_per_step = total_ms / args.steps

    # end to end through the public API with pinned host buffers.  Every step copies its
    # inputs host -> device and reads its outputs back; the steps are pipelined the way a
    # serving loop would run them: two sets of device buffers, the next step's inputs
    # copied on four copy streams while this step computes, its outputs copied back on a
    # fifth stream while the next step computes.
    e2e = None
    if not args.no_e2e:
        names = [n for n in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens") if x[n] is not None]
        host = {n: x[n].cpu().pin_memory() for n in names}
        host["A_log"], host["dt_bias"] = x["A_log"].cpu().pin_memory(), x["dt_bias"].cpu().pin_memory()
        names_all = names + ["A_log", "dt_bias"]
        nbuf = 2
        dev_in = [{n: torch.empty_like(x[n]) for n in names_all} for _ in range(nbuf)]
        outs = [torch.empty_like(out) for _ in range(nbuf)]
        fins = [torch.empty_like(fin) if fin is not None else None for _ in range(nbuf)]
        h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h_fin = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True) if fin is not None else None
        h2d = sum(host[n].numel() * host[n].element_size() for n in names_all)
        d2h = h_out.numel() * 2 + (h_fin.numel() * h_fin.element_size() if h_fin is not None else 0)
        copy_streams = [torch.cuda.Stream(dev) for _ in range(4)]
        d2h_stream = torch.cuda.Stream(dev)
        lane_of = {n: i % len(copy_streams) for i, n in enumerate(names_all)}
        in_free = [None] * nbuf     # events: the kernel that read buffer b is done
        out_free = [None] * nbuf    # events: the copy-back of output buffer b is done
        in_ready = [None] * nbuf

        def issue_h2d(i):
            b = i % nbuf
            evs = []
            for li, cs in enumerate(copy_streams):
                if in_free[b] is not None:
                    cs.wait_event(in_free[b])
                with torch.cuda.stream(cs):
                    for n in names_all:
                        if lane_of[n] == li:
                            dev_in[b][n].copy_(host[n], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                evs.append(ev)
            in_ready[b] = evs

        def issue_compute(i):
            b = i % nbuf
            for ev in in_ready[b]:
                stream.wait_event(ev)
            if out_free[b] is not None:
                stream.wait_event(out_free[b])
            d = dev_in[b]
            kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], outs[b], d["A_log"], d["dt_bias"],
                    x["lower_bound"], initial_state=d.get("initial_state"), final_state=fins[b],
                    cu_seqlens=d.get("cu_seqlens"), workspace=ws, stream=stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            in_free[b] = ev
            d2h_stream.wait_event(ev)
            with torch.cuda.stream(d2h_stream):
                h_out.copy_(outs[b], non_blocking=True)
                if h_fin is not None:
                    h_fin.copy_(fins[b], non_blocking=True)
            ev2 = torch.cuda.Event()
            ev2.record(d2h_stream)
            out_free[b] = ev2

        def run_pipeline(k_steps, e_start=None):
            if e_start is not None:
                for cs in copy_streams:
                    cs.wait_event(e_start)
            issue_h2d(0)
            for i in range(k_steps):
                if i + 1 < k_steps:
                    issue_h2d(i + 1)
                issue_compute(i)
            stream.wait_stream(d2h_stream)

        run_pipeline(2)   # warm-up: first use of the streams and buffers
        torch.cuda.synchronize(dev)
        in_free = [None] * nbuf
        out_free = [None] * nbuf
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_pipeline(args.steps, e0)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        if not (torch.equal(h_out, out.cpu()) and (h_fin is None or torch.equal(h_fin, fin.cpu()))):
            raise SystemExit("end-to-end outputs differ from the device-timed ones")
        e2e = {"value": whole_job_rate(tokens, world, args.steps, e2e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipeline": "double-buffered: step i+1's inputs copied while step i computes"}
        del host, dev_in, outs, fins
    if kda.check_device_error(ws, dev):
        raise SystemExit("device error flags set during the timed steps")

    hbm_gbs, bf16_tf, peak_kind = load_peaks()
    nbytes = compulsory_bytes(w)
    flops = w.token_heads * FLOPS_PER_TOKEN_HEAD
    fwd_mean = statistics.mean(fwd_ms)
    achieved = nbytes / (fwd_mean / 1000.0) / 1e9
    step_s = ms_per_step / 1000.0
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": measured_traffic(w.name),
                "kernel": "kda_chain_kernel (forward runs: the first chain launch)",
                "peak_source": "measured, MEASURED_PEAKS.json hbm_gbs" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": nbytes,
                "step_frac": (nbytes / step_s / 1e9) / hbm_gbs,
                "step_tflops": flops / step_s / 1e12,
                "step_tflops_frac_of_bf16_peak": flops / step_s / 1e12 / bf16_tf,
                "phase_ms": {"schedule": statistics.mean(sch_ms), "forward": fwd_mean,
                             "compose_and_correct": statistics.mean(cmp_ms)}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_cpu = {n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
        v, threads, desc, _ = cpu_oracle_sample(w, x_cpu, budget_s=15.0)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config_dict(w, {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                          "l2": "flushed between timed steps (252 MB write)",
                                          "launch": launch_mode}),
                "roofline": roofline, "cpu_baseline": cpu,
                "clocks": clocks.summary(), "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps,
                "tflops": flops / step_s / 1e12, "hbm_gbs": nbytes / step_s / 1e9,
                "wall_s": t_wall}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_decode(args, w):
    """The recurrent decode step (kda_decode): every call reads and writes each
    (sequence, head) state once; timed per call with CUDA events."""
    import torch

    from gated_delta_rule_51_gb300 import inputs as I
    from gated_delta_rule_51_gb300 import kda

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    kda.load_library()
    x = I.make_inputs(w, device=dev)
    state = x["initial_state"].clone()
    out = torch.empty_like(x["v"])
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(xx):
        kda.decode(xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], xx["scale"], out, xx["A_log"],
                   xx["dt_bias"], xx["lower_bound"], state)

    for _ in range(args.warmup):
        step(x)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            step(x)
            e1.record(stream)
        torch.cuda.synchronize(dev)
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world, dev)
    tokens = w.B * w.T
    value = whole_job_rate(tokens, world, args.steps, total_ms)
    ms = total_ms / args.steps
    state_bytes = w.B * w.H * 128 * 128 * (4 if w.state_dtype == torch.float32 else 2) * 2
    nbytes = state_bytes + w.token_heads * BYTES_PER_TOKEN_HEAD + w.H * (4 + 128 * 4)
    hbm_gbs, _, peak_kind = load_peaks()
    achieved = nbytes / (ms / 1000.0) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
                "traffic": measured_traffic(w.name), "kernel": "kda_decode_kernel",
                "peak_source": "measured, MEASURED_PEAKS.json hbm_gbs" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": nbytes}

    # end to end: every step copies its tokens host -> device and reads its outputs back;
    # pipelined as in the forward's end-to-end run (two input and output buffer sets), while
    # the states stay resident and are updated in order on the compute stream
    e2e = None
    if not args.no_e2e:
        names = ("q", "k", "v", "g", "beta")
        host = {n: x[n].cpu().pin_memory() for n in names}
        nbuf = 2
        dev_in = []
        for _ in range(nbuf):
            d = dict(x)
            d.update({n: torch.empty_like(x[n]) for n in names})
            dev_in.append(d)
        outs = [torch.empty_like(out) for _ in range(nbuf)]
        h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = sum(host[n].numel() * host[n].element_size() for n in names)
        d2h = h_out.numel() * h_out.element_size()
        h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_free, out_free, in_ready = [None] * nbuf, [None] * nbuf, [None] * nbuf

        def issue_h2d(i):
            b = i % nbuf
            if in_free[b] is not None:
                h2d_stream.wait_event(in_free[b])
            with torch.cuda.stream(h2d_stream):
                for n in names:
                    dev_in[b][n].copy_(host[n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(h2d_stream)
            in_ready[b] = ev

        def issue_compute(i):
            b = i % nbuf
            stream.wait_event(in_ready[b])
            if out_free[b] is not None:
                stream.wait_event(out_free[b])
            d = dev_in[b]
            kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], outs[b], d["A_log"], d["dt_bias"],
                       d["lower_bound"], state, stream=stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            in_free[b] = ev
            d2h_stream.wait_event(ev)
            with torch.cuda.stream(d2h_stream):
                h_out.copy_(outs[b], non_blocking=True)
            ev2 = torch.cuda.Event()
            ev2.record(d2h_stream)
            out_free[b] = ev2

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        issue_h2d(0)
        for i in range(args.steps):
            if i + 1 < args.steps:
                issue_h2d(i + 1)
            issue_compute(i)
        stream.wait_stream(d2h_stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e = {"value": whole_job_rate(tokens, world, args.steps, e2e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "note": "states stay resident on the device between steps",
               "pipeline": "double-buffered: step i+1's tokens copied while step i computes"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_cpu = {n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
        v, threads, desc, _ = cpu_oracle_sample(w, x_cpu, budget_s=15.0)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc}
    if rank == 0:
        line = {"metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": config_dict(w, {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                          "l2": "flushed between timed steps (252 MB write); states 4x L2"}),
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks.summary(), "e2e": e2e,
                "gpu_launches": args.steps}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_bwd(args, w):
    """The backward pass (kda_bwd) on workload w, with random bf16 dout and fp32 dfinal:
    every step reads the forward's inputs and writes every gradient; CUDA events around
    each phase (chunked form: the runs' list, the two chains, the state products, the chunk
    gradients; recurrent form: prep, stored-state forward, reverse, chain rule)."""
    import torch

    from gated_delta_rule_51_gb300 import inputs as I
    from gated_delta_rule_51_gb300 import kda

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    kda.load_library()
    x = I.make_inputs(w, device=dev)
    dout, dfinal = bwd_upstream_grads(w, dev, torch.Generator(device=dev).manual_seed(w.seed + 100))
    shape = kda.make_shape(w.B, w.T, w.H, w.N)
    ws = torch.empty(kda.bwd_workspace_size(shape), dtype=torch.uint8, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    B, T, H = w.B, w.T, w.H
    outs = dict(dq=torch.empty((B, T, H, 128), **f32), dk=torch.empty((B, T, H, 128), **f32),
                dv=torch.empty((B, T, H, 128), **f32), dg=torch.empty((B, T, H, 128), **f32),
                dbeta=torch.empty((B, T, H), **f32), dh0=torch.empty((w.N, H, 128, 128), **f32),
                dA_log=torch.empty((H,), **f32), ddt_bias=torch.empty((H, 128), **f32))
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    recurrent = args.bwd_form == "recurrent"

    def step():
        kda.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["A_log"], x["dt_bias"],
                x["lower_bound"], dout, initial_state=x["initial_state"], dfinal=dfinal,
                cu_seqlens=x["cu_seqlens"], workspace=ws, out=outs, recurrent=recurrent)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if kda.check_device_error(ws, dev):
        raise SystemExit("device error flags set during warm-up")
    launches = kda.last_launch_count()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for e in ev:
        for t in e:
            t.record(stream)        # creates the events before their handles are handed out
    torch.cuda.synchronize(dev)
    # each step is one kda_bwd captured in a CUDA graph (as a training loop would run it), so
    # the host-side argument handling does not sit between the GPU's steps
    graphs, launch_mode = capture_steps(torch, dev, stream, kda, step, ev, args.steps)
    with ClockSampler(dev.index) as clocks:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            if graphs:
                graphs[i].replay()
            else:
                kda.set_profile_events(ev[i][1:])
                step()
        kda.set_profile_events(None)
        torch.cuda.synchronize(dev)
    step_ms = [e[0].elapsed_time(e[4]) for e in ev]
    names = (("prep", "stored_state_forward", "reverse", "chain_rule") if recurrent
             else ("runs", "chains", "state_products", "chunk_gradients"))
    ph = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) for j, name in enumerate(names)}
    dominant = "reverse" if recurrent else "chains"
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms = total_ms / args.steps
    tokens = w.B * w.T
    value = whole_job_rate(tokens, world, args.steps, total_ms)
    state_bytes = w.N * w.H * 128 * 128 * 4 * (int(w.has_initial_state) + 2)   # h0 and dfinal in, dh0 out
    nbytes = w.token_heads * BWD_BYTES_PER_TOKEN_HEAD + state_bytes + 2 * w.H * (4 + 128 * 4)
    hbm_gbs, _, peak_kind = load_peaks()
    achieved = nbytes / (ph[dominant] / 1000.0) / 1e9
    kernel = "kda_bwd_reverse_kernel" if recurrent else "kda_chain_kernel<64> (forward and reverse chains)"
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
                "traffic": measured_traffic(("bwd_" if recurrent else "bwd_chunked_") + w.name), "kernel": kernel,
                "peak_source": "measured, MEASURED_PEAKS.json hbm_gbs" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": nbytes,
                "step_frac": (nbytes / (ms / 1000.0) / 1e9) / hbm_gbs, "phase_ms": ph}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_cpu = {n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
        v, threads, desc, _ = bwd_oracle_sample(w, x_cpu, dout.cpu(), dfinal.cpu())
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc}
    if rank == 0:
        line = {"metric": BWD_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32" if recurrent else "bf16", "data": "synthetic",
                "config": config_dict(w, {"pass": "backward", "form": args.bwd_form,
                                          "dout": "bf16 N(0,1)", "dfinal": "fp32 0.1 N(0,1)",
                                          "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                          "l2": "flushed between timed steps (252 MB write)",
                                          "launch": launch_mode}),
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks.summary(), "e2e": None,
                "gpu_launches": launches * args.steps}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bwd-form", choices=("chunked", "recurrent"), default="chunked",
                    help="backward configs: the chunked tensor-core form (the library's default for the "
                         "gate with a lower bound) or the fp32 recurrent one")
    args = ap.parse_args()
    if args.config.startswith("bwd"):
        # the backward pass on a forward workload: "bwd" is the fixed batch, "bwd_<name>" any other
        name = args.config[4:] if args.config.startswith("bwd_") else "fixed"
        (run_bwd_reference if args.impl == "reference" else run_bwd)(args, workload(name))
        return
    w = workload(args.config)
    if args.impl == "reference":
        run_reference(args, w)
    elif w.name.startswith("decode"):
        run_decode(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
