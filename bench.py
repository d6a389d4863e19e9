#!/usr/bin/env python
"""Throughput of exact attention (forward + backward) on GB300.

One step = the whole hot path on one batch: fa_fwd (forward kernel, causal
tile skip, O and LSE) followed by fa_bwd (D preprocess, dK/dV kernel, dQ
kernel) on B=2, H=16, N=4096, d=128, causal, seeded N(0,1) bf16 inputs.
Throughput counts 4*B*H*N^2*d forward FLOPs (halved for causal) plus 2.5x
that for the backward pass.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 each rank (one per GPU) runs its own heads of a batch N times
larger (weak scaling; no data-path collective).  Started without a
torch.distributed environment, ``--gpus N`` launches the N ranks itself
through torch.distributed.run; under torchrun it joins the ranks it was
started with.  Rank 0 prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle instead, on a
bounded sample of the same workload, on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s at 1 GB300 and fraction of dense BF16 tensor peak"
WORKLOAD = dict(B=2, H=16, N=4096, d=128, causal=True)
STEP_WORKLOAD = "fwd+bwd B=2 H=16 N=4096 d=128 causal"
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The library's launch counters by id (FA_KERNEL_*), named for the kernels
# that id launches at head dim 128: the dK/dV id runs the CTA-pair kernel.
KERNEL_NAMES = ["fa_fwd_kernel", "fa_combine_kernel", "fa_bwd_preprocess", "fa_bwd_dkdv_pair_kernel",
                "fa_bwd_dq_kernel"]


def workload_flops(B, H, N, d, causal):
    from exact_attention_92_gb300 import inputs

    f = inputs.fwd_flops(B, H, N, d, causal)
    return f, inputs.bwd_flops(B, H, N, d, causal)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "fa_fwd_kernel": ["fa_fwd.cu", "sm103_primitives.cuh", "fa_common.h"],
    "fa_fwd256_kernel": ["fa_fwd256.cu", "sm103_primitives.cuh", "fa_common.h"],
    "fa_combine_kernel": ["fa_fwd.cu", "sm103_primitives.cuh", "fa_common.h"],
    "fa_bwd_dkdv_kernel": ["fa_bwd.cu", "bwd_elementwise.cuh", "sm103_primitives.cuh", "fa_common.h"],
    "fa_bwd_dkdv_pair_kernel": ["fa_bwd_pair.cu", "bwd_elementwise.cuh", "sm103_pair.cuh", "sm103_primitives.cuh",
                                "fa_common.h"],
    "fa_bwd_preprocess": ["fa_bwd.cu", "bwd_elementwise.cuh", "sm103_primitives.cuh", "fa_common.h"],
    "fa_bwd_dq_kernel": ["fa_bwd.cu", "bwd_elementwise.cuh", "sm103_primitives.cuh", "fa_common.h"],
}


# C/C++ comments and string/char literals (literals are kept as they are).
_C_TOKENS = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'', re.S)


def _code_only(text):
    """Source text without comments and blank lines: what the compiler sees."""
    text = _C_TOKENS.sub(lambda m: "" if m.group(0).startswith("/") else m.group(0), text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel):
    """Hash of the code (comments left out) of the source files a kernel is
    compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_92_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as fh:
            h.update(name.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary,
    if it was taken on the kernel's current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    # Only a capture of the step's own workload describes this launch.
    if not str(ent.get("workload", "")).startswith(STEP_WORKLOAD):
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[4]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        load = [r for r in rows if r[2] >= 50.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(load)}


# -------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max_sum(world, maxes, sums, device):
    """Max over ranks of ``maxes`` and sum over ranks of ``sums`` (lists of floats)."""
    if world == 1:
        return list(maxes), list(sums)
    import torch
    import torch.distributed as dist

    a = torch.tensor(maxes, dtype=torch.float64, device=device)
    b = torch.tensor(sums, dtype=torch.float64, device=device)
    dist.all_reduce(a, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return a.tolist(), b.tolist()


def shard_heads(B, H, world, rank):
    """Weak scaling: the job is ``world`` batches of B x H heads; rank r owns
    batch block r (its own independent heads, no exchange between ranks)."""
    return dict(batch_offset=rank * B, B=B, H=H, seed=5000 + rank)


# ---------------------------------------------------------------- the oracle

def oracle_sample(max_seconds=10.0, max_heads=4, n_tokens=None):
    """Time the fp64 oracle's forward + backward on whole heads of the
    workload (or on its first ``n_tokens`` tokens).  Returns (TFLOP/s,
    seconds, description)."""
    import numpy as np

    from exact_attention_92_gb300 import inputs
    from oracle import attention as att

    w = WORKLOAD
    N = n_tokens or w["N"]
    case = inputs.make_case(1, max_heads, N, w["d"], w["causal"], seed=5000, with_do=True)
    q, k, v, do = (case.f64(n) for n in ("q", "k", "v", "do"))
    done = 0
    t0 = time.perf_counter()
    for h in range(max_heads):
        att.forward_head(q[0, h], k[0, h], v[0, h], case.scale, w["causal"])
        att.backward_head(q[0, h], k[0, h], v[0, h], do[0, h], case.scale, w["causal"])
        done += 1
        if time.perf_counter() - t0 >= max_seconds:
            break
    dt = time.perf_counter() - t0
    f, b = workload_flops(1, done, N, w["d"], w["causal"])
    desc = f"{done} head(s) x N={N} of the workload (d={w['d']}, causal), fp64 forward + backward"
    return (f + b) / dt / 1e12, dt, desc


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------- our arm

def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import exact_attention_92_gb300 as fa
    from exact_attention_92_gb300 import build, inputs

    build.build()
    fa.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = WORKLOAD
    B, H, N, d, causal = w["B"], w["H"], w["N"], w["d"], w["causal"]
    shard = shard_heads(B, H, world, rank)
    case = inputs.make_case(B, H, N, d, causal, seed=shard["seed"], with_do=True)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    q, k, v, do = (to_dev(x) for x in (case.q, case.k, case.v, case.do))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        fa.fa_fwd(q, k, v, o, lse, causal)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st = fa.fa_poll_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {fa.fa_strerror(st)}")

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    count0 = [fa.fa_launch_count(kid) for kid in range(len(KERNEL_NAMES))]
    for i in range(args.steps):
        flush.zero_()  # L2 flush between steps, outside the step's events
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if rank == 0 else None
    count1 = [fa.fa_launch_count(kid) for kid in range(len(KERNEL_NAMES))]
    st = fa.fa_poll_status()
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {fa.fa_strerror(st)}")
    # Per-launch device times come from a second timed region of the same
    # steps with events around every launch: events between kernels stop a
    # launch from overlapping the previous kernel's drain and lengthen a step
    # by a few percent, so the step time above is taken without them.
    barrier(world)
    torch.cuda.synchronize()
    fa.fa_timing_enable(True)
    for i in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    per_kernel = {}
    for kid, name in enumerate(KERNEL_NAMES):
        n, ms = fa.fa_timing_read(kid)
        per_kernel[name] = {"launches": n, "total_ms": ms}
    fa.fa_timing_enable(False)
    st = fa.fa_poll_status()
    if st != 0:
        raise RuntimeError(f"device status after the per-launch timing steps: {fa.fa_strerror(st)}")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    launches = sum(c1 - c0 for c0, c1 in zip(count0, count1))
    kern_ms = [per_kernel[n]["total_ms"] for n in KERNEL_NAMES]
    (total_ms_max, *kern_max), (launches_sum,) = reduce_max_sum(world, [total_ms] + kern_ms, [launches], device)

    f, b = workload_flops(B, H, N, d, causal)
    step_flops_job = (f + b) * world
    value = step_flops_job * args.steps / (total_ms_max / 1e3) / 1e12

    # Dominant kernel and its roofline (tensor-bound: QK^T, PV, and the
    # backward's five GEMMs are dense contractions).
    dom = max(KERNEL_NAMES, key=lambda n: per_kernel[n]["total_ms"])
    dom_ms = kern_max[KERNEL_NAMES.index(dom)] / max(1, per_kernel[dom]["launches"])
    # Algorithmic FLOPs per kernel: the backward's 2.5 F splits into the
    # dK/dV kernel's S, dP, dV and dK products (2 F) and the dQ product
    # (0.5 F); the dQ kernel's recomputed S and dP are not counted.
    dom_flops = {"fa_fwd_kernel": f, "fa_bwd_dkdv_pair_kernel": 0.8 * b, "fa_bwd_dq_kernel": 0.2 * b}.get(dom)
    peaks, peak_src = load_peaks()
    roofline = None
    if dom_flops is not None:
        achieved = dom_flops / (dom_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": recorded_traffic(dom),
                    "peak_source": f"{peak_src} bf16 dense, burst (kernel timed per launch)",
                    "ms_per_launch": round(dom_ms, 4)}

    # End to end: pinned host inputs -> device, forward + backward through the
    # C ABI, gradients -> pinned host, every step.
    e2e = e2e_run(args, fa, case, device, stream, B, H, N, d, causal, f + b, world)

    # Secondary workloads, each with its own clock record (they follow one
    # another without pauses, so a power-capped stretch shows up here).
    target_clocks = {}

    def sampled(name, fn):
        if rank != 0 or args.no_extra:
            return None
        cs = ClockSampler(local)
        cs.start()
        try:
            return fn(fa, device, peaks, args)
        finally:
            target_clocks[name] = cs.stop()

    extra = sampled("fwd_targets", fwd_targets)
    extra_bwd = sampled("bwd_targets", bwd_targets)
    extra_gqa = sampled("gqa_targets", gqa_targets)
    extra_short = sampled("short_targets", short_targets)
    extra_general = sampled("general_targets", general_targets)

    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms_max / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 Q, K, V, dO",
        "config": {"workload": f"fwd+bwd B={B} H={H} N={N} d={d} causal (per GPU)", "B": B * world, "H": H,
                   "N": N, "d": d, "causal": causal,
                   "l2": "flushed between steps (256 MiB write, outside the step events)",
                   "parallelism": f"{world} GPU(s), independent heads per GPU, no collective"},
        "frac_of_peak": round(value / world / peaks["bf16_tflops"], 4),
        "roofline": roofline,
        "kernels": {n: {"launches": v["launches"], "ms_per_launch": round(v["total_ms"] / v["launches"], 4)}
                    for n, v in per_kernel.items() if v["launches"]},
        "kernel_timing": ("per-launch CUDA events in a second timed region of the same steps; the step time "
                          "comes from a region without them"),
        "gpu_launches": int(launches_sum),
        "e2e": e2e,
        "clocks": clk,
    }
    if extra is not None:
        line["fwd_targets"] = extra
    if extra_bwd is not None:
        line["bwd_targets"] = extra_bwd
    if extra_gqa is not None:
        line["gqa_targets"] = extra_gqa
    if extra_short is not None:
        line["short_targets"] = extra_short
    if extra_general is not None:
        line["general_targets"] = extra_general
    if target_clocks:
        line["target_clocks"] = target_clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, dt, desc = oracle_sample()
        line["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                                "sample": f"{desc}; {dt:.1f} s; numpy default BLAS threading"}
    return line


def e2e_run(args, fa, case, device, stream, B, H, N, d, causal, flops, world, nbuf=2):
    """Steps from pinned host memory to pinned host memory through the C ABI:
    every step copies Q, K, V, dO host -> device, runs fa_fwd + fa_bwd and
    copies dQ, dK, dV device -> host.  As a training input pipeline would,
    the copies run on their own streams into ``nbuf`` sets of buffers, so the
    next steps' inputs and the previous steps' gradients move while a step
    computes (CUDA events order each buffer's copy-in, compute and copy-out).
    The timed region covers all K steps' copies and compute."""
    import numpy as np
    import torch

    def pinned(bits):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    shape = (B, H, N, d)
    h_in = [pinned(x) for x in (case.q, case.k, case.v, case.do)]
    h_out = [[torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)] for _ in range(nbuf)]
    d_in = [[torch.empty(shape, dtype=torch.bfloat16, device=device) for _ in range(4)] for _ in range(nbuf)]
    d_out = [[torch.empty(shape, dtype=torch.bfloat16, device=device) for _ in range(3)] for _ in range(nbuf)]
    o = [torch.empty(shape, dtype=torch.bfloat16, device=device) for _ in range(nbuf)]
    lse = [torch.empty(shape[:3], dtype=torch.float32, device=device) for _ in range(nbuf)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    copied_in = [torch.cuda.Event() for _ in range(nbuf)]
    computed = [torch.cuda.Event() for _ in range(nbuf)]
    copied_out = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf

    def step(i):
        b = i % nbuf
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(computed[b])  # step i-nbuf no longer reads these inputs
            for dst, src in zip(d_in[b], h_in):
                dst.copy_(src, non_blocking=True)
            copied_in[b].record(s_in)
        stream.wait_event(copied_in[b])
        if used[b]:
            stream.wait_event(copied_out[b])  # step i-nbuf's gradients have left these buffers
        q, k, v, do = d_in[b]
        dq, dk, dv = d_out[b]
        fa.fa_fwd(q, k, v, o[b], lse[b], causal, stream=stream)
        fa.fa_bwd(q, k, v, o[b], lse[b], do, dq, dk, dv, causal, stream=stream)
        computed[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[b])
            for dst, src in zip(h_out[b], d_out[b]):
                dst.copy_(src, non_blocking=True)
            copied_out[b].record(s_out)
        used[b] = True

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    n = max(1, args.steps)
    barrier(world)
    a.record(stream)
    s_in.wait_event(a)  # the first copy-in starts inside the timed region
    for i in range(n):
        step(i)
    stream.wait_stream(s_out)  # the last copy-out ends inside the timed region
    stream.wait_stream(s_in)
    e.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e)
    (ms_max,), _ = reduce_max_sum(world, [ms], [0.0], device)
    elem = B * H * N * d * 2
    return {"value": round(flops * world * n / (ms_max / 1e3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": 4 * elem, "d2h_bytes_per_step": 3 * elem,
            "ms_per_step": round(ms_max / n, 4),
            "copies": f"pinned host buffers; copy-in, compute and copy-out on three streams, {nbuf} buffer sets"}


def bwd_targets(fa, device, peaks, args):
    """Backward-only throughput (fa_bwd: D preprocess, dQ and dK/dV kernels)
    on the 16K-token sweep at d=128, N >= 4K; 2.5x the forward FLOPs."""
    import torch

    from exact_attention_92_gb300 import inputs

    out = []
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for N in (4096, 8192, 16384):
        for causal in (False, True):
            B, H, d = 16384 // N, 16, 128
            g = torch.Generator(device=device)
            g.manual_seed(5000)
            shape = (B, H, N, d)
            q, k, v, do = (torch.randn(shape, generator=g, device=device).to(torch.bfloat16) for _ in range(4))
            o = torch.empty_like(q)
            lse = torch.empty(shape[:3], dtype=torch.float32, device=device)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            fa.fa_fwd(q, k, v, o, lse, causal)
            for _ in range(3):
                fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal)
            torch.cuda.synchronize()
            # All repetitions are queued before one synchronise, so the host's
            # enqueue time never shows inside the events.
            reps = 10
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for s, e in ev:
                flush.zero_()
                s.record(stream)
                fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal)
                e.record(stream)
            torch.cuda.synchronize()
            tot = sum(s.elapsed_time(e) for s, e in ev)
            st = fa.fa_poll_status()
            if st != 0:
                raise RuntimeError(f"device status after the backward cases: {fa.fa_strerror(st)}")
            fl = 2.5 * inputs.fwd_flops(B, H, N, d, causal)
            tf = fl * reps / (tot / 1e3) / 1e12
            out.append({"case": f"B={B} H={H} N={N} d={d} {'causal' if causal else 'non-causal'}",
                        "tflops": round(tf, 1), "frac": round(tf / peaks["bf16_tflops"], 4),
                        "ms": round(tot / reps, 4)})
            del q, k, v, do, o, lse, dq, dk, dv
    return out


def short_targets(fa, device, peaks, args):
    """The short-sequence half of the sweep, where the data, not the tensor
    cores, bound the time: the single head B=1 H=1 N=128 d=64 (launch
    latency, microseconds per call), B=4 H=16 N=1024 d=64, and the 16K-token
    sweep at d=64 (every N) and at d=128 for N <= 2048.  Each case reports the
    forward's TFLOP/s and its algorithmic HBM bytes per second (Q, K, V read
    and O written as bf16, LSE as fp32) against the measured copy bandwidth;
    the N=1024 d=64 and N=512 cases also time the backward (Q, K, V, O, dO
    read, dQ, dK, dV written as bf16, LSE and D as fp32)."""
    import torch

    from exact_attention_92_gb300 import inputs

    cases = [(1, 1, 128, 64), (4, 16, 1024, 64)]
    for d in (64, 128):
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            if d == 128 and N > 2048:
                continue
            cases.append((16384 // N, 2048 // d, N, d))
    with_bwd = {(4, 16, 1024, 64), (32, 32, 512, 64), (32, 16, 512, 128)}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    hbm = peaks["hbm_gbs"]
    out = []

    def timed(fn, reps=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for st, en in ev:  # queued before one synchronise (host time stays out)
            flush.zero_()
            st.record(stream)
            fn()
            en.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / reps

    for (B, H, N, d) in cases:
        for causal in (False, True):
            g = torch.Generator(device=device)
            g.manual_seed(3000)
            shape = (B, H, N, d)
            q, k, v, do = (torch.randn(shape, generator=g, device=device).to(torch.bfloat16) for _ in range(4))
            o = torch.empty_like(q)
            lse = torch.empty(shape[:3], dtype=torch.float32, device=device)
            ms = timed(lambda: fa.fa_fwd(q, k, v, o, lse, causal))
            fl = inputs.fwd_flops(B, H, N, d, causal)
            nbytes = 8 * B * H * N * d + 4 * B * H * N
            gbs = nbytes / ms / 1e6
            rec = {"case": f"B={B} H={H} N={N} d={d} {'causal' if causal else 'non-causal'} forward",
                   "us": round(ms * 1e3, 2), "tflops": round(fl / ms / 1e9, 1),
                   "frac_tensor": round(fl / ms / 1e9 / peaks["bf16_tflops"], 4),
                   "hbm_gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4), "bytes": nbytes}
            out.append(rec)
            if (B, H, N, d) in with_bwd:
                dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
                ms_b = timed(lambda: fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal))
                nb = 16 * B * H * N * d + 8 * B * H * N
                gb = nb / ms_b / 1e6
                out.append({"case": f"B={B} H={H} N={N} d={d} {'causal' if causal else 'non-causal'} backward",
                            "us": round(ms_b * 1e3, 2), "tflops": round(2.5 * fl / ms_b / 1e9, 1),
                            "frac_tensor": round(2.5 * fl / ms_b / 1e9 / peaks["bf16_tflops"], 4),
                            "hbm_gbs": round(gb, 1), "frac_hbm": round(gb / hbm, 4), "bytes": nb})
                del dq, dk, dv
            del q, k, v, do, o, lse
    st = fa.fa_poll_status()
    if st != 0:
        raise RuntimeError(f"device status after the short-sequence cases: {fa.fa_strerror(st)}")
    return out


def visible_pairs(Nq, Nk, causal, align):
    """(query, key) pairs the mask lets through, per head."""
    if not causal:
        return Nq * Nk
    off = 0 if align == "top_left" else Nk - Nq
    # row i sees min(Nk, max(0, i + off + 1)) keys
    tot = 0
    for i in range(Nq):
        tot += min(Nk, max(0, i + off + 1))
    return tot


def general_targets(fa, device, peaks, args):
    """Head dims 96 and 256 (hidden 2016 / 2048 at 16K tokens), and queries
    shorter than the keys with bottom-right causal alignment: a grouped-query
    decode step (one query row per head over 8192 keys, HBM-bound: the K, V
    reads are the traffic) and a 1024-row chunk over 8192 keys.  FLOPs are
    4 d per visible (query, key) pair (2.5x for the backward)."""
    import torch

    cases = [
        # (name, B, H, Hkv, Nq, Nk, d, causal, backward too)
        ("d=96 B=8 H=21 N=2048 non-causal", 8, 21, 21, 2048, 2048, 96, False, True),
        ("d=96 B=8 H=21 N=2048 causal", 8, 21, 21, 2048, 2048, 96, "top_left", True),
        ("d=96 B=4 H=21 N=4096 causal", 4, 21, 21, 4096, 4096, 96, "top_left", True),
        ("d=256 B=4 H=8 N=4096 non-causal", 4, 8, 8, 4096, 4096, 256, False, True),
        ("d=256 B=4 H=8 N=4096 causal", 4, 8, 8, 4096, 4096, 256, "top_left", True),
        ("d=256 B=1 H=8 N=16384 causal", 1, 8, 8, 16384, 16384, 256, "top_left", False),
        ("decode GQA B=8 H=32 Hkv=8 Nq=1 Nk=8192 d=128 bottom-right", 8, 32, 8, 1, 8192, 128, "bottom_right", False),
        ("chunk B=1 H=32 Nq=1024 Nk=8192 d=128 bottom-right", 1, 32, 32, 1024, 8192, 128, "bottom_right", True),
    ]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    out = []

    def timed(fn, reps=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for st, en in ev:  # queued before one synchronise (host time stays out)
            flush.zero_()
            st.record(stream)
            fn()
            en.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / reps

    for name, B, H, Hkv, Nq, Nk, d, causal, bwd in cases:
        g = torch.Generator(device=device)
        g.manual_seed(7000)
        q, do = (torch.randn((B, H, Nq, d), generator=g, device=device).to(torch.bfloat16) for _ in range(2))
        k, v = (torch.randn((B, Hkv, Nk, d), generator=g, device=device).to(torch.bfloat16) for _ in range(2))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=device)
        pairs = B * H * visible_pairs(Nq, Nk, bool(causal), causal if causal else "top_left")
        fl = 4.0 * d * pairs
        ms = timed(lambda: fa.fa_fwd_general(q, k, v, o, lse, causal))
        nbytes = 2 * d * (2 * B * H * Nq + 2 * B * Hkv * Nk) + 4 * B * H * Nq
        gbs = nbytes / ms / 1e6
        out.append({"case": name + " forward", "us": round(ms * 1e3, 2), "tflops": round(fl / ms / 1e9, 1),
                    "frac_tensor": round(fl / ms / 1e9 / peaks["bf16_tflops"], 4), "hbm_gbs": round(gbs, 1),
                    "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)})
        if bwd:
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ms_b = timed(lambda: fa.fa_bwd_general(q, k, v, o, lse, do, dq, dk, dv, causal))
            out.append({"case": name + " backward", "us": round(ms_b * 1e3, 2),
                        "tflops": round(2.5 * fl / ms_b / 1e9, 1),
                        "frac_tensor": round(2.5 * fl / ms_b / 1e9 / peaks["bf16_tflops"], 4)})
            del dq, dk, dv
        del q, k, v, do, o, lse
    st = fa.fa_poll_status()
    if st != 0:
        raise RuntimeError(f"device status after the general cases: {fa.fa_strerror(st)}")
    return out


def gqa_targets(fa, device, peaks, args):
    """Grouped-query attention (fa_fwd_gqa, fa_bwd_gqa): 32 query heads over 8
    key/value heads, B=2, N=4096, d=128, causal; FLOPs counted per query head
    as for multi-head attention."""
    import torch

    from exact_attention_92_gb300 import inputs

    B, H, Hkv, N, d, causal = 2, 32, 8, 4096, 128, True
    g = torch.Generator(device=device)
    g.manual_seed(6000)
    q, do = (torch.randn((B, H, N, d), generator=g, device=device).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn((B, Hkv, N, d), generator=g, device=device).to(torch.bfloat16) for _ in range(2))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def timed(fn, reps=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for s, e in ev:  # queued before one synchronise (host time stays out)
            flush.zero_()
            s.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return sum(s.elapsed_time(e) for s, e in ev) / reps

    ms_f = timed(lambda: fa.fa_fwd_gqa(q, k, v, o, lse, causal))
    ms_b = timed(lambda: fa.fa_bwd_gqa(q, k, v, o, lse, do, dq, dk, dv, causal))
    st = fa.fa_poll_status()
    if st != 0:
        raise RuntimeError(f"device status after the GQA cases: {fa.fa_strerror(st)}")
    f = inputs.fwd_flops(B, H, N, d, causal)
    name = f"B={B} H={H} Hkv={Hkv} N={N} d={d} causal"
    return [{"case": name + " forward", "tflops": round(f / ms_f / 1e9, 1),
             "frac": round(f / ms_f / 1e9 / peaks["bf16_tflops"], 4), "ms": round(ms_f, 4)},
            {"case": name + " backward", "tflops": round(2.5 * f / ms_b / 1e9, 1),
             "frac": round(2.5 * f / ms_b / 1e9 / peaks["bf16_tflops"], 4), "ms": round(ms_b, 4)}]


def fwd_targets(fa, device, peaks, args):
    """Forward-only throughput on the long-sequence, d=128 problems."""
    import torch

    from exact_attention_92_gb300 import inputs

    cases = [("GPT layer B=8 H=32 N=4096 d=128 causal, Q,K ~ N(0,3^2)", dict(B=8, H=32, N=4096, d=128, causal=True),
              3.0)]
    # The 16K-token sweep at d=128 (hidden 2048), N >= 4K.
    for N in (4096, 8192, 16384):
        for causal in (False, True):
            cases.append((f"B={16384 // N} H=16 N={N} d=128 {'causal' if causal else 'non-causal'}",
                          dict(B=16384 // N, H=16, N=N, d=128, causal=causal), 1.0))
    cases.append(("B=1 H=1 N=65536 d=128 causal, split-KV", dict(B=1, H=1, N=65536, d=128, causal=True), 1.0))
    cases.append(("B=1 H=1 N=65536 d=128 non-causal, split-KV", dict(B=1, H=1, N=65536, d=128, causal=False), 1.0))
    out = []
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for name, c, qk_std in cases:
        g = torch.Generator(device=device)
        g.manual_seed(4000)
        shape = (c["B"], c["H"], c["N"], c["d"])
        q = (torch.randn(shape, generator=g, device=device) * qk_std).to(torch.bfloat16)
        k = (torch.randn(shape, generator=g, device=device) * qk_std).to(torch.bfloat16)
        v = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty(shape[:3], dtype=torch.float32, device=device)
        for _ in range(3):
            fa.fa_fwd(q, k, v, o, lse, c["causal"])
        torch.cuda.synchronize()
        reps = 10
        fa.fa_timing_enable(True)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for s, e in ev:  # queued before one synchronise (host time stays out)
            flush.zero_()
            s.record(stream)
            fa.fa_fwd(q, k, v, o, lse, c["causal"])
            e.record(stream)
        torch.cuda.synchronize()
        tot = sum(s.elapsed_time(e) for s, e in ev)
        nk, kms = fa.fa_timing_read(0)
        for kid in range(1, 5):
            fa.fa_timing_read(kid)
        fa.fa_timing_enable(False)
        fl = inputs.fwd_flops(c["B"], c["H"], c["N"], c["d"], c["causal"])
        tf = fl * reps / (tot / 1e3) / 1e12
        ktf = fl * nk / (kms / 1e3) / 1e12 if nk else None
        out.append({"case": name, "tflops": round(tf, 1), "frac": round(tf / peaks["bf16_tflops"], 4),
                    "fwd_kernel_tflops": round(ktf, 1) if ktf else None, "ms": round(tot / reps, 4)})
        del q, k, v, o, lse
    return out


# ----------------------------------------------------------- ncu captures

def run_profile(case):
    """Two warm-up launches, then one launch, of the forward kernel on the GPT
    layer (B=8 H=32 N=4096 d=128 causal), on B=4 H=16 N=1024 d=64
    non-causal (``fwd_short``, 33.6 MB: the DRAM figures there are those of
    a problem below the L2 size), on B=4 H=32 N=4096 d=64 non-causal
    (``fwd64``, 268 MB) or on B=4 H=8 N=4096 d=256 causal
    (``fwd256``); of the split-KV forward and its merge on one head of 65536
    tokens (``splitkv``); or of the backward on the fwd+bwd workload; for
    ``ncu -s 2 -c 1`` captures."""
    import torch

    import exact_attention_92_gb300 as fa
    from exact_attention_92_gb300 import build

    build.build()
    # Replayed passes of a profiler can stretch a launch far beyond its normal
    # length; give the bounded device waits room so they do not give up.
    fa.fa_set_wait_timeout_ns(60_000_000_000)
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    if case == "fwd":
        shape, causal = (8, 32, 4096, 128), True
    elif case == "fwd_short":
        shape, causal = (4, 16, 1024, 64), False
    elif case == "fwd64":
        shape, causal = (4, 32, 4096, 64), False
    elif case == "splitkv":
        shape, causal = (1, 1, 65536, 128), True
    elif case in ("fwd256", "bwd256"):
        shape, causal = (4, 8, 4096, 256), True
    elif case == "decode":
        shape, causal = (8, 32, 1, 128), "bottom_right"
    else:
        w = WORKLOAD
        shape, causal = (w["B"], w["H"], w["N"], w["d"]), w["causal"]
    q, k, v, do = (torch.randn(shape, generator=g, device=dev).to(torch.bfloat16) for _ in range(4))
    if case == "decode":  # one query row per head over 8192 keys of 8 key/value heads
        k, v = (torch.randn((8, 8, 8192, 128), generator=g, device=dev).to(torch.bfloat16) for _ in range(2))
    if case == "fwd":  # the GPT layer's peaky logits: Q, K ~ N(0, 3^2)
        q, k = (q.float() * 3.0).to(torch.bfloat16), (k.float() * 3.0).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    if case in ("bwd", "bwd256"):
        fa.fa_fwd(q, k, v, o, lse, causal)
    for _ in range(3):
        if case in ("fwd", "fwd_short", "fwd64", "fwd256"):
            fa.fa_fwd_ex(q, k, v, o, lse, causal, None, 1)
        elif case == "splitkv":
            fa.fa_fwd(q, k, v, o, lse, causal)
        elif case == "decode":
            fa.fa_fwd_general(q, k, v, o, lse, causal)
        else:
            fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal)
    torch.cuda.synchronize()
    st = fa.fa_poll_status()
    print(json.dumps({"profile": case, "shape": list(shape), "causal": causal, "status": st}))
    if st != 0:
        raise SystemExit(1)


# ----------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    """The oracle as it stands, on host cores: each step is a bounded sample
    of the workload (one head, the first 1024 tokens, forward + backward)."""
    if rank != 0:
        return None
    for _ in range(args.warmup):
        oracle_sample(max_seconds=0.0, max_heads=1, n_tokens=1024)
    tot = 0.0
    flops = 0.0
    desc = ""
    for _ in range(args.steps):
        tf, dt, desc = oracle_sample(max_seconds=0.0, max_heads=1, n_tokens=1024)
        tot += dt
        flops += tf * 1e12 * dt
    value = flops / tot / 1e12
    w = WORKLOAD
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: seeded N(0,1) bf16 Q, K, V, dO (upcast to f64)",
        "config": {"workload": f"fwd+bwd B={w['B']} H={w['H']} N={w['N']} d={w['d']} causal (per GPU)",
                   "B": w["B"], "H": w["H"], "N": w["N"], "d": w["d"], "causal": w["causal"],
                   "parallelism": "CPU oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def free_port():
    import socket

    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_ranks(n, argv):
    """Run this script as ``n`` ranks on this node (torch.distributed.run,
    rendezvous on 127.0.0.1) with the same arguments; returns the launcher's
    exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the forward-only and backward-only target cases")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle")
    ap.add_argument("--profile", choices=["fwd", "fwd_short", "fwd64", "splitkv", "fwd256", "decode", "bwd", "bwd256"],
                    help="3 launches of one kernel (or of the split-KV forward and its merge), for ncu")
    args = ap.parse_args(argv)
    if args.profile:
        run_profile(args.profile)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        raise SystemExit(launch_ranks(args.gpus, sys.argv[1:] if argv is None else list(argv)))
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
