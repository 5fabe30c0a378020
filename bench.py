#!/usr/bin/env python3
"""Benchmark of the fused post-backward ZeRO step (ring reduce-scatter + unscale + overflow check +
AdamW + cast + all-gather write) on GB300.

Default workload: the 1.3B transformer shapes (145 tensors, 1,311,080,448 params, 33 buckets of at
most 50M params), W = 8 emulated workers, bf16 gradients and parameters, ZeRO-3 memory plan. One step
is one launch of the fused kernel over every bucket. Inputs (55 GB read+written per step) are far
larger than the 129 MB L2, so no flush is needed between steps.

Prints one JSON line: Gparams/s (value), the roofline of the fused kernel against the measured HBM
copy bandwidth, the oracle timed on the host cores (cpu_baseline), and the end-to-end rate through
zr_step_from_host with pinned host gradients (e2e).

--impl reference times the CPU oracle (the only reference this method has) on the same metric.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD_DEFAULT = "7b"
# the other workload held to the HBM target, timed after the default one and reported under its own key
SECOND_DEFAULT = "1p3b"


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The largest value of x over all ranks (x itself when running alone)."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, seconds_max: float, ws: int) -> float:
    """Units processed by all ranks per second of the slowest rank, in billions."""
    return ws * units_per_rank / seconds_max / 1e9


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _traffic_record(workload: str, prefix: str = "fused_step", key: str = "traffic_bytes_per_launch",
                    files=("zr_step_kernel.cuh", "zr_device.cuh")):
    """DRAM bytes of the fused kernel per launch (or of the in-place step's two launches, per step) from the
    committed ncu summary, if the kernel source has not changed since it was taken (the summary records the
    hash of the kernel's source files)."""
    import hashlib
    src = os.path.join(ROOT, "zero_gradient_reduction_gb300", "csrc")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(src, f), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    path = os.path.join(ROOT, "profiles", f"{prefix}_{workload}.md")
    if not os.path.exists(path):
        return None, digest
    rec = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                rec[k.strip()] = v.strip().split()[0].strip("`")
    if rec.get("kernel_source_sha256_16") != digest:
        return None, digest
    try:
        return float(rec[key]), digest
    except Exception:
        return None, digest


class ClockSampler:
    """nvidia-smi clock and throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return out
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        load = [s for s, p in zip(sm, power) if p > 300.0] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        out.update(sm_mhz=statistics.median(load) if load else None, sm_max_mhz=max(mx) if mx else None,
                   reasons=reasons, samples=len(rows), power_w_max=max(power) if power else None)
        return out


def oracle_sample(w, plan_buckets, offsets, seconds_target: float, max_buckets: int = 64, window: int = 0):
    """Time the CPU oracle on whole buckets (window == 0) or on a mini-bucket of `window` elements per ring
    block taken from bucket 0, until about `seconds_target` of oracle time is spent. Returns
    (params processed, oracle seconds, description)."""
    import oracle
    import zrgen
    from zrgen.layout import Layout
    sig = zrgen.sigma_per_tensor(w)
    layout = Layout(w.tensors, offsets, sig, w.seed, w.dtype, w.master_sigma)
    total_params, total_s, used = 0, 0.0, 0
    hyper = oracle.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    for b in range(min(len(plan_buckets), max_buckets)):
        start, n, C = (int(x) for x in plan_buckets[b])
        if window:
            idx = np.concatenate([np.arange(start + c * C, start + c * C + min(window, max(0, n - c * C)))
                                  for c in range(w.W)])
            Cw = window
        else:
            idx = np.arange(start, start + n)
            Cw = C
        lo = idx
        grads = []
        runs = np.flatnonzero(np.diff(lo) != 1) + 1
        for r in range(w.W * w.A):
            g = np.empty(len(lo), np.uint16)
            for seg in np.split(np.arange(len(lo)), runs):
                a, e = int(lo[seg[0]]), int(lo[seg[-1]]) + 1
                g[seg] = layout.grads_host(a, e, 1, r, w.init_scale)
            grads.append(g)
        master = np.empty(len(lo), np.float32)
        for seg in np.split(np.arange(len(lo)), runs):
            a, e = int(lo[seg[0]]), int(lo[seg[-1]]) + 1
            master[seg] = layout.master_host(a, e)
        m = np.zeros(len(lo), np.float32)
        v = np.zeros(len(lo), np.float32)
        p = np.zeros(len(lo), np.uint16)
        sc = oracle.new_scaler(w.init_scale, w.dynamic)
        t0 = time.perf_counter()
        oracle.step(w.W, w.A, w.dtype, np.array([[0, len(lo), Cw]]), grads, master, m, v, p, hyper, sc)
        total_s += time.perf_counter() - t0
        total_params += len(lo)
        used += 1
        if total_s >= seconds_target:
            break
    what = (f"{used} whole bucket(s) of the {w.name} workload ({total_params} params, W={w.W})" if not window else
            f"{used} mini-bucket(s) of {window} params per ring block of the {w.name} workload "
            f"({total_params} params, W={w.W})")
    return total_params, total_s, what


def run_reference(args, w):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return 0
    import oracle
    import zrgen
    oracle.build()
    zrgen.build_host()
    b, offs = oracle.bucket_plan(list(w.tensors), w.cap, w.W)
    # every step: one mini-bucket of 32768 params per ring block, timed on one host core
    for _ in range(args.warmup):
        oracle_sample(w, b, offs, 0.0, max_buckets=1, window=32768)
    params, secs = 0, 0.0
    what = ""
    for _ in range(args.steps):
        p, s, what = oracle_sample(w, b, offs, 0.0, max_buckets=1, window=32768)
        params += p
        secs += s
    value = params / secs / 1e9
    ms = secs / args.steps * 1e3
    line = {
        "impl": "reference", "metric": "fused reduce-scatter+AdamW step Gparams/s", "value": value,
        "unit": "Gparams/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _config(w, b, "oracle on host cores; per step a sample of the workload"),
        "cpu_baseline": {"value": value, "unit": "Gparams/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step: {what}"},
        "e2e": {"value": value, "unit": "Gparams/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(w, buckets, l2_note, launch=None, inplace=False):
    cfg = {"workload": f"{w.name}: {w.description}", "W": w.W, "A": w.A, "stage": w.stage,
           "params": w.n, "buckets": int(len(buckets)), "grad_dtype": "fp16" if w.dtype == 0 else "bf16",
           "state_dtype": "fp32 master/m/v (one set, updated in place)" if inplace else
           "fp32 master/m/v (ping-pong sets)",
           "alg_bytes_per_param": w.alg_bytes_per_param() + (2 * w.W * w.A if inplace else 0), "l2": l2_note,
           "parallelism": "replicas"}
    if launch:
        cfg["launch"] = launch
    return cfg


def measure_overlap(torch, zr, plan, grads, state, hyper, dev, stream, tokens: int = 8192, reps: int = 3,
                    budget_caps=(16, 38, 76, 152, 304), step_bytes=None):
    """Bucketed overlap against a synthetic backward: on a compute stream, bucket b's "backward" is a bf16 GEMM
    of about 4 * tokens * n_b FLOPs (weight and input gradients of n_b parameters), after which an event marks
    the bucket's gradients ready and zr_step_bucket(b) runs on a side stream. Compared with backward followed by
    the one-launch step."""
    K = 2048
    ns = [max(1, int(round(4 * tokens * int(n_b) / (2 * tokens * K)))) for _, n_b, _ in plan.buckets]
    a_mat = torch.randn(tokens, K, device=dev, dtype=torch.bfloat16)
    b_flat = torch.randn(K * max(ns), device=dev, dtype=torch.bfloat16)
    c_flat = torch.empty(tokens * max(ns), device=dev, dtype=torch.bfloat16)
    # the bucket steps get the higher priority, so a ready bucket is scheduled as soon as SMs free up
    # (torch maps an out-of-range priority to the nearest valid one; lower numbers are higher priority)
    compute = torch.cuda.Stream(dev, priority=0)
    side = torch.cuda.Stream(dev, priority=-100)

    def backward(events=None):
        with torch.cuda.stream(compute):
            for b, nb in enumerate(ns):
                torch.matmul(a_mat, b_flat[:K * nb].view(K, nb), out=c_flat[:tokens * nb].view(tokens, nb))
                if events is not None:
                    events[b].record(compute)

    def timed(fn):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / reps * 1e3

    def serial():
        backward()
        stream.wait_stream(compute)
        plan.step(grads, state, hyper, stream=stream)
        compute.wait_stream(stream)

    def overlapped():
        events = [torch.cuda.Event() for _ in ns]
        side.wait_stream(compute)
        backward(events)
        plan.step_overlapped(grads, state, hyper, events, side)
        compute.wait_stream(side)

    def step_only():
        plan.step(grads, state, hyper, stream=stream)

    def buckets_only():
        for b in range(len(plan.buckets)):
            plan.step_bucket(b, grads, state, hyper, stream=side)
        compute.wait_stream(side)

    for fn in (backward, step_only, serial, overlapped):
        fn()
    t_bwd, t_step = timed(backward), timed(step_only)
    t_serial, t_over = timed(serial), timed(overlapped)
    # the same overlap with every bucket launch capped at a block budget (zr_plan_set_bucket_blocks), as a
    # communication library keeps to a few SMs; 0 = uncapped (one block per tile). Beside each, the bucket
    # launches alone at that budget: the step's rate per block, i.e. how many SMs it needs to keep HBM busy.
    budgets = {}
    for cap in budget_caps:
        plan.set_bucket_blocks(cap)
        buckets_only()
        t_alone = timed(buckets_only)
        overlapped()
        t_cap = timed(overlapped)
        budgets[str(cap)] = {"overlapped_ms": t_cap,
                             "hidden_fraction_of_step": (t_serial - t_cap) / t_step if t_step > 0 else None,
                             "step_alone_ms": t_alone,
                             "step_alone_GBs_per_block": (step_bytes / t_alone / 1e6 / cap) if step_bytes else None}
    plan.set_bucket_blocks(0)
    return {"backward_ms": t_bwd, "step_ms": t_step, "serial_ms": t_serial, "overlapped_ms": t_over,
            "hidden_fraction_of_step": (t_serial - t_over) / t_step if t_step > 0 else None,
            "block_budget_sweep": budgets,
            "synthetic_backward": f"bf16 GEMM {tokens} x {K} x n_b/1024 per bucket (~4*{tokens}*n_b FLOPs)",
            "api": "zr_step_bucket per bucket on a side stream after the bucket's ready event; the sweep caps each "
                   "bucket launch with zr_plan_set_bucket_blocks"}


def _host_memory_short(bytes_per_rank: int, local_ranks: int):
    """None if the host has room to pin bytes_per_rank for each of this node's ranks (with a tenth to spare), else
    the reason it has not (read from /proc/meminfo; unknown counts as room)."""
    try:
        with open("/proc/meminfo") as f:
            avail = next(int(l.split()[1]) * 1024 for l in f if l.startswith("MemAvailable:"))
    except (OSError, StopIteration, ValueError):
        return None
    need = int(1.1 * bytes_per_rank * local_ranks)
    if avail >= need:
        return None
    return (f"host memory: {local_ranks} rank(s) x {bytes_per_rank / 1e9:.1f} GB of pinned gradients need "
            f"{need / 1e9:.0f} GB, {avail / 1e9:.0f} GB available")


def _e2e_host_memory_short(bytes_per_rank: int, ws: int, device=None):
    """Whether the end-to-end leg must be left out for want of host memory to pin each rank's gradients: the
    reason, or None. Every rank takes the same decision, since the leg has a barrier and a max over ranks."""
    short = _host_memory_short(bytes_per_rank, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))
    if max_over_ranks(1.0 if short else 0.0, ws, device) > 0.0 and not short:
        short = "host memory: another rank of this job has too little to pin its gradients"
    return short


def _link_rates(torch, host, dev_buf, dev, stream, max_bytes: int = 4 << 30, reps: int = 3, rounds: int = 3):
    """Host<->device copy bandwidth: `rounds` rounds of `reps` copies of up to max_bytes between a pinned host
    tensor and a device tensor, each direction timed with CUDA events on the launching stream; the best round
    counts (the link is shared with the host's other traffic, so single rounds vary)."""
    k = min(host.numel(), dev_buf.numel(), max_bytes // host.element_size())
    h, d = host[:k], dev_buf[:k]
    nbytes = k * host.element_size()
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        best = 0.0
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)
            torch.cuda.synchronize(dev)
            for _ in range(rounds):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    dst.copy_(src, non_blocking=True)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                best = max(best, nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9)
        out[f"link_{name}_GBs"] = best
    out["link_copy_bytes"] = int(nbytes)
    out["link_how"] = (f"pinned host <-> device tensor copy_ (one cudaMemcpyAsync), CUDA events, best of {rounds} "
                       f"rounds of {reps} copies, single stream")
    return out


def _setup(w, zr, zrgen, dev, stream, inplace_main):
    """Plan, seeded state and step-1 gradients of workload w on the device."""
    import torch
    from zrgen.layout import Layout
    plan = zr.Plan(list(w.tensors), W=w.W, A=w.A, dtype=w.dtype, stage=w.stage, cap=w.cap,
                   scaler=zr.Scaler(w.init_scale, w.dynamic))
    hyper = zr.AdamW(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    layout = Layout(w.tensors, plan.tensor_offsets, zrgen.sigma_per_tensor(w), w.seed, w.dtype, w.master_sigma)
    cs = stream.cuda_stream
    table = torch.from_numpy(zrgen.normal_table().copy()).to(dev)
    n = plan.numel
    # the main step: ping-pong sets (zr_step), or one set stepped in place (zr_step_inplace) for a workload
    # whose two sets do not fit, or on request
    if inplace_main:
        state = plan.new_state1(dev)
        master0, param0 = state.master, state.param
    else:
        state = plan.new_state(dev)
        master0, param0 = state.master[0], state.param[0]
    master0.zero_()
    layout.master_dev(master0, table, cs)
    zr.all_gather(master0, [param0])
    grads = [torch.zeros(n, dtype=plan.torch_dtype(), device=dev) for _ in range(w.W * w.A)]
    for r in range(w.W * w.A):
        layout.grads_dev(grads[r], 1, r, w.init_scale, table, cs)
    torch.cuda.synchronize(dev)
    return plan, hyper, state, grads


def _measure_step(args, w, zr, plan, hyper, state, grads, dev, stream, ws, gpu_index, inplace_main):
    """The timed region: args.steps replays of the step captured as a CUDA graph, CUDA events on the launching
    stream, clocks sampled throughout; re-taken once if a thermal or hardware slowdown was seen. Returns the
    numbers of the JSON line for this workload."""
    import torch

    def timed(k):
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            graph.replay()  # one fused-step launch (two in place)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if ws > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1)

    for _ in range(args.warmup):
        if inplace_main:
            plan.step_inplace(grads, state, hyper, stream=stream)
        else:
            plan.step(grads, state, hyper, stream=stream)
    torch.cuda.synchronize(dev)
    # the step as a one-launch CUDA graph, so small workloads are not bound by host launch overhead
    graph = plan.capture(grads, state, hyper)
    torch.cuda.synchronize(dev)

    attempts = 0
    while True:
        sampler = ClockSampler(gpu_index)
        sampler.start()
        ms_total = timed(args.steps)
        clocks = sampler.stop()
        attempts += 1
        bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"} & set(clocks.get("reasons", []))
        if not bad or attempts >= 2:
            break
    rep = plan.report(stream)
    assert rep.overflow == 0 and rep.steps == args.warmup + args.steps * attempts, rep.as_dict()
    del graph

    ms_max = max_over_ranks(ms_total, ws, dev)
    ms_step = ms_max / args.steps
    value = whole_job_rate(plan.n_real, ms_step * 1e-3, ws)

    # roofline of the fused kernel: one launch per step, algorithmic bytes (2*W*A + 26) per param; in place,
    # of the step's two launches together, (4*W*A + 26) per param
    peak, peak_kind = _peaks()
    step_bytes = rep.bytes_alg + (2 * w.W * w.A * plan.n_real if inplace_main else 0)
    achieved = step_bytes / (ms_total / args.steps * 1e-3) / 1e9
    staging = _staging_name(zr, plan)
    if inplace_main:
        traffic, _digest = _traffic_record(w.name, "inplace_step", "traffic_bytes_per_step")
        kernel = ("fused_step_kernel flag pass + in-place update (bytes and time of the step's two launches "
                  "together)")
    elif staging in ("bulk", "bulk_io"):
        traffic, _digest = _traffic_record(w.name, TRAFFIC_PREFIX[staging], files=KERNEL_FILES[staging])
        kernel = ("fused_bulk_kernel (one launch per step; loads staged by cp.async.bulk into shared memory" +
                  (", results written back by cp.async.bulk)" if staging == "bulk_io" else ")"))
    else:
        traffic, _digest = _traffic_record(w.name)
        kernel = "fused_step_kernel (one launch per step; loads staged in registers)"
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "peak_source": f"{peak_kind} HBM copy bandwidth",
                "frac_of_8tbs_nominal": achieved / 8000.0, "kernel": kernel}
    clk = {"sm_mhz": clocks.get("sm_mhz"), "sm_max_mhz": clocks.get("sm_max_mhz"), "reasons": clocks.get("reasons"),
           "samples": clocks.get("samples"), "power_w_max": clocks.get("power_w_max"), "attempts": attempts}
    return {"ms_step": ms_step, "value": value, "step_bytes": step_bytes, "achieved": achieved,
            "roofline": roofline, "clocks": clk, "current": rep.current,
            "staging": "one state set in place (register staging)" if inplace_main else staging}


# the fused kernels' source files, whose hash a committed traffic record must match
KERNEL_FILES = {"registers": ("zr_step_kernel.cuh", "zr_device.cuh"),
                "bulk": ("zr_step_bulk.cuh", "zr_step_kernel.cuh", "zr_device.cuh"),
                "bulk_io": ("zr_step_bulk.cuh", "zr_step_kernel.cuh", "zr_device.cuh")}
TRAFFIC_PREFIX = {"registers": "fused_step", "bulk": "fused_bulk", "bulk_io": "fused_bulk_io"}


def _staging_name(zr, plan) -> str:
    return {zr.STAGING_BULK: "bulk", zr.STAGING_BULK_IO: "bulk_io"}.get(plan.staging, "registers")


def _measure_other_staging(args, w, zr, plan, hyper, state, grads, dev, stream, steps=20):
    """The same step with the other load staging than the plan's (bulk copies into shared memory, or 16-byte loads
    into registers), captured as a CUDA graph and timed like the main step on the same buffers; the plan's own
    staging is restored afterwards."""
    import torch
    own = plan.staging
    other = zr.STAGING_REGISTERS if own == zr.STAGING_BULK else zr.STAGING_BULK
    try:
        plan.set_staging(other)
    except zr.ZrError as ex:
        return {"unavailable": str(ex)}
    name = _staging_name(zr, plan)
    for _ in range(3):
        plan.step(grads, state, hyper, stream=stream)
    torch.cuda.synchronize(dev)
    g = plan.capture(grads, state, hyper)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    rep = plan.report(stream)
    assert rep.overflow == 0, rep.as_dict()
    plan.set_staging(own)
    del g
    ms = e0.elapsed_time(e1) / steps
    peak, _ = _peaks()
    achieved = rep.bytes_alg / (ms * 1e-3) / 1e9
    traffic, _ = _traffic_record(w.name, TRAFFIC_PREFIX[name], files=KERNEL_FILES[name])
    return {"staging": name, "ms_per_step": ms, "Gparams_per_s": plan.n_real / ms / 1e6, "hbm_GBs": achieved,
            "frac_of_measured_copy": achieved / peak, "traffic": traffic, "steps": steps,
            "call": "zr_step after zr_plan_set_staging to the other staging, captured as a CUDA graph"}


def _measure_noalloc(zr, plan, hyper, state, grads, w, dev, stream, current, reps=10):
    """zr_step_noalloc (scratch in a static device array, nothing allocated) against zr_step on the same
    buffers, both launched eagerly, CUDA events on the launching stream. Every step here is clean, so the
    caller-side live set flips after each call."""
    import torch
    of = torch.zeros(1, dtype=torch.int32, device=dev)
    cur = current
    for _ in range(3):
        zr.step_noalloc(plan.buckets, w.W, w.A, w.dtype, grads, state, cur, hyper, w.init_scale, 1, of,
                        stream=stream)
        cur = 1 - cur
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(reps):
        zr.step_noalloc(plan.buckets, w.W, w.A, w.dtype, grads, state, cur, hyper, w.init_scale, 2 + i, of,
                        stream=stream)
        cur = 1 - cur
    e1.record(stream)
    torch.cuda.synchronize(dev)
    assert int(of.item()) == 0
    na_ms = e0.elapsed_time(e1) / reps
    for _ in range(3):
        plan.step(grads, state, hyper, stream=stream)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(reps):
        plan.step(grads, state, hyper, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    st_ms = e0.elapsed_time(e1) / reps
    return {"ms_per_step": na_ms, "zr_step_ms_per_step": st_ms, "ratio_to_zr_step": na_ms / st_ms,
            "launches_per_step": 2, "steps": reps,
            "call": "zr_step_noalloc (set-up launch + the fused kernel, eager) against zr_step (eager)"}


def run_zr(args, w):
    import torch
    ws, rank, local = _dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    else:
        torch.cuda.set_device(0)
    dev = torch.device(f"cuda:{local if ws > 1 else 0}")
    gpu_index = local if ws > 1 else 0

    import __graft_entry__
    if rank == 0 or ws == 1:
        __graft_entry__.build()
    if ws > 1:
        torch.distributed.barrier()
        __graft_entry__.build()  # no-op once built
    import zero_gradient_reduction_gb300 as zr
    import zrgen

    stream = torch.cuda.current_stream(dev)
    inplace_main = args.inplace or w.state_sets == 1
    plan, hyper, state, grads = _setup(w, zr, zrgen, dev, stream, inplace_main)
    if args.staging:
        plan.set_staging({"bulk": zr.STAGING_BULK, "bulk_io": zr.STAGING_BULK_IO,
                          "registers": zr.STAGING_REGISTERS}[args.staging])
    n = plan.numel
    main = _measure_step(args, w, zr, plan, hyper, state, grads, dev, stream, ws, gpu_index, inplace_main)
    ms_step, value, step_bytes = main["ms_step"], main["value"], main["step_bytes"]
    peak, _ = _peaks()
    rep = plan.report(stream)
    # the in-place step (zr_step_inplace: a flag pass, then AdamW in place on ONE state set, for runs with
    # no room for a second set), timed right after the step it is compared with, on the live set of the
    # ping-pong state so that it needs no memory of its own: (4*W*A + 26) bytes per param, two launches
    inplace = None
    if not args.no_chain and not inplace_main:
        k = plan.report(stream).current
        one = zr.State1.of(state.master[k], state.m[k], state.v[k], state.param[k])
        for _ in range(3):
            plan.step_inplace(grads, one, hyper, stream=stream)
        torch.cuda.synchronize(dev)
        g_ip = plan.capture(grads, one, hyper)
        torch.cuda.synchronize(dev)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(args.chain_steps):
            g_ip.replay()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        ip_rep = plan.report(stream)
        assert ip_rep.overflow == 0 and ip_rep.current == k, ip_rep.as_dict()
        ip_ms = c0.elapsed_time(c1) / args.chain_steps
        ip_bpp = 4 * w.W * w.A + 26
        inplace = {"ms_per_step": ip_ms, "Gparams_per_s": plan.n_real / ip_ms / 1e6, "alg_bytes_per_param": ip_bpp,
                   "hbm_GBs": ip_bpp * plan.n_real / ip_ms / 1e6,
                   "frac_of_measured_copy": ip_bpp * plan.n_real / ip_ms / 1e6 / peak,
                   "launches_per_step": 2, "state_bytes_saved_GB": 14 * n / 1e9,
                   "call": "zr_step_inplace captured as a CUDA graph (flag pass, then the update in place)"}
        del g_ip, one

    # the same step with the other load staging (register loads, or bulk copies into shared memory)
    other = None
    if not args.no_chain and not inplace_main:
        other = _measure_other_staging(args, w, zr, plan, hyper, state, grads, dev, stream)

    # comparison point: the same step as the unfused chain of standalone calls (reduce-scatter per bucket
    # into fp32 sums, flag pass + AdamW in place, cast/all-gather), (2W + 38) bytes per param
    chain = None
    side = not args.no_chain and not inplace_main  # the side measurements use the ping-pong sets
    if w.A == 1 and side:
        sums = torch.empty(n, dtype=torch.float32, device=dev)
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
        k = rep.current

        def chain_step():
            for (b0, blen, _c) in plan.buckets:
                views = [g[b0:b0 + blen] for g in grads]
                zr.reduce_scatter(views, sums[b0:b0 + blen], flag, stream=stream)
            zr.adamw_shard_step(sums, state.m[k], state.v[k], state.master[k], hyper, w.init_scale, w.W, 1, flag,
                                stream=stream)
            zr.all_gather(state.master[k], [state.param[k]], stream=stream)

        for _ in range(3):
            chain_step()
        torch.cuda.synchronize(dev)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(args.chain_steps):
            chain_step()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        chain_ms = c0.elapsed_time(c1) / args.chain_steps
        chain_bytes = (2 * w.W + 38) * plan.n_real
        chain = {"ms_per_step": chain_ms, "Gparams_per_s": plan.n_real / chain_ms / 1e6,
                 "alg_bytes_per_param": 2 * w.W + 38, "hbm_GBs": chain_bytes / chain_ms / 1e6,
                 "launches_per_step": len(plan.buckets) + 3,
                 "calls": "zr_reduce_scatter per bucket, zr_adamw_shard_step, zr_all_gather"}
        del sums
    if w.A > 1 and side:
        # the standalone accumulate path: A zr_accumulate passes per worker into fp32, then the step on the
        # fp32 sums (W*(2A + 4(A-1) + 4A) + 4W + 26 bytes per param against 2WA + 26 fused)
        acc_plan = zr.Plan(list(w.tensors), W=w.W, A=1, dtype=w.dtype, stage=w.stage, cap=w.cap,
                           scaler=zr.Scaler(w.init_scale, w.dynamic), fp32_grads=True)
        accs = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(w.W)]

        def acc_step():
            for wk in range(w.W):
                for q in range(w.A):
                    zr.accumulate(grads[wk * w.A + q], accs[wk], q == 0, stream=stream)
            acc_plan.step(accs, state, hyper, stream=stream)

        for _ in range(3):
            acc_step()
        torch.cuda.synchronize(dev)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(args.chain_steps):
            acc_step()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        acc_ms = c0.elapsed_time(c1) / args.chain_steps
        acc_bytes = (w.W * (2 * w.A + 4 * (w.A - 1) + 4 * w.A) + 4 * w.W + 26) * plan.n_real
        chain = {"ms_per_step": acc_ms, "Gparams_per_s": plan.n_real / acc_ms / 1e6,
                 "alg_bytes_per_param": acc_bytes // plan.n_real, "hbm_GBs": acc_bytes / acc_ms / 1e6,
                 "launches_per_step": w.W * w.A + 1,
                 "calls": "zr_accumulate per worker and micro-batch, then zr_step on the fp32 sums"}
        acc_plan.close()
        del accs

    # ZeRO-3: the parameter all-gather before each layer's forward/backward, bucket by bucket, from the W
    # shards into a transient replica (2 bytes read + 2 written per param)
    zero3 = None
    if side:
        shards = plan.new_shards(dev)
        plan.shard_params(state.param[rep.current], shards, stream=stream)
        transient = torch.empty_like(state.param[0])

        def gather_all():
            for b in range(len(plan.buckets)):
                plan.gather_params(shards, transient, b, b + 1, stream=stream)

        for _ in range(3):
            gather_all()
        torch.cuda.synchronize(dev)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(args.chain_steps):
            gather_all()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        g_ms = c0.elapsed_time(c1) / args.chain_steps
        # the same launches captured once as a CUDA graph: no host launch gap between buckets
        gg = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.graph(gg, stream=side):
            for b in range(len(plan.buckets)):
                plan.gather_params(shards, transient, b, b + 1, stream=side)
        stream.wait_stream(side)
        gg.replay()
        torch.cuda.synchronize(dev)
        c0.record(stream)
        for _ in range(args.chain_steps):
            gg.replay()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        gg_ms = c0.elapsed_time(c1) / args.chain_steps
        zero3 = {"ms_all_buckets": g_ms, "launches": len(plan.buckets), "hbm_GBs": 4 * plan.numel / g_ms / 1e6,
                 "frac_of_measured_copy": 4 * plan.numel / g_ms / 1e6 / _peaks()[0],
                 "ms_all_buckets_graph": gg_ms, "frac_of_measured_copy_graph": 4 * plan.numel / gg_ms / 1e6 / _peaks()[0],
                 "call": "zr_gather_params per bucket (the all-gather before each layer's forward and backward); "
                         "eager launches, and the same launches as one CUDA graph"}
        del gg
        del shards, transient

    overlap = None
    if side and w.A == 1:
        overlap = measure_overlap(torch, zr, plan, grads, state, hyper, dev, stream, step_bytes=step_bytes)

    offload = None
    if side and w.A == 1 and ws == 1:
        # ZeRO-Offload: reduce-scatter on the GPU, AdamW on the host cores over host-resident fp32 state,
        # 4 B/param of sums down and 2 B/param of parameters back over the host link
        nthreads = os.cpu_count() or 8
        sums_dev = torch.empty(n, dtype=torch.float32, device=dev)
        sums_host = torch.empty(n, dtype=torch.float32, pin_memory=True)
        param_host = torch.empty(n, dtype=plan.torch_dtype(), pin_memory=True)
        h_master = np.full(n, 0.01, np.float32)
        h_m = np.zeros(n, np.float32)
        h_v = np.zeros(n, np.float32)
        plan.offload_step(grads, sums_dev, sums_host, h_master, h_m, h_v, param_host, state.param[0], hyper,
                          w.init_scale, 1, nthreads, stream=stream)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(2):
            plan.offload_step(grads, sums_dev, sums_host, h_master, h_m, h_v, param_host, state.param[0], hyper,
                              w.init_scale, 2 + i, nthreads, stream=stream)
        torch.cuda.synchronize(dev)
        o_ms = (time.perf_counter() - t0) / 2 * 1e3
        # the host-side bounds of that step: the host AdamW alone (zr_offload_adamw: a flag pass reading the 4-byte
        # sums, then 4 + 12 bytes read and 12 + 2 written per param of host memory) on the same arrays, and a
        # plain multi-threaded host copy
        t0 = time.perf_counter()
        zr.offload_adamw(sums_host, h_master, h_m, h_v, param_host, w.dtype, hyper, w.init_scale, w.W, 4, nthreads)
        ha_s = time.perf_counter() - t0
        k = min(n, 1 << 30)
        src = torch.from_numpy(h_m[:k])
        dst = torch.from_numpy(h_v[:k])
        dst.copy_(src)
        t0 = time.perf_counter()
        for _ in range(3):
            dst.copy_(src)
        hc_s = (time.perf_counter() - t0) / 3
        offload = {"ms_per_step": o_ms, "Gparams_per_s": plan.n_real / o_ms / 1e6, "host_threads": nthreads,
                   "link_bytes_per_param": 6, "host_state_GB": 12 * n / 1e9,
                   # host memory per param and step: the update's 16 read + 14 written, the sums copied in (4)
                   # and the parameters copied out (2)
                   "host_bytes_per_param": 36, "host_GBs": 36 * n / o_ms / 1e6,
                   "host_adamw_ms": ha_s * 1e3, "host_adamw_GBs": 34 * n / ha_s / 1e9,
                   "host_copy_GBs": 8 * k / hc_s / 1e9, "host_copy_threads": torch.get_num_threads(),
                   "call": "zr_offload_step (reduce-scatter on GPU, AdamW on the host CPU, params back); "
                           "host_adamw: zr_offload_adamw alone on the same host arrays (its flag pass over the sums, "
                           "then the update: 34 B/param of host memory); "
                           "host_copy: torch CPU copy_ of 4 GB fp32 (read + write bytes)"}
        del src, dst
        del sums_dev, sums_host, param_host, h_master, h_m, h_v

    e2e = None
    cpu = None
    e2e_short = None if args.no_e2e else _e2e_host_memory_short(2 * n * w.W * w.A, ws, dev)
    if not args.no_e2e and e2e_short:
        e2e = {"unavailable": e2e_short}
    elif not args.no_e2e:
        # end to end through the public API: pinned host gradients copied in every step, report read back
        host = [torch.empty(n, dtype=plan.torch_dtype(), pin_memory=True) for _ in range(w.W * w.A)]
        for r in range(w.W * w.A):
            host[r].copy_(grads[r])
        if inplace_main:
            # one set in place: the pinned host gradients are copied into the device replicas bucket by
            # bucket, then the in-place step reads them twice in HBM
            def e2e_step():
                return plan.step_inplace_from_host(host, grads, state, hyper, stream=stream)
            api = "zr_step_inplace_from_host (pinned host grads copied to the device, in-place step, report read back)"
        else:
            dgr = [torch.empty_like(g) for g in grads]

            def e2e_step():
                return plan.step_from_host(host, dgr, state, hyper, stream=stream)
            api = "zr_step_from_host (pinned host grads -> device, fused step, report read back)"
        e2e_step()  # warm
        if ws > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            r = e2e_step()
        dt = max_over_ranks(time.perf_counter() - t0, ws, dev)
        e2e = {"value": whole_job_rate(plan.n_real * args.e2e_steps, dt, ws), "unit": "Gparams/s",
               "h2d_bytes_per_step": int(2 * n * w.W * w.A), "d2h_bytes_per_step": int(ctypes.sizeof(r)),
               "ms_per_step": dt / args.e2e_steps * 1e3, "steps": args.e2e_steps, "api": api}
        # the host link itself: one large pinned copy per direction (cudaMemcpyAsync through torch), CUDA events
        link = _link_rates(torch, host[0], grads[0], dev, stream)
        e2e.update(link)
        e2e["frac_of_link_h2d"] = (e2e["h2d_bytes_per_step"] / (e2e["ms_per_step"] * 1e-3) / 1e9) / link["link_h2d_GBs"]
        del host, e2e_step
        if not inplace_main:
            del dgr

    rep_buckets = plan.buckets
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        ob, ooffs = oracle.bucket_plan(list(w.tensors), w.cap, w.W)  # the oracle's own table, not the plan's
        params, secs, what = oracle_sample(w, ob, ooffs, args.cpu_seconds)
        cpu = {"value": params / secs / 1e9, "unit": "Gparams/s", "cores": 1, "kind": "oracle",
               "sample": f"{what}, step 1 inputs; {secs:.1f} s single-threaded on the host"}

    # the other workload held to the HBM target, timed the same way on its own buffers once this workload's
    # are freed; with zr_step_noalloc beside it (its static scratch holds this workload's tile schedule)
    second = None
    if args.second and args.second != w.name and ws == 1:
        del plan, state, grads
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        w2 = zrgen.workload(args.second)
        plan2, hyper2, state2, grads2 = _setup(w2, zr, zrgen, dev, stream, False)
        m2 = _measure_step(args, w2, zr, plan2, hyper2, state2, grads2, dev, stream, ws, gpu_index, False)
        other2 = _measure_other_staging(args, w2, zr, plan2, hyper2, state2, grads2, dev, stream)
        noalloc = None
        try:
            noalloc = _measure_noalloc(zr, plan2, hyper2, state2, grads2, w2, dev, stream, m2["current"])
        except Exception as ex:  # a workload beyond the static scratch is refused by the call itself
            noalloc = {"unavailable": str(ex).splitlines()[0]}
        second = {"config": dict(_config(w2, plan2.buckets, f"inputs larger than L2: {m2['step_bytes'] / 1e9:.1f} GB "
                                         "moved per step", launch="zr_step captured once as a CUDA graph, replayed "
                                         "once per timed step"), staging=m2["staging"]),
                  "value": m2["value"], "unit": "Gparams/s", "ms_per_step": m2["ms_step"], "steps": args.steps,
                  "warmup": args.warmup, "hbm_tbs": m2["achieved"] / 1e3, "roofline": m2["roofline"],
                  "clocks": m2["clocks"], "gpu_launches": args.steps, "other_staging": other2,
                  "noalloc_step": noalloc}
        plan2.close()
        del plan2, state2, grads2
    else:
        plan.close()

    line = {
        "metric": "fused reduce-scatter+AdamW step Gparams/s", "value": value, "unit": "Gparams/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Philox4x32-10 normal draws, the workload's shapes and sigmas)",
        "config": _config(w, rep_buckets, f"inputs larger than L2: {step_bytes / 1e9:.1f} GB moved per step"
                          if step_bytes > 4 * 129e6 else
                          f"{step_bytes / 1e6:.0f} MB per step: L2-resident, reported, not an HBM figure",
                          launch="zr_step_inplace (flag pass + update) captured once as a CUDA graph, replayed once "
                          "per timed step" if inplace_main else
                          "zr_step captured once as a CUDA graph, replayed once per timed step", inplace=inplace_main),
        "hbm_tbs": main["achieved"] / 1e3,
        "roofline": main["roofline"],
        "staging": main["staging"],
        "cpu_baseline": cpu,
        "e2e": e2e,
        "unfused_chain": chain,
        "zero3_param_gather": zero3,
        "inplace_step": inplace,
        "other_staging": other,
        "bucketed_overlap": overlap,
        "zero_offload": offload,
        "gpu_launches": args.steps * (2 if inplace_main else 1),
        "clocks": main["clocks"],
        f"workload_{args.second}": second,
    }
    if second is None:
        del line[f"workload_{args.second}"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of the job: one rank each, launched by torch.distributed.run (independent replicas)")
    ap.add_argument("--steps", type=int, default=100, help="timed steps")
    ap.add_argument("--warmup", type=int, default=5, help="untimed steps before them (at least 3)")
    ap.add_argument("--impl", choices=["zr", "reference"], default="zr",
                    help="zr: this library on the GPU; reference: the oracle on the host cores")
    ap.add_argument("--workload", default=WORKLOAD_DEFAULT,
                    help="7b, 1p3b, gpt2, gpt2_W<W>, tiny, 13b, 7b_slice or sweep_W{2,4,8}_cap2^{19..28}")
    ap.add_argument("--second", default=None,
                    help=f"a second workload timed after the first, on freed memory (default: {SECOND_DEFAULT} when "
                         f"the workload is {WORKLOAD_DEFAULT}; 'none' for no second workload)")
    ap.add_argument("--e2e-steps", type=int, default=3, help="steps of the end-to-end leg (host gradients)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target seconds of the oracle's CPU baseline")
    ap.add_argument("--no-e2e", action="store_true", help="leave out the end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="leave out the oracle's CPU baseline")
    ap.add_argument("--no-chain", action="store_true",
                    help="leave out the side measurements (unfused chain, ZeRO-3 gather, in place, overlap, offload)")
    ap.add_argument("--chain-steps", type=int, default=5, help="steps of the unfused chain")
    ap.add_argument("--staging", choices=["bulk", "bulk_io", "registers"], default=None,
                    help="load staging of the main step's zr_step (default: the plan's own choice)")
    ap.add_argument("--inplace", action="store_true",
                    help="time zr_step_inplace on one state set as the main step (always so for 13b)")
    args = ap.parse_args()
    if args.warmup < 3:
        print(f"bench: raising --warmup {args.warmup} to the minimum of 3", file=sys.stderr)
        args.warmup = 3
    ws = _dist_env()[0]
    if args.gpus != ws:
        print(f"bench: --gpus {args.gpus} but {ws} process(es): N ranks come from torch.distributed.run "
              f"(--nproc-per-node N); measuring with {ws}", file=sys.stderr)
    import zrgen
    w = zrgen.workload(args.workload)
    if args.second is None:
        args.second = SECOND_DEFAULT if args.workload == WORKLOAD_DEFAULT else None
    elif args.second == "none":
        args.second = None
    if args.impl == "reference":
        return run_reference(args, w)
    return run_zr(args, w)


if __name__ == "__main__":
    sys.exit(main())
