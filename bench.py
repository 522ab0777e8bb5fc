#!/usr/bin/env python3
"""Benchmark: the fused R-way sum + bias + residual + RMSNorm on GB300.

One step = one ar_residual_rmsnorm call over the TP prefill workload
(R=8 bf16 partials, tokens=8192 per GPU, hidden=8192, bias, residual, weight,
eps=1e-6) through the C ABI, inputs resident in HBM.  `value` is effective
HBM GB/s over all GPUs (algorithmic bytes = R*n*s + residual + bias + weight
+ both outputs, per call), the unit of the headline metric; `us_per_call`
gives the other half of it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): each rank owns its own block of
8192 token rows (weak scaling, no data-path collective); time is the max over
ranks.  `--impl reference` times the CPU oracle on a bounded sample of the
same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/call and effective HBM GB/s (fraction of GB300 peak) for R-way reduce+RMSNorm"
WORKLOAD = "TP prefill: R=8 bf16 partials, tokens=8192 per GPU, hidden=8192, bias, residual, RESIDUAL_RMS_NORM, eps=1e-6"
R, TOKENS, HIDDEN, EPS = 8, 8192, 8192, 1e-6
DATA = ("synthetic, seeded: partials N(0,1/8), residual N(0,4), bias N(0,0.02), weight N(1,0.05) "
        "(second argument = variance), drawn in fp32 and rounded to bf16")
FALLBACK_HBM_GBS = 6800.0
# Device code of the fused bulk-copy kernel, whose DRAM counters a committed
# ncu summary records: its own file, the helpers it uses and its argument
# block.  The launch shape (threads, stages, blocks per SM, shared memory,
# hence the grid) is checked separately, through the launch plan.
KERNEL_SOURCES = ["ar_kernels.cuh", "ar_tma.cuh", "ar_internal.h"]


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--strategy", default="AUTO", choices=["AUTO", "ONESHOT", "TWOSHOT"])
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--tokens", type=int, default=TOKENS, help="token rows per GPU (default: the workload's 8192)")
    p.add_argument("--no-extras", action="store_true", help="skip the secondary workloads")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


# ----------------------------------------------------------------------------- helpers

def algorithmic_bytes(R_, T, H, s, has_bias=True):
    n = T * H
    return R_ * n * s + n * s + (H * s if has_bias else 0) + H * s + 2 * n * s


def kernel_sources_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_allreduce_residual_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


def plan_key(plan: dict) -> str:
    """The launch shape of a fused call, as recorded beside its ncu counters."""
    return ":".join(str(plan[k]) for k in ("kernel_name", "threads_per_block", "units_per_thread", "stages",
                                           "blocks_per_sm", "smem_bytes"))


def profiled_traffic(kernel_tag: str, launch_plan: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on the current device code and
    the same launch shape; None otherwise."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    want = kernel_sources_hash()
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        text = open(os.path.join(pdir, name)).read()
        m_tag = re.search(r"^roofline_kernel:\s*(\S+)", text, re.M)
        m_hash = re.search(r"^kernel_sources_sha256:\s*(\S+)", text, re.M)
        m_plan = re.search(r"^launch_plan:\s*(\S+)", text, re.M)
        m_tr = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        if (m_tag and m_hash and m_plan and m_tr and m_tag.group(1) == kernel_tag and m_hash.group(1) == want
                and m_plan.group(1) == launch_plan):
            return float(m_tr.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU works."""
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuids):
        self.uuids = {u.lower().replace("gpu-", "") for u in uuids}
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 10:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append({"t": ts, "uuid": parts[1].lower().replace("gpu-", ""),
                             "sm": float(parts[2]), "sm_max": float(parts[3]),
                             "power": float(parts[4]) if parts[4] not in ("[N/A]", "") else None,
                             "hw": parts[6], "hw_thermal": parts[7], "sw_thermal": parts[8], "sw_power": parts[9]})
            except ValueError:
                continue
        self.file.close()
        os.unlink(self.file.name)
        mine = [r for r in rows if r["uuid"] in self.uuids]
        return mine if mine else rows   # uuid not matched: every visible GPU

    @staticmethod
    def summarize(rows, t0, t1):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        window = [r for r in rows if t0 - 0.05 <= r["t"] <= t1 + 0.05]
        if not window:  # region shorter than the sampling period: the nearest sample
            window = [min(rows, key=lambda r: abs(r["t"] - (t0 + t1) / 2))]
        reasons = set()
        for r in window:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in window),
                "sm_max_mhz": max(r["sm_max"] for r in window),
                "reasons": sorted(reasons), "samples": len(window)}


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    global TOKENS
    TOKENS = args.tokens
    import torch
    import torch.distributed as dist

    import tensor_allreduce_residual_gb300 as ar
    import workloads
    from tensor_allreduce_residual_gb300.dist import max_over_ranks, shard_range

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ar.lib()  # raises if the CUDA library is missing: there is no other path

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # Inputs: this rank's block of the global batch's rows (TOKENS per GPU),
    # drawn on the GPU, seeded per rank.
    row_begin, row_end = shard_range(TOKENS * world, rank, world)
    assert row_end - row_begin == TOKENS
    inp = workloads.tp_prefill(TOKENS, HIDDEN, seed=rank, device="cuda")
    parts, resid, weight, bias = inp.partials, inp.residual, inp.weight, inp.bias
    out = torch.empty_like(resid)
    res_out = torch.empty_like(resid)
    ws = torch.empty(ar.ar_workspace_size_rows(R, HIDDEN, TOKENS, ar.AR_BF16), dtype=torch.uint8, device=dev)
    bytes_call = algorithmic_bytes(R, TOKENS, HIDDEN, 2)
    stream = torch.cuda.current_stream()
    plan = ar.ar_query_launch(R, HIDDEN, TOKENS, ar.AR_BF16, args.strategy)
    resolved = ar.STRATEGY_NAMES[plan["strategy"]]
    warps = (plan["threads_per_row"] + 31) // 32
    launches_per_step = 1 if resolved == "ONESHOT" else 2

    def step(strategy=args.strategy):
        ar.ar_residual_rmsnorm(parts, resid, weight, EPS, bias=bias, out=out, residual_out=res_out,
                               intermediate=ws, strategy=strategy, stream=stream)

    uuids = [str(torch.cuda.get_device_properties(dev).uuid)]
    if world > 1:
        gathered = [None] * world
        dist.all_gather_object(gathered, uuids[0])
        uuids = gathered
    sampler = ClockSampler(uuids) if rank == 0 else None
    if sampler:
        sampler.start()

    for _ in range(args.warmup):
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    wall0 = time.time()
    t_begin.record(stream)
    for s0, s1 in ev:
        s0.record(stream)
        step()
        s1.record(stream)
    t_end.record(stream)
    barrier()
    wall1 = time.time()
    region_ms = t_begin.elapsed_time(t_end)
    per_step = [a.elapsed_time(b) for a, b in ev]
    clocks = ClockSampler.summarize(sampler.stop(), wall0, wall1) if sampler else None
    region_ms_max = max_over_ranks(region_ms, dev)

    value = bytes_call * world * args.steps / (region_ms_max * 1e-3) / 1e9
    ms_step = region_ms_max / args.steps
    peak, peak_src = measured_peaks()
    mean_launch_ms = statistics.fmean(per_step)
    achieved = bytes_call / (mean_launch_ms * 1e-3) / 1e9
    kernel_tag = plan["kernel_name"]
    traffic = profiled_traffic(kernel_tag, plan_key(plan))
    roofline = {"bound": "hbm", "kernel": kernel_tag, "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_src,
                "traffic": traffic, "algorithmic_bytes_per_launch": bytes_call,
                "launch_ms_mean": round(mean_launch_ms, 5), "launch_ms_median": round(statistics.median(per_step), 5)}

    # End to end through the C ABI on HOST buffers: every step,
    # ar_residual_rmsnorm_host copies that step's inputs from pinned host
    # memory, runs the fused kernels and copies both outputs back, in chunks
    # of 4096 rows (the last ones in shrinking pieces) with the copies
    # overlapping the kernels (4096-row chunks measured 233.5-233.7 GB/s
    # against 232.6-232.8 for 2048 and 230.3-230.7 for 1024).  Timed on the
    # stream until the outputs are in host memory.
    host_parts = [t.cpu().pin_memory() for t in parts]
    host_res, host_w, host_b = (t.cpu().pin_memory() for t in (resid, weight, bias))
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    chunk = 4096
    staging = torch.empty(ar.ar_host_staging_size(R, HIDDEN, chunk, ar.AR_BF16), dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host_parts + [host_res, host_w, host_b])
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def e2e_step():
        ar.ar_residual_rmsnorm_host(host_parts, host_res, host_w, EPS, staging, host_out[0], host_out[1],
                                    bias=host_b, chunk_tokens=chunk, strategy=args.strategy, stream=stream)

    for _ in range(5):
        e2e_step()
    # Three timed regions of e2e_steps steps each; the line reports the median region.  The host link
    # and host memory are shared with the box's other GPUs: now and then a whole region runs at about
    # half the rate (most often the first after two warm-up steps, hence five) while the copies alone,
    # timed next, do not, so one region alone is not representative.
    regions = []
    for _ in range(3):
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        barrier()
        regions.append(max_over_ranks(e0.elapsed_time(e1), dev))
    e2e_ms = statistics.median(regions)
    e2e = {"value": round(bytes_call * world * args.e2e_steps / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
           "us_per_call": round(e2e_ms * 1e3 / args.e2e_steps, 1),
           "regions_GBps": [round(bytes_call * world * args.e2e_steps / (ms * 1e-3) / 1e9, 2) for ms in regions],
           "statistic": "median of the 3 regions",
           "note": ("ar_residual_rmsnorm_host on pinned host buffers: inputs copied in and both outputs copied "
                    f"out inside the timed region, {chunk}-row chunks (the last in shrinking pieces) pipelined against "
                    "the kernels")}
    # The host link's bound for the same bytes: the step's copies alone (inputs in on one stream, the
    # outputs' bytes out on another, no kernels), device-timed the same way.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def copies_only():
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        with torch.cuda.stream(s_in):
            for h_, d_ in zip(host_parts + [host_res], list(parts) + [resid]):
                d_.copy_(h_, non_blocking=True)
        with torch.cuda.stream(s_out):
            host_out[0].copy_(out, non_blocking=True)
            host_out[1].copy_(res_out, non_blocking=True)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    copies_only()
    torch.cuda.synchronize()
    copy_regions = []
    for _ in range(3):  # median of three regions of three steps' copies, as for the call
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(3):
            copies_only()
        c1.record(stream)
        torch.cuda.synchronize()
        copy_regions.append(c0.elapsed_time(c1) * 1e3 / 3)
    copy_us = statistics.median(copy_regions)
    e2e["copies_only_us"] = round(copy_us, 1)
    e2e["frac_of_copies_only"] = round(copy_us / e2e["us_per_call"], 4)
    del host_parts, host_out, staging

    extras = None
    if not args.no_extras and rank == 0:
        extras = run_extras(ar, torch, workloads, parts, resid, weight, bias, out, res_out, ws, bytes_call, stream)

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": DATA,
        "config": {"workload": WORKLOAD.replace("tokens=8192", f"tokens={TOKENS}"), "R": R, "tokens_per_gpu": TOKENS, "global_tokens": TOKENS * world,
                   "hidden": HIDDEN, "io_dtype": "bf16", "eps": EPS, "strategy": args.strategy,
                   "resolved_strategy": resolved, "warps_per_token": warps,
                   "launch": {k: v for k, v in plan.items() if k != "strategy"},
                   "bytes_per_call": bytes_call, "parallelism": f"rows sharded over {world} GPU(s), no collective",
                   "l2": f"inputs larger than L2 ({bytes_call / 1e9:.2f} GB per call vs 129 MB L2): no flush between steps"},
        "us_per_call": round(ms_step * 1e3, 2), "frac_of_peak": round(value / world / peak, 4),
        "clocks": clocks, "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "roofline": roofline,
    }
    if extras is not None:
        line["extras"] = extras
    return line


def _time_calls(torch, fn, stream, n, warm=3):
    for _ in range(warm):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def _time_cold(torch, fn, stream, flush, n):
    """Mean per-call time with L2 flushed before every call.

    One event pair per call: on this GPU an event interval resolves only
    2.048 us, so each sample is quantized.  The mean of the samples averages
    the quantization out (the median would sit on a multiple of 2.048 us).

    `flush` is two buffers larger than L2: the first is written, then the
    second is read, so that the timed call finds L2 holding clean lines of
    the second buffer only.  (With the write alone, the timed call also paid
    for writing back up to an L2's worth of the flush's dirty lines.)  A
    fixed 50,000-cycle device sleep then keeps the GPU busy while the host
    enqueues the timed call, so the events bracket device time only, not the
    host's launch latency.
    """
    fn()  # a first call loads the kernel: not a sample
    torch.cuda.synchronize()
    ts = []
    for _ in range(n):
        flush[0].zero_()
        flush[1].amax()
        torch.cuda._sleep(50000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts)


def _time_graph(torch, fn, n=20, reps=5):
    """Median device time per call of `fn`, captured n times in a CUDA graph and replayed (no host overhead)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(n):
                fn()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / n)
    del g
    return statistics.median(ts)


def _time_graph_precise(torch, fn, nbytes):
    """Median over 11 replays of a graph of up to 100 calls (about 20 ms of work per replay at most)."""
    est_us = nbytes / 6.5e3 + 2.0
    return _time_graph(torch, fn, n=max(3, min(100, int(20000 / est_us))), reps=11)


def _time_rotate(torch, fns, stream, rounds=10):
    """Mean device time per call of back-to-back calls that cycle through `fns`, each on its own inputs:
    with the input sets together several times the size of L2, every call finds its inputs evicted by
    the others (L2-cold inputs, no flush between calls, launches overlapped as in a stream of layers)."""
    for f in fns:
        f()
    torch.cuda.synchronize()
    torch.cuda._sleep(50000)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(rounds):
        for f in fns:
            f()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (rounds * len(fns))


def _lamport_l2_bound(ar, torch, R, T, H, s, us):
    """The Lamport-style call's bound on one GPU.  Its buffer stays in L2 (a ring two grid steps deep), so
    its DRAM traffic is the fused call's, but every byte of the R partials is written into L2 twice (the
    push, then the marker that empties it again) besides the two outputs: (2R + 2) T H s bytes of L2
    writes.  The ceiling for those is measured here with the library's own streaming store kernel (the
    marker fill, ar_lamport_init, on an L2-resident 64 MB buffer, replayed from a CUDA graph).  The R + 1
    inputs stream in from DRAM at the same time and share that limit, so the call cannot reach it."""
    fill = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    w_ms = _time_graph(torch, lambda: ar.ar_lamport_init(fill, torch.bfloat16), n=50, reps=7)
    del fill
    w_gbps = (64 << 20) / w_ms / 1e6
    l2_write = (2 * R + 2) * T * H * s
    achieved = l2_write / us / 1e3
    return {"bound": "l2_write", "l2_write_bytes": l2_write, "achieved_GBps": round(achieved, 1),
            "peak_GBps": round(w_gbps, 1), "frac": round(achieved / w_gbps, 4),
            "floor_us": round(l2_write / w_gbps / 1e3, 1)}


def run_extras(ar, torch, workloads, parts, resid, weight, bias, out, res_out, ws, bytes_call, stream):
    """Secondary numbers: each fixed strategy on the prefill inputs, decode latency, reduce-only bandwidth.

    Calls run on the current stream (the capturing stream inside a graph capture).

    us_warm / us_cold: one Python call per timed call (host launch overhead
    included; cold = L2 flushed before each call).  us_graph: device time per
    call from a replayed CUDA graph of 20 calls (L2 warm).
    """
    ex = {}
    for s in ("ONESHOT", "TWOSHOT"):
        ms = _time_calls(torch, lambda s=s: ar.ar_residual_rmsnorm(
            parts, resid, weight, EPS, bias=bias, out=out, residual_out=res_out, intermediate=ws,
            strategy=s), stream, 100)
        ex[f"prefill_{s}"] = {"us_per_call": round(ms * 1e3, 2), "GBps": round(bytes_call / ms / 1e6, 1)}
    # The Lamport-style call on the same inputs.  Its buffer (a ring of two
    # grid steps of rows) is written, read and emptied through L2: 3 R n s
    # bytes beyond the fused call's pass there, not through DRAM.  GBps and
    # frac count the fused call's algorithmic bytes.
    T0, H0 = resid.shape
    lam = ar.lamport_buffer(len(parts), H0, T0, resid.dtype, resid.device)
    ms = _time_calls(torch, lambda: ar.ar_residual_rmsnorm_lamport(parts, resid, weight, EPS, bias=bias, out=out,
                                                                   residual_out=res_out, buffer=lam), stream, 30)
    peak0, _ = measured_peaks()
    ex["prefill_LAMPORT"] = {"us_per_call": round(ms * 1e3, 2), "GBps": round(bytes_call / ms / 1e6, 1),
                             "frac_of_peak": round(bytes_call / ms / 1e6 / peak0, 4),
                             "buffer_bytes": lam.numel(),
                             "over_oneshot": round(ms * 1e3 / ex["prefill_ONESHOT"]["us_per_call"], 3),
                             "l2_bound": _lamport_l2_bound(ar, torch, len(parts), T0, H0, resid.element_size(),
                                                           ms * 1e3)}
    del lam
    # The unfused route (the pages' "all-reduce, then norm"): ar_sum into a
    # temporary, then the residual + bias + norm call with that sum as its one
    # partial.  It moves (R+1)n s + 4n s + 2H s bytes against the fused
    # (R+3)n s + 2H s; GBps_effective counts the fused call's bytes.
    tmp = torch.empty_like(resid)

    def unfused():
        ar.ar_sum(parts, out=tmp)
        ar.ar_residual_rmsnorm([tmp], resid, weight, EPS, bias=bias, out=out, residual_out=res_out, intermediate=ws)

    ms = _time_calls(torch, unfused, stream, 50)
    T_, H_ = resid.shape
    moved = (len(parts) + 1) * T_ * H_ * 2 + 4 * T_ * H_ * 2 + 2 * H_ * 2
    ex["prefill_unfused_sum_then_norm"] = {
        "us_per_call": round(ms * 1e3, 2), "GBps_effective": round(bytes_call / ms / 1e6, 1),
        "bytes_moved": moved, "GBps_moved": round(moved / ms / 1e6, 1),
        "fused_speedup": round(ms * 1e3 / ex["prefill_ONESHOT"]["us_per_call"], 3)}
    # USE_MEMCPY (AllReduceStrategyConfig): the partials are first copied into
    # the registered workspace, then reduced from there -- the cost of staging.
    ws_cfg = torch.empty(ar.ar_config_workspace_size(len(parts), T_ * H_, H_, ar.AR_BF16), dtype=torch.uint8,
                         device=resid.device)
    prm = ar.make_params(parts, out, bias=bias, residual=resid, weight=weight, eps=EPS, hidden=H_,
                         residual_out=res_out, workspace=ws_cfg)
    ms = _time_calls(torch, lambda: ar.ar_allreduce_config(prm, ar.AR_FUSION_NONE, "AUTO",
                                                           ar.AR_CONFIG_USE_MEMCPY | ar.AR_CONFIG_RESIDUAL_RMS_NORM),
                     stream, 30)
    ex["prefill_use_memcpy"] = {"us_per_call": round(ms * 1e3, 2), "GBps_effective": round(bytes_call / ms / 1e6, 1),
                                "copy_bytes": 2 * len(parts) * T_ * H_ * 2,
                                "staging_cost_vs_in_place": round(ms * 1e3 / ex["prefill_ONESHOT"]["us_per_call"], 3)}
    del ws_cfg, prm
    ms = _time_calls(torch, lambda: ar.ar_rmsnorm(res_out, weight, EPS, out=out), stream, 50)
    nb = 2 * T_ * H_ * 2 + H_ * 2
    ex["prefill_rmsnorm_alone"] = {"us_per_call": round(ms * 1e3, 2), "bytes": nb, "GBps": round(nb / ms / 1e6, 1)}
    del tmp

    flush = (torch.empty(256 << 20, dtype=torch.uint8, device="cuda"),
             torch.zeros(256 << 20, dtype=torch.uint8, device="cuda"))
    # The prefill curve: R=8 bf16 H=8192 at 512 .. 4096 tokens (90 .. 738 MB
    # a call) through AUTO.  Cold: each call alone after an L2 flush, mean of
    # 20 (launch latency and the cold start of an isolated call included).
    # Cold stream: back to back on input sets that together exceed L2 several
    # times, so every call's inputs come from DRAM.  Warm: back-to-back calls
    # on the same inputs.  copy_us_cold: a plain device copy of the same
    # number of bytes timed like `cold` (half of them read; after the flush
    # L2 holds only clean lines, so the copy's writes, like the call's, stay
    # in the write-back L2 within the interval and its time is mostly that of
    # its reads); read_same_bytes_us_cold: a read-only pass (a sum) over as
    # many bytes as the call reads (its 9 inputs), timed the same way -- the
    # floor this way of timing sets for the call's reads at each size (an
    # isolated launch between events costs about 4 us here by itself).
    peak, _ = measured_peaks()
    curve = {}
    for T in (512, 1024, 2048, 4096):
        b = algorithmic_bytes(8, T, 8192, 2, has_bias=True)
        nsets = max(2, -(-400_000_000 // b))
        sets = []
        for k in range(nsets):
            f = workloads.tp_prefill(tokens=T, seed=k, device="cuda")
            o, r = torch.empty_like(f.residual), torch.empty_like(f.residual)
            wT = torch.empty(ar.ar_workspace_size_rows(8, 8192, T, ar.AR_BF16), dtype=torch.uint8, device="cuda")
            sets.append((f, o, r, wT))
        fns = [lambda f=f, o=o, r=r, wT=wT: ar.ar_residual_rmsnorm(
            f.partials, f.residual, f.weight, f.eps, bias=f.bias, out=o, residual_out=r, intermediate=wT,
            strategy="AUTO") for f, o, r, wT in sets]
        cold = _time_cold(torch, fns[0], stream, flush, 20)
        cold_stream = _time_rotate(torch, fns, stream)
        warm = _time_calls(torch, fns[0], stream, 50)
        src = torch.empty(b // 2, dtype=torch.uint8, device="cuda")
        dst = torch.empty_like(src)
        copy_cold = _time_cold(torch, lambda: dst.copy_(src), stream, flush, 20)
        reads = torch.zeros(9 * T * 8192 // 2, dtype=torch.float32, device="cuda")
        read_cold = _time_cold(torch, lambda: reads.sum(), stream, flush, 20)
        curve[f"T{T}"] = {"bytes": b, "kernel": ar.ar_query_launch(8, 8192, T, ar.AR_BF16, "AUTO")["kernel_name"],
                          "us_cold": round(cold * 1e3, 2), "GBps_cold": round(b / cold / 1e6, 1),
                          "frac_cold": round(b / cold / 1e6 / peak, 4),
                          "us_cold_stream": round(cold_stream * 1e3, 2),
                          "frac_cold_stream": round(b / cold_stream / 1e6 / peak, 4),
                          "us_warm": round(warm * 1e3, 2), "GBps_warm": round(b / warm / 1e6, 1),
                          "copy_us_cold": round(copy_cold * 1e3, 2),
                          "copy_frac_cold": round(b / copy_cold / 1e6 / peak, 4),
                          "read_same_bytes_us_cold": round(read_cold * 1e3, 2)}
        del sets, fns, src, dst, reads
    ex["prefill_curve_R8_bf16_H8192_AUTO"] = curve
    # PR1 reference case: R=2 fp32, 4 x 64, fusion NONE and RESIDUAL_RMS_NORM.
    p1 = workloads.pr1(seed=0)
    p1d = [t.cuda() for t in p1.partials]
    p1r, p1w, p1b = p1.residual.cuda(), p1.weight.cuda(), p1.bias.cuda()
    ex["pr1_R2_fp32_T4_H64"] = {
        "fused_us_graph": round(_time_graph(torch, lambda: ar.ar_residual_rmsnorm(p1d, p1r, p1w, p1.eps, bias=p1b,
                                                                                  strategy="AUTO")) * 1e3, 2),
        "sum_us_graph": round(_time_graph(torch, lambda: ar.ar_sum(p1d, strategy="AUTO")) * 1e3, 2)}
    dec_all = {}
    for T in workloads.TP_DECODE_TOKENS:
        f = workloads.tp_decode(T, device="cuda")
        o, r = torch.empty_like(f.residual), torch.empty_like(f.residual)
        dec_all[T] = round(_time_graph(torch, lambda f=f, o=o, r=r: ar.ar_residual_rmsnorm(
            f.partials, f.residual, f.weight, f.eps, bias=f.bias, out=o, residual_out=r, strategy="ONESHOT"),
            n=20, reps=3) * 1e3, 2)
    ex["tp_decode_R2_fp16_H4096_us_graph_by_tokens"] = dec_all
    dec = {}
    for T in (1, 8, 32):
        f = workloads.tp_decode(T, device="cuda")
        o, r = torch.empty_like(f.residual), torch.empty_like(f.residual)
        fn = lambda f=f, o=o, r=r: ar.ar_residual_rmsnorm(f.partials, f.residual, f.weight, f.eps, bias=f.bias,  # noqa: E731
                                                          out=o, residual_out=r, strategy="ONESHOT")
        lam = ar.lamport_buffer(2, 4096, T, torch.float16)
        fl = lambda f=f, o=o, r=r, lam=lam: ar.ar_residual_rmsnorm_lamport(  # noqa: E731
            f.partials, f.residual, f.weight, f.eps, bias=f.bias, out=o, residual_out=r, buffer=lam)
        dec[f"T{T}"] = {"us_warm": round(_time_calls(torch, fn, stream, 200) * 1e3, 2),
                        "us_cold": round(_time_cold(torch, fn, stream, flush, 30) * 1e3, 2),
                        "us_graph": round(_time_graph(torch, fn) * 1e3, 2),
                        "us_graph_lamport": round(_time_graph(torch, fl) * 1e3, 2)}
    ex["tp_decode_R2_fp16_H4096"] = dec
    r8 = {}
    for T in workloads.DECODE_R8_TOKENS:
        f = workloads.decode_r8(T, device="cuda")
        o, r = torch.empty_like(f.residual), torch.empty_like(f.residual)
        w8 = torch.empty(ar.ar_workspace_size_rows(8, 8192, T, ar.AR_BF16), dtype=torch.uint8, device="cuda")
        fn = lambda f=f, o=o, r=r, w8=w8: ar.ar_residual_rmsnorm(f.partials, f.residual, f.weight, f.eps,  # noqa: E731
                                                                 out=o, residual_out=r, intermediate=w8,
                                                                 strategy="AUTO")
        b = algorithmic_bytes(8, T, 8192, 2, has_bias=False)
        graph = {}   # the three strategies and the Lamport call back to back, before any L2 flush
        for s in ("ONESHOT", "TWOSHOT", "AUTO"):
            graph[s] = _time_graph(torch, lambda f=f, o=o, r=r, w8=w8, s=s: ar.ar_residual_rmsnorm(
                f.partials, f.residual, f.weight, f.eps, out=o, residual_out=r, intermediate=w8, strategy=s)) * 1e3
        lam = ar.lamport_buffer(8, 8192, T, torch.bfloat16)
        graph["LAMPORT"] = _time_graph(torch, lambda f=f, o=o, r=r, lam=lam: ar.ar_residual_rmsnorm_lamport(
            f.partials, f.residual, f.weight, f.eps, out=o, residual_out=r, buffer=lam)) * 1e3
        cold = _time_cold(torch, fn, stream, flush, 30)
        r8[f"T{T}"] = {"us_warm": round(_time_calls(torch, fn, stream, 100) * 1e3, 2), "us_cold": round(cold * 1e3, 2),
                       "GBps_cold": round(b / cold / 1e6, 1), "us_graph": round(graph["AUTO"], 2),
                       "us_graph_oneshot": round(graph["ONESHOT"], 2), "us_graph_twoshot": round(graph["TWOSHOT"], 2),
                       "us_graph_lamport": round(graph["LAMPORT"], 2),
                       "us_graph_after_flush": round(_time_graph(torch, fn) * 1e3, 2),
                       "auto": ar.STRATEGY_NAMES[ar.ar_query_strategy(8, T * 8192, 8192, ar.AR_BF16)[0]]}
    for v in r8.values():   # AUTO against the better fixed strategy (graph replay)
        v["auto_over_best_fixed"] = round(v["us_graph"] / min(v["us_graph_oneshot"], v["us_graph_twoshot"]), 3)
    ex["decode_R8_bf16_H8192"] = r8
    # Reduce-only sweep, R=4 fp16, n = 2^9 .. 2^27: device time per call
    # from a replayed graph of up to 100 calls, median of 11 replays (about
    # 0.01 us of resolution at the smallest sizes; working sets below L2,
    # 129 MB, are served partly by L2), each fixed partition and AUTO, with
    # AUTO's ratio to the better fixed one.  From 2^23 (84 MB) up also
    # L2-cold: each call alone after an L2 flush (`us_cold`), and back to back
    # on input sets that together exceed L2 several times (`us_cold_stream`).
    red = {}
    big = workloads.reduce_only(1 << 27, device="cuda")
    o_big = torch.empty_like(big.partials[0])
    for k in range(9, 28):
        n = 1 << k
        parts_n = [p[:n] for p in big.partials]
        o = o_big[:n]
        b = workloads.sum_algorithmic_bytes(4, n, "fp16")
        row = {}
        for s in ("ONESHOT", "TWOSHOT", "AUTO"):
            ms = _time_graph_precise(torch, lambda s=s: ar.ar_sum(parts_n, out=o, strategy=s), b)
            row[s] = {"us": round(ms * 1e3, 3), "GBps": round(b / ms / 1e6, 1)}
        row["auto"] = ar.STRATEGY_NAMES[ar.ar_query_strategy(4, n, 0, ar.AR_FP16, ar.AR_FUSION_NONE)[0]]
        row["auto_over_best_fixed"] = round(row["AUTO"]["us"] / min(row["ONESHOT"]["us"], row["TWOSHOT"]["us"]), 3)
        if k >= 23:
            sets = [(parts_n, o)] + [([torch.empty_like(p) for p in parts_n], torch.empty_like(o))
                                     for _ in range(max(1, -(-400_000_000 // b)) - 1)]
            for ps, _ in sets[1:]:
                for p, q in zip(ps, parts_n):
                    p.copy_(q)
            cold = _time_cold(torch, lambda: ar.ar_sum(parts_n, out=o, strategy="AUTO"), stream, flush, 20)
            fns = [lambda ps=ps, oo=oo: ar.ar_sum(ps, out=oo, strategy="AUTO") for ps, oo in sets]
            stream_cold = _time_rotate(torch, fns, stream)
            row["us_cold"] = round(cold * 1e3, 2)
            row["frac_cold"] = round(b / cold / 1e6 / peak, 4)
            row["us_cold_stream"] = round(stream_cold * 1e3, 2)
            row["frac_cold_stream"] = round(b / stream_cold / 1e6 / peak, 4)
            del sets, fns
        red[f"2^{k}"] = row
    ex["reduce_only_R4_fp16_sweep"] = red
    del flush
    # R=1 (the tpSize=1 passthrough): a copy into another buffer, and the
    # in-place call, which launches nothing.
    src = big.partials[0]
    b1 = workloads.sum_algorithmic_bytes(1, src.numel(), "fp16")
    ms = _time_calls(torch, lambda: ar.ar_sum([src], out=o_big), stream, 20)
    ms_in = _time_calls(torch, lambda: ar.ar_sum([src], out=src), stream, 200)
    ex["r1_passthrough_fp16_2^27"] = {"copy_us": round(ms * 1e3, 2), "copy_GBps": round(b1 / ms / 1e6, 1),
                                      "in_place_host_us": round(ms_in * 1e3, 2)}   # no kernel: host time only
    del big, o_big
    torch.cuda.empty_cache()
    return ex


# ----------------------------------------------------------------------------- the oracle

def oracle_sample(rows: int):
    import workloads
    return workloads.tp_prefill(tokens=rows, hidden=HIDDEN, seed=0)


def cpu_baseline(target_s: float = 10.0, rows: int = 512):
    """The CPU oracle, as it stands, on a bounded sample of the workload's rows (1 core)."""
    import oracle
    oracle.build()
    inp = oracle_sample(rows)
    b = algorithmic_bytes(R, rows, HIDDEN, 2)
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, inp.eps, "bf16")
        calls += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return {"value": round(b * calls / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{calls} calls x {rows} rows of the workload (R=8 bf16, hidden=8192), {el:.1f} s, "
                      f"single-threaded binary64 C, host {os.uname().machine}"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    rows = 64 if args.steps <= 200 else max(1, int(64 * 200 / args.steps))
    inp = oracle_sample(rows)
    b = algorithmic_bytes(R, rows, HIDDEN, 2)
    call = lambda: oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, inp.eps, "bf16")  # noqa: E731
    for _ in range(args.warmup):
        call()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        call()
    el = time.perf_counter() - t0
    value = b * args.steps / el / 1e9
    ms = el * 1e3 / args.steps
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": {"workload": WORKLOAD.replace("tokens=8192", f"tokens={TOKENS}"), "R": R, "tokens_per_gpu": TOKENS, "hidden": HIDDEN, "io_dtype": "bf16",
                   "eps": EPS, "sample_rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} rows of the workload per step, single-threaded binary64 C oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        print("bench.py: --warmup must be >= 3", file=sys.stderr)
        return 2
    if world > 1 and args.impl == "reference":
        line = run_reference(args, rank, world)
        if line:
            print(json.dumps(line), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.impl == "reference":
            line = run_reference(args, rank, world)
        else:
            line = run_ours(args, rank, world, local_rank)
            if line is not None and world == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline()
        if line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
