"""Measures the fused path's launch choices and writes the AUTO table.

    python -m tensor_allreduce_residual_gb300.tune sweep results.jsonl [--cases A,B] [--shapes S1,S2] [--tokens T1,T2] [--cold] [--alone]
    python -m tensor_allreduce_residual_gb300.tune table results.jsonl
    python -m tensor_allreduce_residual_gb300.tune sumsweep sums.jsonl
    python -m tensor_allreduce_residual_gb300.tune sumtable sums.jsonl

`sweep` times every one-shot shape (units per thread x where the row is kept
x when residual_out is written) and the two-shot path on the row shapes of
the measured workloads, each shape in its own process (the shape override
AR_ONESHOT_SHAPE is read once per process, by the test build libar_test.so,
which the children load).  Calls are captured in a CUDA graph and replayed,
so the numbers are device time without Python launch overhead.  With
`--cold`, a call whose working set is 64 MB or more is timed instead back to
back on several input sets that together exceed L2 several times, so that
every call reads its inputs from DRAM, as a layer's partials would be after
the rest of a layer's work has passed through L2.  With `--alone` as well,
such a call is also timed alone after an L2 flush (a 256 MB buffer written,
then another read, a device sleep, one event pair per call, mean of 30),
recorded as `us_alone`; the table ignores it.  `table` keeps the fastest choice per (element size, R, row
length, tokens) and rewrites csrc/ar_auto_table.h.  This is the measured
counterpart of heuristic_min_warp_number / selectImplementation.

`sumsweep` times the reduce-only call's two work partitions (one slice, R
rank slices) for n = 2^9 .. 2^27 elements at several rank counts and element
sizes, each point as the median of 11 replays of a graph of up to 100 calls
(enough to resolve 0.1 us at the smallest sizes); `sumtable` keeps the faster
partition per point and writes the reduce-only table of the same header.
"""
from __future__ import annotations

import json
import os
import statistics
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
TABLE = os.path.join(PKG, "csrc", "ar_auto_table.h")

# (name, R, dtype, hidden, bias, token counts)
CASES = [
    ("tp_decode_R2_fp16_H4096", 2, "fp16", 4096, True, [1, 2, 4, 8, 16, 32, 64, 256, 1024, 8192]),
    ("R8_bf16_H8192", 8, "bf16", 8192, False, [1, 8, 32, 64, 256, 512, 1024, 2048, 4096, 8192]),
    ("R4_fp16_H8192", 4, "fp16", 8192, True, [1, 64, 1024, 4096, 8192]),
    ("R8_bf16_H4096", 8, "bf16", 4096, True, [1, 64, 1024, 4096, 8192]),
    ("R2_bf16_H16384", 2, "bf16", 16384, True, [1, 64, 1024, 4096]),
    ("R16_bf16_H8192", 16, "bf16", 8192, True, [1, 64, 2048, 8192]),
    ("R3_fp16_H4096", 3, "fp16", 4096, True, [1, 64, 2048, 8192]),
]
SHAPES = ([f"{v}:{m}:{e}" for v in (1, 2, 4, 8) for m in (0, 1) for e in (0, 1)]
          + [f"{v}:2:{e}" for v in (2, 4) for e in (0, 1)]
          + [f"{v}:3:{e}:{b}" for v in (1, 2, 4, 8) for e in (0, 1) for b in (1, 2)]
          # the bulk-copy ring with fewer stages than fit (less in flight per SM)
          + [f"{v}:3:1:{b}:{st}" for v in (1, 2, 4, 8) for b in (1, 2) for st in (2, 4, 8)]
          + [f"{v}:4:1:{c}" for v in (1, 2, 4) for c in (2, 4, 8)])


# OneShotMode of a shape -> the ar_kernel codes a launch plan may report for it (the persistent
# mode runs as shared-memory rows where its kernel cannot take the row).
KERNEL_OF_MODE = {0: (1,), 1: (2,), 2: (2, 3), 3: (4,), 4: (6,)}


def shape_taken(plan: dict, shape: str) -> bool:
    """Whether a launch plan (ar_query_launch) is the one-shot shape "vpt:mode[:early[:bps[:stages]]]"
    that was asked for.  A shape that does not fit the row falls back to the rule's shape, and a
    sweep must not record that time under the name of the shape it asked for."""
    f = [int(x) for x in shape.split(":")]
    vpt, mode = f[0], f[1]
    early = int(len(f) > 2 and f[2] != 0)
    bps = f[3] if len(f) > 3 and f[3] > 0 else 1
    stages = f[4] if len(f) > 4 else 0
    if plan["strategy"] != 1 or plan["kernel"] not in KERNEL_OF_MODE.get(mode, ()):
        return False
    if plan["units_per_thread"] != vpt or plan["early_residual"] != early:
        return False
    if mode == 4 and plan["cluster"] != bps:
        return False
    if mode == 3 and (plan["blocks_per_sm"] != bps or (stages > 0 and plan["stages"] > stages)):
        return False
    return True


def _graph_time(torch, fn, n=10, reps=5):
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
    return statistics.median(ts)


COLD_MIN_BYTES = 64 << 20


def _cold_stream_time(torch, fns, rounds=10, reps=3):
    """Median over `reps` of the mean device time per call of back-to-back calls cycling through `fns`."""
    s = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        for f in fns:
            f()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(rounds):
            for f in fns:
                f()
        b.record(s)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / (rounds * len(fns)))
    return statistics.median(ts)


def _alone_time(torch, fn, n=30):
    """Mean device time of `fn` called alone after an L2 flush (written, then a second buffer read, so
    that L2 holds clean lines only), with a device sleep covering the host's launch of the call."""
    flush = (torch.empty(256 << 20, dtype=torch.uint8, device="cuda"),
             torch.zeros(256 << 20, dtype=torch.uint8, device="cuda"))
    s = torch.cuda.current_stream()
    fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(n):
        flush[0].zero_()
        flush[1].amax()
        torch.cuda._sleep(50000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts)


def _measure(strategy: str, shape: str, out, cases=None, token_filter=None, cold=False, alone=False):
    """Runs in a child process (AR_ONESHOT_SHAPE already set)."""
    sys.path.insert(0, ROOT)
    import torch

    import tensor_allreduce_residual_gb300 as ar
    import workloads
    ar.use_test_library()
    torch.cuda.set_device(0)
    for name, R, dtype, H, has_bias, tokens in CASES:
        if cases and name not in cases:
            continue
        for T in tokens:
            if token_filter and T not in token_filter:
                continue
            if strategy == "ONESHOT" and shape != "-":
                code = {"fp32": ar.AR_FP32, "fp16": ar.AR_FP16, "bf16": ar.AR_BF16}[dtype]
                try:
                    plan = ar.ar_query_launch(R, H, T, code, "ONESHOT")
                except ar.ARError:
                    continue   # no one-shot kernel holds this row
                if not shape_taken(plan, shape):
                    continue   # the shape does not fit this row: the rule's shape would run instead
            nbytes = workloads.fused_algorithmic_bytes(R, T, H, dtype, has_bias)
            timed_cold = cold and nbytes >= COLD_MIN_BYTES
            nsets = max(2, -(-(400 << 20) // nbytes)) if timed_cold else 1
            fns = []
            for k in range(nsets):
                f = workloads.fused_inputs(R, T, H, dtype, partial_dist=("N", 0.0, 1.0 / R),
                                           residual_dist=("N", 0.0, 4.0),
                                           bias_dist=("N", 0.0, 0.02) if has_bias else None,
                                           weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=k, device="cuda")
                o, r = torch.empty_like(f.residual), torch.empty_like(f.residual)
                ws = torch.empty(ar.ar_workspace_size_rows(R, H, T, ar.dtype_code(f.residual.dtype)),
                                 dtype=torch.uint8, device="cuda")
                fns.append(lambda f=f, o=o, r=r, ws=ws: ar.ar_residual_rmsnorm(
                    f.partials, f.residual, f.weight, f.eps, bias=f.bias, out=o, residual_out=r, intermediate=ws,
                    strategy=strategy))
            try:
                us = (_cold_stream_time(torch, fns) if timed_cold else _graph_time(torch, fns[0])) * 1e3
            except ar.ARError:
                continue
            rec = {"case": name, "R": R, "esize": workloads.ELEM_SIZE[dtype], "units_row": H * workloads.ELEM_SIZE[dtype] // 16,
                   "T": T, "strategy": strategy, "shape": shape, "us": round(us, 3),
                   "timing": "cold stream" if timed_cold else "graph replay"}
            if alone and timed_cold:
                rec["us_alone"] = round(_alone_time(torch, fns[0]) * 1e3, 3)
            if ar.ar_device_status() != ar.AR_OK:
                raise RuntimeError(f"{strategy} {shape} T={T}: a kernel gave up a bounded wait")
            out.write(json.dumps(rec) + "\n")
            out.flush()
            del fns
            torch.cuda.empty_cache()


def sweep(path: str, cases=None, shapes=None, tokens=None, cold=False, alone=False):
    with open(path, "w") as out:
        runs = [("TWOSHOT", "-")] + [("ONESHOT", s) for s in (shapes or SHAPES)]
        for strategy, shape in runs:
            env = dict(os.environ)
            env.pop("AR_ONESHOT_SHAPE", None)
            if shape != "-":
                env["AR_ONESHOT_SHAPE"] = shape
            extra = [",".join(cases or []), ",".join(str(t) for t in (tokens or [])), "cold" if cold else "",
                     "alone" if alone else ""]
            res = subprocess.run([sys.executable, "-m", "tensor_allreduce_residual_gb300.tune", "_child",
                                  strategy, shape, *extra], cwd=ROOT, env=env, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"sweep child {strategy} {shape} failed:\n{res.stderr[-2000:]}")
            out.write(res.stdout)
            out.flush()
            print(f"swept {strategy} {shape}", file=sys.stderr)


def table(path: str):
    best = {}
    with open(path) as f:
        for line in f:
            r = json.loads(line)
            key = (r["esize"], r["R"], r["units_row"], r["T"])
            if key not in best or r["us"] < best[key]["us"]:
                best[key] = r
    lines = []
    groups = {}
    for (esize, R, units, T), r in sorted(best.items()):
        groups.setdefault((esize, R, units), []).append((T, r))
    for (esize, R, units), items in groups.items():
        items.sort()
        for i, (T, r) in enumerate(items):
            tmax = T if i + 1 < len(items) else 2147483647
            how = " cold" if r.get("timing") == "cold stream" else ""
            if r["strategy"] == "TWOSHOT":
                lines.append(f"    {{{esize}, {R}, {units}, {tmax}, 2, 0, 0, 0, 1, 0}},  // {r['case']} T={T}: "
                             f"two-shot {r['us']} us{how}")
            else:
                parts = [int(x) for x in r["shape"].split(":")]
                v, m = parts[0], parts[1]
                e = parts[2] if len(parts) > 2 else 0
                b = parts[3] if len(parts) > 3 else 1
                st = parts[4] if len(parts) > 4 else 0
                lines.append(f"    {{{esize}, {R}, {units}, {tmax}, 1, {v}, {m}, {e}, {b}, {st}}},  // {r['case']} T={T}: "
                             f"one-shot {r['us']} us{how}")
    header = open(TABLE).read()
    start = header.index("static const AutoEntry kAutoTable[] = {")
    end = header.index("};", start)
    body = "static const AutoEntry kAutoTable[] = {\n" + "\n".join(lines) + \
        "\n    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0},  // sentinel\n"
    header = header[:start] + body + header[end:]
    header = header.replace("// No measured entries yet: every shape takes the rule in ar_api.cu.\n", "")
    with open(TABLE, "w") as f:
        f.write(header)
    print(f"wrote {len(lines)} entries to {TABLE}")


SUM_RANKS = (2, 3, 4, 8, 16)
SUM_DTYPES = ("fp16", "fp32")
SUM_LOG2N = range(9, 28)


def _graph_time_precise(torch, fn, est_us):
    """Median over 11 replays of a graph of up to 100 calls (about 20 ms of work per replay at most)."""
    n = max(3, min(100, int(20000 / max(est_us, 1.0))))
    return _graph_time(torch, fn, n=n, reps=11)


def sum_sweep(path: str):
    sys.path.insert(0, ROOT)
    import torch

    import tensor_allreduce_residual_gb300 as ar
    import workloads
    torch.cuda.set_device(0)
    with open(path, "w") as out:
        for dtype in SUM_DTYPES:
            es = workloads.ELEM_SIZE[dtype]
            for R in SUM_RANKS:
                nmax = 1 << max(SUM_LOG2N)
                big = workloads.sum_inputs(R, nmax, dtype, ("U", -1.0, 1.0), seed=R, device="cuda")
                o_big = torch.empty_like(big.partials[0])
                for k in SUM_LOG2N:
                    n = 1 << k
                    parts = [p[:n] for p in big.partials]
                    o = o_big[:n]
                    est = (R + 1) * n * es / 6.5e3 + 2.0   # us at about 6.5 TB/s, plus the launch
                    for strategy in ("ONESHOT", "TWOSHOT"):
                        us = _graph_time_precise(
                            torch, lambda s=strategy: ar.ar_sum(parts, out=o, strategy=s), est) * 1e3
                        rec = {"R": R, "esize": es, "n": n, "units": n * es // 16, "strategy": strategy,
                               "us": round(us, 3)}
                        out.write(json.dumps(rec) + "\n")
                        out.flush()
                del big, o_big
                torch.cuda.empty_cache()
                print(f"swept sums R={R} {dtype}", file=sys.stderr)


def sum_table(path: str, margin: float = 0.02):
    """Writes kSumAutoTable: per (element size, R), the faster partition at each measured n -- the R
    rank slices only where they beat one slice by more than `margin` (below that the two are within
    the noise of the measurement, and one slice is kept) -- merged into ascending ranges of 16-byte
    vectors, the last one open."""
    times = {}
    with open(path) as f:
        for line in f:
            r = json.loads(line)
            times.setdefault((r["esize"], r["R"], r["units"]), {})[r["strategy"]] = r
    best = {}
    for key, t in times.items():
        one, two = t.get("ONESHOT"), t.get("TWOSHOT")
        best[key] = two if one is None or (two is not None and two["us"] < one["us"] * (1.0 - margin)) else one
    groups = {}
    for (esize, R, units), r in sorted(best.items()):
        groups.setdefault((esize, R), []).append((units, r))
    lines = []
    for (esize, R), items in sorted(groups.items()):
        items.sort()
        code = {"ONESHOT": 1, "TWOSHOT": 2}
        run_start = 0
        for i, (units, r) in enumerate(items):
            last = i + 1 == len(items)
            if last or code[items[i + 1][1]["strategy"]] != code[r["strategy"]]:
                umax = "9223372036854775807LL" if last else f"{units}LL"
                first = items[run_start][0]
                lines.append(f"    {{{esize}, {R}, {umax}, {code[r['strategy']]}}},  // {first}..{units} vectors: "
                             f"{'one slice' if r['strategy'] == 'ONESHOT' else f'{R} rank slices'}")
                run_start = i + 1
    header = open(TABLE).read()
    start = header.index("static const SumAutoEntry kSumAutoTable[] = {")
    end = header.index("};", start)
    body = "static const SumAutoEntry kSumAutoTable[] = {\n" + "\n".join(lines) + \
        "\n    {0, 0, 0, 0},  // sentinel\n"
    with open(TABLE, "w") as f:
        f.write(header[:start] + body + header[end:])
    print(f"wrote {len(lines)} reduce-only entries to {TABLE}")


if __name__ == "__main__":
    cmd = sys.argv[1] if len(sys.argv) > 1 else ""
    if cmd == "_child":
        cases = [c for c in sys.argv[4].split(",") if c] if len(sys.argv) > 4 else None
        toks = [int(t) for t in sys.argv[5].split(",") if t] if len(sys.argv) > 5 else None
        _measure(sys.argv[2], sys.argv[3], sys.stdout, cases, toks, cold=len(sys.argv) > 6 and sys.argv[6] == "cold",
                 alone=len(sys.argv) > 7 and sys.argv[7] == "alone")
    elif cmd == "sweep":
        # sweep OUT [--cases a,b] [--shapes s1,s2] [--tokens t1,t2] [--cold] [--alone]
        args = sys.argv[3:]
        cold = "--cold" in args
        alone = "--alone" in args
        args = [a for a in args if a not in ("--cold", "--alone")]
        opts = dict(zip(args[0::2], args[1::2]))
        sweep(sys.argv[2], cases=[c for c in opts.get("--cases", "").split(",") if c] or None,
              shapes=[c for c in opts.get("--shapes", "").split(",") if c] or None,
              tokens=[int(t) for t in opts.get("--tokens", "").split(",") if t] or None, cold=cold, alone=alone)
    elif cmd == "table":
        table(sys.argv[2])
    elif cmd == "sumsweep":
        sum_sweep(sys.argv[2])
    elif cmd == "sumtable":
        sum_table(sys.argv[2])
    else:
        print(__doc__)
        sys.exit(2)
