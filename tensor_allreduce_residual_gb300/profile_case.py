"""Runs one case of the library a fixed number of times, for a profiler.

    python -m tensor_allreduce_residual_gb300.profile_case fused \
        --R 8 --tokens 1024 --hidden 8192 --dtype bf16 --strategy ONESHOT --calls 3
    python -m tensor_allreduce_residual_gb300.profile_case sum --R 4 --n 33554432 --dtype fp16
    python -m tensor_allreduce_residual_gb300.profile_case rmsnorm --tokens 8192 --hidden 8192 --dtype bf16
    python -m tensor_allreduce_residual_gb300.profile_case lamport --R 8 --tokens 2048 --hidden 8192

Inputs are the seeded synthetic workloads (drawn on the device), the calls go
through the C ABI, and nothing is timed or checked: the point is a short,
deterministic launch sequence that `ncu -k <kernel> -s <skip> -c <count>`
can select from.  `--warmup` calls run first, then `--calls` more.
`--test-library` loads libar_test.so, whose launch shape follows
AR_ONESHOT_SHAPE (to profile a shape AUTO does not pick).
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None) -> int:
    p = argparse.ArgumentParser(description="run one library case for a profiler")
    p.add_argument("op", choices=["fused", "sum", "rmsnorm", "lamport"])
    p.add_argument("--R", type=int, default=8)
    p.add_argument("--tokens", type=int, default=1024)
    p.add_argument("--hidden", type=int, default=8192)
    p.add_argument("--n", type=int, default=1 << 25)
    p.add_argument("--dtype", default="bf16", choices=["fp32", "fp16", "bf16"])
    p.add_argument("--strategy", default="AUTO", choices=["ONESHOT", "TWOSHOT", "AUTO"])
    p.add_argument("--no-bias", action="store_true")
    p.add_argument("--warmup", type=int, default=2)
    p.add_argument("--calls", type=int, default=3)
    p.add_argument("--test-library", action="store_true", help="load libar_test.so (AR_ONESHOT_SHAPE applies)")
    a = p.parse_args(argv)

    import torch

    import tensor_allreduce_residual_gb300 as ar
    import workloads

    if a.test_library:
        ar.use_test_library()
    torch.cuda.set_device(0)
    ar.lib()
    if a.op == "sum":
        s = workloads.sum_inputs(a.R, a.n, a.dtype, ("U", -1.0, 1.0), seed=0, device="cuda")
        out = torch.empty_like(s.partials[0])
        call = lambda: ar.ar_sum(s.partials, out=out, strategy=a.strategy)  # noqa: E731
    elif a.op == "rmsnorm":
        x = workloads.draw(("N", 0.0, 4.0), a.tokens * a.hidden, a.dtype, 0, 100, "cuda").view(a.tokens, a.hidden)
        w = workloads.draw(("N", 1.0, 0.05), a.hidden, a.dtype, 0, 300, "cuda")
        out = torch.empty_like(x)
        call = lambda: ar.ar_rmsnorm(x, w, 1e-6, out=out)  # noqa: E731
    else:
        f = workloads.fused_inputs(a.R, a.tokens, a.hidden, a.dtype, partial_dist=("N", 0.0, 1.0 / a.R),
                                   residual_dist=("N", 0.0, 4.0),
                                   bias_dist=None if a.no_bias else ("N", 0.0, 0.02),
                                   weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=0, device="cuda")
        out, res = torch.empty_like(f.residual), torch.empty_like(f.residual)
        if a.op == "lamport":
            lam = ar.lamport_buffer(a.R, a.hidden, a.tokens, f.residual.dtype)
            call = lambda: ar.ar_residual_rmsnorm_lamport(f.partials, f.residual, f.weight, f.eps,  # noqa: E731
                                                          bias=f.bias, out=out, residual_out=res, buffer=lam)
        ws = torch.empty(max(1, ar.ar_workspace_size_rows(a.R, a.hidden, a.tokens, ar.dtype_code(f.residual.dtype))),
                         dtype=torch.uint8, device="cuda")
        if a.op == "fused":
            call = lambda: ar.ar_residual_rmsnorm(f.partials, f.residual, f.weight, f.eps,  # noqa: E731
                                                  bias=f.bias, out=out, residual_out=res, intermediate=ws,
                                                  strategy=a.strategy)
    torch.cuda.synchronize()
    for _ in range(a.warmup + a.calls):
        call()
    torch.cuda.synchronize()
    print(f"profile_case {a.op}: {a.warmup} + {a.calls} calls done")
    return 0


if __name__ == "__main__":
    sys.exit(main())
