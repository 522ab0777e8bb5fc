"""Child process for test_lamport_gpu.test_lamport_shape_parity: parity of the
Lamport-style call under the launch shape that AR_ONESHOT_SHAPE forces (set by
the parent): whole rows at a given number of vectors per thread (mode 0), or
rows split over C blocks (mode 4, C in the fourth field).  Shapes that do not
fit a case fall back to the call's own rule, so every case runs either way."""
import sys

import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tests import tolerance as tol

ar.use_test_library()   # the settings the parent puts in the environment are read by the test build only


def check(inp, rows=None, buf=None):
    parts = [p.cuda() for p in inp.partials]
    out, res = ar.ar_residual_rmsnorm_lamport(parts, inp.residual.cuda(), inp.weight.cuda(), inp.eps,
                                              bias=None if inp.bias is None else inp.bias.cuda(), buffer=buf)
    torch.cuda.synchronize()
    if rows is not None:
        idx = torch.tensor(rows)
        inp = workloads.FusedInputs(inp.R, len(rows), inp.hidden, inp.dtype, inp.eps,
                                    [p[idx].contiguous() for p in inp.partials], inp.residual[idx].contiguous(),
                                    inp.weight, inp.bias)
        out, res = out[idx.cuda()], res[idx.cuda()]
    o_out, o_res, inv = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, inp.eps, inp.dtype)
    T, H = inp.tokens, inp.hidden
    terms = [p.reshape(T, H) for p in inp.partials]
    if inp.bias is not None:
        terms.append(inp.bias.expand(T, H).contiguous())
    terms.append(inp.residual)
    tol.check_sum(res.cpu(), o_res, terms, inp.dtype, "residual_out", R=inp.R, hidden=H)
    tol.check_fused_out(out.cpu(), o_out, terms, inp.weight, inv, inp.dtype, H, "out", R=inp.R)


def fused(R, T, H, dtype, seed, bias=True):
    return workloads.fused_inputs(R, T, H, dtype, partial_dist=("N", 0.0, 1.0 / R), residual_dist=("N", 0.0, 4.0),
                                  bias_dist=("N", 0.0, 0.02) if bias else None, weight_dist=("N", 1.0, 0.05),
                                  eps=1e-6, seed=seed)


def main():
    torch.cuda.set_device(0)
    check(workloads.decode_r8(3, seed=2))
    check(workloads.tp_decode(5, seed=1))
    check(fused(4, 33, 1024, "fp32", 3))
    check(fused(3, 21, 4096, "fp16", 7))                  # no compile-time rank count
    check(fused(8, 6, 8200, "bf16", 9))                   # ragged slices and chunks
    # many more row groups than resident blocks: blocks stride over them
    big = fused(8, 2000, 1024, "bf16", 5)
    check(big, rows=[0, 1, 151, 152, 999, 1000, 1500, 1998, 1999])
    # more rows than the ring holds, so ring rows are reused within the call
    ring = fused(8, 3000, 2048, "bf16", 6)
    check(ring, rows=[0, 1, 511, 512, 1023, 1024, 1025, 2047, 2048, 2999])
    # one buffer, several calls
    buf = ar.lamport_buffer(8, 8192, 8, torch.bfloat16)
    for seed in (11, 12):
        check(workloads.decode_r8(8, seed=seed), buf=buf)
    assert ar.ar_device_status() == ar.AR_OK
    print("lamport shape ok")


if __name__ == "__main__":
    sys.exit(main())
