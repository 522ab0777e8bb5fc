"""Child process for test_oneshot_shapes_gpu: parity of the one-shot fused path
under the shape that AR_ONESHOT_SHAPE forces (set by the parent)."""
import sys

import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tests import tolerance as tol

ar.use_test_library()   # the settings the parent puts in the environment are read by the test build only


def check(inp, rows=None):
    parts = [p.cuda() for p in inp.partials]
    out, res = ar.ar_residual_rmsnorm(parts, inp.residual.cuda(), inp.weight.cuda(), inp.eps,
                                      bias=None if inp.bias is None else inp.bias.cuda(), strategy="ONESHOT")
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


def main():
    torch.cuda.set_device(0)
    check(workloads.tp_decode(5, seed=1))
    check(workloads.decode_r8(3, seed=2))
    check(workloads.fused_inputs(4, 33, 1024, "fp32", partial_dist=("N", 0.0, 0.25), residual_dist=("N", 0.0, 1.0),
                                 bias_dist=("N", 0.0, 0.1), weight_dist=("N", 1.0, 0.1), eps=1e-5, seed=3))
    check(workloads.fused_inputs(2, 9, 16384, "bf16", partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                                 bias_dist=None, weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=4))
    # more rows than resident blocks: persistent blocks stride over rows
    big = workloads.tp_prefill(tokens=3000, seed=5)
    check(big, rows=[0, 1, 151, 152, 999, 1500, 2047, 2048, 2998, 2999])
    # rows of 1000 vectors: the last chunk of each row is ragged
    check(workloads.fused_inputs(8, 37, 8000, "bf16", partial_dist=("N", 0.0, 0.125), residual_dist=("N", 0.0, 4.0),
                                 bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=6))
    # a rank count without a compile-time specialisation
    check(workloads.fused_inputs(3, 21, 4096, "fp16", partial_dist=("N", 0.0, 0.3), residual_dist=("N", 0.0, 4.0),
                                 bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-5, seed=7))
    # Aliasing under this shape (persistent kernels prefetch later rows):
    # out on one of the partials, residual_out on the residual.
    al = workloads.tp_prefill(tokens=700, seed=8)
    ref = oracle.residual_rmsnorm(al.partials, al.bias, al.residual, al.weight, al.eps, al.dtype)
    ap = [p.cuda() for p in al.partials]
    ares = al.residual.cuda()
    o, r = ar.ar_residual_rmsnorm(ap, ares, al.weight.cuda(), al.eps, bias=al.bias.cuda(), out=ap[5],
                                  residual_out=ares, strategy="ONESHOT")
    torch.cuda.synchronize()
    assert o.data_ptr() == ap[5].data_ptr() and r.data_ptr() == ares.data_ptr()
    terms = [p.reshape(700, 8192) for p in al.partials] + [al.bias.expand(700, 8192).contiguous(), al.residual]
    tol.check_sum(r.cpu(), ref[1], terms, "bf16", "aliased residual_out", R=al.R, hidden=8192)
    tol.check_fused_out(o.cpu(), ref[0], terms, al.weight, ref[2], "bf16", 8192, "aliased out", R=al.R)
    # The norm on its own under the same shape: the register-resident kernel
    # with these units per thread, or the bulk-copy-fed kernel streaming x alone.
    for T, H, dt in [(37, 8192, "bf16"), (21, 8000, "bf16"), (9, 4096, "fp16"), (5, 1024, "fp32")]:
        g = torch.Generator().manual_seed(T + H)
        x = (torch.randn(T, H, generator=g, dtype=torch.float64) * 2).to(workloads.DTYPES[dt]).contiguous()
        w = (1 + 0.05 * torch.randn(H, generator=g, dtype=torch.float64)).to(workloads.DTYPES[dt]).contiguous()
        got = ar.ar_rmsnorm(x.cuda(), w.cuda(), 1e-6)
        torch.cuda.synchronize()
        ref, inv = oracle.rmsnorm(x, w, 1e-6, dt)
        tol.check_fused_out(got.cpu(), ref, [x], w, inv, dt, H, f"rmsnorm {T}x{H} {dt}", R=1)
    assert ar.ar_device_status() == ar.AR_OK, "a kernel gave up a bounded wait"
    print("shape ok")


if __name__ == "__main__":
    sys.exit(main())
