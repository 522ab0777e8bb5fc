"""Child process for test_lamport_gpu.test_lamport_timeout: the Lamport call
runs with rank 1's pushes left out (AR_TEST_LAMPORT_SKIP_RANK, set by the
parent), so its slot keeps the empty marker and every poll of it runs out.
The call must return, ar_device_status must report the timeout once, and
the context must stay usable: a one-shot fused call, and a Lamport call on
a freshly filled buffer for a single rank (rank 1 does not exist there, so
nothing is left out), both match the oracle."""
import sys
import time

import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tests import tolerance as tol

ar.use_test_library()   # the settings the parent puts in the environment are read by the test build only


def _check(f, out, res, what):
    ro, rr, inv = oracle.residual_rmsnorm(f.partials, f.bias, f.residual, f.weight, f.eps, f.dtype)
    terms = [p.reshape(f.tokens, f.hidden) for p in f.partials] + [f.residual]
    tol.check_sum(res.cpu(), rr, terms, f.dtype, "residual_out " + what, R=f.R, hidden=f.hidden)
    tol.check_fused_out(out.cpu(), ro, terms, f.weight, inv, f.dtype, f.hidden, "out " + what, R=f.R)


def main():
    torch.cuda.set_device(0)
    assert ar.ar_device_status() == ar.AR_OK
    f = workloads.fused_inputs(2, 16, 4096, "bf16", partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                               bias_dist=None, weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=1)
    parts = [p.cuda() for p in f.partials]
    buf = ar.lamport_buffer(2, 4096, 16, torch.bfloat16)
    t0 = time.time()
    ar.ar_residual_rmsnorm_lamport(parts, f.residual.cuda(), f.weight.cuda(), f.eps, buffer=buf)
    torch.cuda.synchronize()
    took = time.time() - t0
    status = ar.ar_device_status()
    assert status == ar.AR_ERR_TIMEOUT, status
    assert ar.ar_device_status() == ar.AR_OK            # the record was cleared
    assert 0.5 < took < 30.0, took                      # the polls ran out after about a second
    # The context still works.
    out, res = ar.ar_residual_rmsnorm(parts, f.residual.cuda(), f.weight.cuda(), f.eps, strategy="ONESHOT")
    torch.cuda.synchronize()
    _check(f, out, res, "one-shot after timeout")
    g = workloads.fused_inputs(1, 16, 4096, "bf16", partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                               bias_dist=None, weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=2)
    ar.ar_lamport_init(buf, torch.bfloat16)
    out, res = ar.ar_residual_rmsnorm_lamport([g.partials[0].cuda()], g.residual.cuda(), g.weight.cuda(), g.eps,
                                              buffer=buf)
    torch.cuda.synchronize()
    _check(g, out, res, "Lamport after timeout")
    assert ar.ar_device_status() == ar.AR_OK
    # The same with separate push and reduce warps (many rows, the ring reused within the call):
    # rank 1's pushes are left out, every poll of its slot runs out, the call returns.
    h = workloads.fused_inputs(2, 3000, 1024, "bf16", partial_dist=("N", 0.0, 0.5),
                               residual_dist=("N", 0.0, 4.0), bias_dist=None, weight_dist=("N", 1.0, 0.05),
                               eps=1e-6, seed=3)
    assert ar.ar_lamport_supported(2, 1024, 3000, torch.bfloat16) is not None
    big = ar.lamport_buffer(2, 1024, 3000, torch.bfloat16)
    t0 = time.time()
    ar.ar_residual_rmsnorm_lamport([p.cuda() for p in h.partials], h.residual.cuda(), h.weight.cuda(), h.eps,
                                   buffer=big)
    torch.cuda.synchronize()
    took2 = time.time() - t0
    assert ar.ar_device_status() == ar.AR_ERR_TIMEOUT
    assert 0.5 < took2 < 60.0, took2
    print(f"lamport timeout ok ({took:.2f} s, {took2:.2f} s with separate push and reduce warps)")


if __name__ == "__main__":
    sys.exit(main())
