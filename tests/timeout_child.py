"""Child process for test_wait_timeout_gpu.

`python -m tests.timeout_child` (test build, libar_test.so): the bulk-copy-fed
kernel runs with one ring stage of every block left unarmed
(AR_TEST_STALL_STAGE, set by the parent with the shape override that selects
that kernel).  Its bounded waits must run out, the call must return,
ar_device_status must report the timeout once, and the context must stay
usable for the next calls.

`python -m tests.timeout_child product` (the product library, libar.so, same
environment): the library reads neither setting, so the same call takes the
launch AUTO picks, returns within milliseconds with results that match the
oracle, and no wait gives up."""
import sys
import time

import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tests import tolerance as tol


def product():
    torch.cuda.set_device(0)
    assert ar.ar_device_status() == ar.AR_OK
    f = workloads.fused_inputs(2, 64, 8192, "bf16", partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                               bias_dist=None, weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=1)
    parts, resid, w = [p.cuda() for p in f.partials], f.residual.cuda(), f.weight.cuda()
    ar.ar_residual_rmsnorm(parts, resid, w, f.eps, strategy="ONESHOT")   # first call: module loading
    torch.cuda.synchronize()
    t0 = time.time()
    out, res = ar.ar_residual_rmsnorm(parts, resid, w, f.eps, strategy="ONESHOT")
    torch.cuda.synchronize()
    took = time.time() - t0
    assert took < 0.1, took                             # no bounded wait ran out
    assert ar.ar_device_status() == ar.AR_OK
    ro, rr, inv = oracle.residual_rmsnorm(f.partials, None, f.residual, f.weight, f.eps, "bf16")
    terms = [p.reshape(64, 8192) for p in f.partials] + [f.residual]
    tol.check_sum(res.cpu(), rr, terms, "bf16", "residual_out, product library", R=f.R, hidden=8192)
    tol.check_fused_out(out.cpu(), ro, terms, f.weight, inv, "bf16", 8192, "out, product library", R=f.R)
    print(f"product library ignores the test settings ({took * 1e3:.2f} ms)")


def main():
    ar.use_test_library()
    torch.cuda.set_device(0)
    assert ar.ar_device_status() == ar.AR_OK
    f = workloads.fused_inputs(2, 64, 8192, "bf16", partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                               bias_dist=None, weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=1)
    assert ar.ar_query_launch(2, 8192, 64, ar.AR_BF16, "ONESHOT")["kernel_name"] == "k_fused_oneshot_tma"
    t0 = time.time()
    ar.ar_residual_rmsnorm([p.cuda() for p in f.partials], f.residual.cuda(), f.weight.cuda(), f.eps,
                           strategy="ONESHOT")
    torch.cuda.synchronize()
    took = time.time() - t0
    status = ar.ar_device_status()
    assert status == ar.AR_ERR_TIMEOUT, status
    assert ar.ar_device_status() == ar.AR_OK            # the record was cleared
    assert 0.5 < took < 30.0, took                      # the waits ran out after about a second
    # The context still works: a reduce (no bounded waits) and the fused call through two-shot.
    s = workloads.reduce_only(4099, seed=3)
    got = ar.ar_sum([p.cuda() for p in s.partials])
    out, res = ar.ar_residual_rmsnorm([p.cuda() for p in f.partials], f.residual.cuda(), f.weight.cuda(), f.eps,
                                      strategy="TWOSHOT")
    torch.cuda.synchronize()
    tol.check_sum(got.cpu(), oracle.sum(s.partials, "fp16"), s.partials, "fp16", "sum after timeout", R=len(s.partials))
    ro, rr, inv = oracle.residual_rmsnorm(f.partials, None, f.residual, f.weight, f.eps, "bf16")
    terms = [p.reshape(64, 8192) for p in f.partials] + [f.residual]
    tol.check_sum(res.cpu(), rr, terms, "bf16", "residual_out after timeout", R=f.R, hidden=8192)
    tol.check_fused_out(out.cpu(), ro, terms, f.weight, inv, "bf16", 8192, "out after timeout", R=f.R)
    assert ar.ar_device_status() == ar.AR_OK
    print(f"timeout ok ({took:.2f} s)")


if __name__ == "__main__":
    sys.exit(product() if sys.argv[1:] == ["product"] else main())
