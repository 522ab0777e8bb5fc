"""ar_residual_rmsnorm_noalloc, the fused call for callers that cannot
allocate device memory (code under an allocator that owns all of the
device's memory, or code that must not wait on cudaMalloc / cudaFree): its
two-shot scratch is an array the library keeps on the device, so the caller
passes only inputs and outputs.

Each check calls it through the C ABI and compares it with the existing
ar_residual_rmsnorm (AR_TWOSHOT, caller workspace) on the same inputs:
residual_out must be bit-identical, out within the tolerance the parity
tests use (1e-5 of the row scale for fp32, 2 ulp of the element type for
fp16 / bf16).  Two calls in a row with different shapes and values show that
what the first call leaves in the shared array does not leak into the
second.  This file is collected last so that a run stopping at the first
failure has run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import tensor_allreduce_residual_gb300 as ar
import workloads
from tensor_allreduce_residual_gb300 import _build
from tests import tolerance as tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    _build.build()
    ar.lib()


def _to_cuda(inp):
    return ([p.cuda() for p in inp.partials], inp.residual.cuda(), inp.weight.cuda(),
            None if inp.bias is None else inp.bias.cuda())


def _existing(inp, parts, resid, weight, bias):
    ws = torch.empty(ar.ar_workspace_size_rows(inp.R, inp.hidden, inp.tokens, ar.dtype_code(resid.dtype)),
                     dtype=torch.uint8, device="cuda")
    return ar.ar_residual_rmsnorm(parts, resid, weight, inp.eps, bias=bias, intermediate=ws, strategy="TWOSHOT")


def _noalloc(inp, parts, resid, weight, bias):
    out, res_out = torch.empty_like(resid), torch.empty_like(resid)
    return ar.ar_residual_rmsnorm_noalloc(parts, resid, weight, inp.eps, bias=bias, out=out,
                                          residual_out=res_out)


def _compare(inp, new, old):
    (n_out, n_res), (o_out, o_res) = new, old
    torch.cuda.synchronize()
    assert torch.equal(n_res.cpu().view(torch.uint8), o_res.cpu().view(torch.uint8)), "residual_out differs"
    g = n_out.cpu().double().numpy().reshape(inp.tokens, inp.hidden)
    w = o_out.cpu().double().numpy().reshape(inp.tokens, inp.hidden)
    err = np.abs(g - w)
    if inp.dtype == "fp32":
        bound = 1e-5 * np.abs(w).max(axis=1, keepdims=True)
    else:
        bound = 2 * tol.ulp(w, inp.dtype)
    assert np.all(np.isfinite(g)) and np.all(err <= bound), f"out differs: max err {err.max()}"


def test_noalloc_matches_the_two_shot_call_on_two_calls_in_a_row():
    first = workloads.tp_prefill(tokens=300, seed=21)   # R=8 bf16, hidden 8192, bias
    second = workloads.tp_decode(7, seed=22)            # R=2 fp16, hidden 4096, fewer scratch entries
    for inp in (first, second):
        args = _to_cuda(inp)
        _compare(inp, _noalloc(inp, *args), _existing(inp, *args))


def test_noalloc_at_the_scratch_limit_and_beyond():
    # hidden == 1 takes the element-wise path with one chunk per row: the
    # scratch holds one fp32 per token, so 2^18 tokens fill 1 MiB exactly.
    limit_tokens = ar.AR_NOALLOC_SCRATCH_BYTES // 4
    assert ar.ar_workspace_size_rows(2, 1, limit_tokens, ar.AR_FP32) == ar.AR_NOALLOC_SCRATCH_BYTES
    inp = workloads.fused_inputs(2, limit_tokens, 1, "fp32", partial_dist=("N", 0.0, 0.5),
                                 residual_dist=("N", 0.0, 1.0), bias_dist=("N", 0.0, 0.1),
                                 weight_dist=("N", 1.0, 0.1), eps=1e-5, seed=23)
    args = _to_cuda(inp)
    _compare(inp, _noalloc(inp, *args), _existing(inp, *args))

    over = workloads.fused_inputs(2, limit_tokens + 1, 1, "fp32", partial_dist=("N", 0.0, 0.5),
                                  residual_dist=("N", 0.0, 1.0), weight_dist=("N", 1.0, 0.1), eps=1e-5, seed=24)
    parts, resid, weight, _ = _to_cuda(over)
    with pytest.raises(ar.ARError) as e:
        ar.ar_residual_rmsnorm_noalloc(parts, resid, weight, over.eps, out=torch.empty_like(resid),
                                       residual_out=torch.empty_like(resid))
    assert e.value.status == ar.AR_ERR_WORKSPACE
