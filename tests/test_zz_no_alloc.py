"""ar_residual_rmsnorm_noalloc, the fused call for callers that cannot
allocate device memory (code under an allocator that owns all of the
device's memory, or code that must not wait on cudaMalloc / cudaFree): its
two-shot scratch is an array the library keeps on the device, so the caller
passes only inputs and outputs.

Each check calls it through the C ABI and compares it with the CPU oracle
under the parity tests' rules (tests/tolerance.py: 1e-5 of the row scale for
fp32; 2 ulp plus the fp32 accumulation floor for fp16 / bf16), and with the
existing ar_residual_rmsnorm (AR_TWOSHOT, caller workspace) on the same
inputs: both outputs must be bit-identical to that call's, since the two
launch the same kernels.  Two calls in a row with different shapes and
values show that what the first call leaves in the shared array does not
leak into the second.  This file is collected last so that a run stopping at
the first failure has run every other test; it also passes alone in a fresh
process.
"""
import pytest
import torch

import oracle
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


def _terms(inp):
    T, H = inp.tokens, inp.hidden
    t = [p.reshape(T, H) for p in inp.partials]
    if inp.bias is not None:
        t.append(inp.bias.expand(T, H).contiguous())
    t.append(inp.residual)
    return t


def _compare(inp, new, old):
    (n_out, n_res), (o_out, o_res) = new, old
    torch.cuda.synchronize()
    n_out, n_res = n_out.cpu(), n_res.cpu()
    # Against the oracle, under the parity tests' tolerance.
    ref_out, ref_res, inv = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, inp.eps,
                                                    inp.dtype)
    terms = _terms(inp)
    tol.check_sum(n_res, ref_res, terms, inp.dtype, "noalloc residual_out", R=inp.R, hidden=inp.hidden)
    tol.check_fused_out(n_out, ref_out, terms, inp.weight, inv, inp.dtype, inp.hidden, "noalloc out", R=inp.R)
    # Against the call with a caller workspace: the same kernels, so the same bits.
    assert torch.equal(n_res.view(torch.uint8), o_res.cpu().view(torch.uint8)), "residual_out differs"
    assert torch.equal(n_out.view(torch.uint8), o_out.cpu().view(torch.uint8)), "out differs"


def test_noalloc_matches_the_two_shot_call_on_two_calls_in_a_row():
    first = workloads.tp_prefill(tokens=300, seed=21)   # R=8 bf16, hidden 8192, bias
    second = workloads.tp_decode(7, seed=22)            # R=2 fp16, hidden 4096, fewer scratch entries
    for inp in (first, second):
        args = _to_cuda(inp)
        _compare(inp, _noalloc(inp, *args), _existing(inp, *args))


def test_noalloc_at_the_scratch_limit_and_beyond():
    # Rows of 4 fp32 values are one 16-byte vector, one two-shot chunk a row:
    # the scratch holds one fp32 per token, so 2^18 tokens fill 1 MiB exactly.
    limit_tokens = ar.AR_NOALLOC_SCRATCH_BYTES // 4
    assert ar.ar_workspace_size_rows(2, 4, limit_tokens, ar.AR_FP32) == ar.AR_NOALLOC_SCRATCH_BYTES
    inp = workloads.fused_inputs(2, limit_tokens, 4, "fp32", partial_dist=("N", 0.0, 0.5),
                                 residual_dist=("N", 0.0, 1.0), bias_dist=("N", 0.0, 0.1),
                                 weight_dist=("N", 1.0, 0.1), eps=1e-5, seed=23)
    args = _to_cuda(inp)
    _compare(inp, _noalloc(inp, *args), _existing(inp, *args))

    over = workloads.fused_inputs(2, limit_tokens + 1, 4, "fp32", partial_dist=("N", 0.0, 0.5),
                                  residual_dist=("N", 0.0, 1.0), weight_dist=("N", 1.0, 0.1), eps=1e-5, seed=24)
    parts, resid, weight, _ = _to_cuda(over)
    with pytest.raises(ar.ARError) as e:
        ar.ar_residual_rmsnorm_noalloc(parts, resid, weight, over.eps, out=torch.empty_like(resid),
                                       residual_out=torch.empty_like(resid))
    assert e.value.status == ar.AR_ERR_WORKSPACE


def test_noalloc_at_the_limit_of_a_prefill_shape():
    # R=2 bf16 rows of 8192: 16 chunks of 512 vectors a row, so 16384 tokens
    # fill the 1 MiB scratch.  Both outputs are compared bit for bit with the
    # two-shot call on every row, and with the oracle on sampled rows.
    T, H = 16384, 8192
    assert ar.ar_workspace_size_rows(2, H, T, ar.AR_BF16) == ar.AR_NOALLOC_SCRATCH_BYTES
    f = workloads.fused_inputs(2, T, H, "bf16", partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                               bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=25,
                               device="cuda")
    new = _noalloc(f, f.partials, f.residual, f.weight, f.bias)
    old = _existing(f, f.partials, f.residual, f.weight, f.bias)
    torch.cuda.synchronize()
    assert torch.equal(new[1].view(torch.int16), old[1].view(torch.int16)), "residual_out differs"
    assert torch.equal(new[0].view(torch.int16), old[0].view(torch.int16)), "out differs"
    g = torch.Generator().manual_seed(25)
    rows = torch.cat([torch.randint(0, T, (192,), generator=g), torch.arange(T - 64, T)])
    sub = workloads.FusedInputs(2, rows.numel(), H, "bf16", f.eps, [p[rows.cuda()].cpu() for p in f.partials],
                                f.residual[rows.cuda()].cpu(), f.weight.cpu(), f.bias.cpu())
    _compare(sub, (new[0][rows.cuda()], new[1][rows.cuda()]), (old[0][rows.cuda()], old[1][rows.cuda()]))

    parts = [p[:1].expand(T + 1, H).contiguous() for p in f.partials]
    resid = f.residual[:1].expand(T + 1, H).contiguous()
    with pytest.raises(ar.ARError) as e:
        ar.ar_residual_rmsnorm_noalloc(parts, resid, f.weight, f.eps, out=torch.empty_like(resid),
                                       residual_out=torch.empty_like(resid))
    assert e.value.status == ar.AR_ERR_WORKSPACE
