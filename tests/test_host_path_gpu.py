"""ar_residual_rmsnorm_host: the fused call on host tensors, copies pipelined
through device staging.  Its outputs must match the oracle like the device
call's, residual_out bit for bit with the device call, for row counts that
split into several chunks with a ragged last one, a single chunk, chunk
sizes of one row, and a last chunk cut into shrinking pieces."""
import pytest
import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tests import tolerance as tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    ar.lib()


def _pin(t):
    return None if t is None else t.contiguous().pin_memory()


def _run_host(inp, chunk, strategy="AUTO"):
    parts = [_pin(p.reshape(inp.tokens, inp.hidden)) for p in inp.partials]
    res, w, b = _pin(inp.residual), _pin(inp.weight), _pin(inp.bias)
    out = torch.empty_like(res).pin_memory()
    rout = torch.empty_like(res).pin_memory()
    staging = torch.empty(ar.ar_host_staging_size(inp.R, inp.hidden, min(chunk, inp.tokens),
                                                  ar.dtype_code(res.dtype)), dtype=torch.uint8, device="cuda")
    ar.ar_residual_rmsnorm_host(parts, res, w, inp.eps, staging, out, rout, bias=b, chunk_tokens=chunk,
                                strategy=strategy)
    torch.cuda.current_stream().synchronize()
    return out, rout


def _check(inp, out, rout):
    ref = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, inp.eps, inp.dtype)
    terms = [p.reshape(inp.tokens, inp.hidden) for p in inp.partials]
    if inp.bias is not None:
        terms.append(inp.bias.expand(inp.tokens, inp.hidden).contiguous())
    terms.append(inp.residual)
    tol.check_sum(rout, ref[1], terms, inp.dtype, "residual_out", R=inp.R, hidden=inp.hidden)
    tol.check_fused_out(out, ref[0], terms, inp.weight, ref[2], inp.dtype, inp.hidden, "out", R=inp.R)
    d_out, d_rout = ar.ar_residual_rmsnorm([p.cuda() for p in inp.partials], inp.residual.cuda(), inp.weight.cuda(),
                                           inp.eps, bias=None if inp.bias is None else inp.bias.cuda())
    assert torch.equal(d_rout.cpu().view(torch.uint8), rout.view(torch.uint8))


@pytest.mark.parametrize("chunk", [1, 8, 16, 64])
def test_host_path_chunks(chunk):
    inp = workloads.fused_inputs(8, 37, 8192, "bf16", partial_dist=("N", 0.0, 0.125), residual_dist=("N", 0.0, 4.0),
                                 bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=chunk)
    _check(inp, *_run_host(inp, chunk))


def test_host_path_decode_shape_no_bias_and_strategies():
    inp = workloads.tp_decode(5, seed=3)
    for s in ("ONESHOT", "TWOSHOT", "AUTO"):
        _check(inp, *_run_host(inp, 2, s))
    inp = workloads.decode_r8(9, seed=4)
    _check(inp, *_run_host(inp, 4))


def test_host_path_repeated_calls_share_nothing_stale():
    a = workloads.tp_prefill(tokens=24, hidden=4096, seed=5)
    b = workloads.tp_prefill(tokens=24, hidden=4096, seed=6)
    for inp in (a, b, a):
        _check(inp, *_run_host(inp, 5))


def test_host_path_shrinking_tail():
    """The last chunk's rows go in halves until at most 128 are left: 1000 rows in chunks of 700 are pieces
    of 700, 150, 75 and 75 rows (ragged, and more pieces than staging buffers)."""
    inp = workloads.fused_inputs(4, 1000, 1024, "bf16", partial_dist=("N", 0.0, 0.25), residual_dist=("N", 0.0, 4.0),
                                 bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=21)
    _check(inp, *_run_host(inp, 700))


def test_host_path_full_prefill_sampled_rows():
    """The end-to-end configuration bench.py times: 8192 x 8192 R=8 bf16 with bias on pinned host buffers,
    4096-row chunks (one whole chunk, then pieces of 2048, 1024, 512, 256, 128 and 128 rows), AUTO;
    sampled rows, the pieces' first and last among them, against the oracle, and residual_out bit for bit
    with the device call."""
    inp = workloads.tp_prefill(seed=3)
    T, H = inp.tokens, inp.hidden
    out, rout = _run_host(inp, 4096)
    g = torch.Generator().manual_seed(11)
    edges = [0, 4095, 4096, 6143, 6144, 7167, 7168, 7679, 7680, 7935, 7936, 8063, 8064, T - 1]
    rows = sorted(set(edges + torch.randint(0, T, (16,), generator=g).tolist()))
    ridx = torch.tensor(rows)
    sub = workloads.FusedInputs(inp.R, len(rows), H, inp.dtype, inp.eps,
                                [p[ridx].contiguous() for p in inp.partials], inp.residual[ridx].contiguous(),
                                inp.weight, inp.bias)
    _check(sub, out[ridx].contiguous(), rout[ridx].contiguous())
