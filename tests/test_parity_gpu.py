"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Covers the five measured workloads (PR1 fp32, TP decode fp16 R=2, R=8 bf16
decode / small prefill, reduce-only R=4 fp16 up to 2^27 elements, TP prefill
R=8 bf16 8192x8192), every strategy, and the edge cases: empty inputs, ragged
tails, element-wise (misaligned / odd hidden) paths, generic rank counts,
R=1 passthrough, aliasing, determinism, guard bands and unmodified inputs.
Full-size workloads are checked on sampled rows or elements that the oracle
computes one by one.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tensor_allreduce_residual_gb300 import _build
from tests import tolerance as tol

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_h8.json")
STRATS = ["ONESHOT", "TWOSHOT", "AUTO"]
TD = workloads.DTYPES


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    assert torch.cuda.is_available()
    _build.build()
    ar.lib()   # raises if the library did not build: no fallback exists


def dev(t):
    return None if t is None else t.cuda()


def bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


def run_fused(inp, strategy, **kw):
    out, res = ar.ar_residual_rmsnorm([dev(p) for p in inp.partials], dev(inp.residual), dev(inp.weight),
                                      inp.eps, bias=dev(inp.bias), strategy=strategy, **kw)
    torch.cuda.synchronize()
    return out.cpu(), res.cpu()


def terms_of(inp):
    T, H = inp.tokens, inp.hidden
    t = [p.reshape(T, H) for p in inp.partials]
    if inp.bias is not None:
        t.append(inp.bias.expand(T, H).contiguous())
    t.append(inp.residual)
    return t


def check_fused(inp, out, res, ref=None):
    if ref is None:
        ref = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, inp.eps, inp.dtype)
    o_out, o_res, inv = ref
    terms = terms_of(inp)
    r1 = tol.check_sum(res, o_res, terms, inp.dtype, "residual_out", R=inp.R, hidden=inp.hidden)
    r2 = tol.check_fused_out(out, o_out, terms, inp.weight, inv, inp.dtype, inp.hidden, "out", R=inp.R)
    return r1, r2


# ------------------------------------------------------------ worked example

@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("strategy", STRATS)
def test_hand_worked_example_exact(dtype, strategy):
    d = json.load(open(GOLDEN))
    mk = lambda v: torch.tensor(v, dtype=torch.float64).to(TD[dtype]).cuda()  # noqa: E731
    out, res = ar.ar_residual_rmsnorm([mk(d["p0"]), mk(d["p1"])], mk(d["residual"]), mk(d["weight"]),
                                      d["eps"], bias=mk(d["bias"]), strategy=strategy)
    s = ar.ar_sum([mk(d["p0"]), mk(d["p1"])], strategy=strategy)
    assert out.double().tolist() == d["expected_out"]
    assert res.double().tolist() == d["expected_residual_out"]
    assert s.double().tolist() == d["expected_sum"]


# ------------------------------------------------------------ the five workloads

@pytest.mark.parametrize("strategy", STRATS)
def test_pr1_fused_and_sum(strategy):
    inp = workloads.pr1(seed=0)
    out, res = run_fused(inp, strategy)
    check_fused(inp, out, res)
    s = ar.ar_sum([dev(p) for p in inp.partials], strategy=strategy).cpu()
    tol.check_sum(s, oracle.sum(inp.partials, "fp32"), inp.partials, "fp32", R=inp.R)


def test_tp_decode_all_token_counts():
    for T in workloads.TP_DECODE_TOKENS:
        inp = workloads.tp_decode(T, seed=0)
        out, res = run_fused(inp, "ONESHOT")
        check_fused(inp, out, res)


@pytest.mark.parametrize("T", workloads.DECODE_R8_TOKENS)
@pytest.mark.parametrize("strategy", STRATS)
def test_decode_r8(T, strategy):
    inp = workloads.decode_r8(T, seed=0)
    out, res = run_fused(inp, strategy)
    check_fused(inp, out, res)


@pytest.mark.parametrize("n", [2 ** k for k in range(9, 21)])
def test_reduce_only_full_compare(n):
    inp = workloads.reduce_only(n, seed=0)
    ref = oracle.sum(inp.partials, "fp16")
    outs = []
    for strategy in STRATS:
        s = ar.ar_sum([dev(p) for p in inp.partials], strategy=strategy).cpu()
        tol.check_sum(s, ref, inp.partials, "fp16", R=inp.R)
        outs.append(s)
    assert all(torch.equal(bits(outs[0]), bits(o)) for o in outs[1:])


@pytest.mark.parametrize("n", [2 ** 21, 2 ** 24, 2 ** 27])
def test_reduce_only_large_sampled(n):
    inp = workloads.reduce_only(n, seed=0)
    g = torch.Generator().manual_seed(n)
    idx = torch.cat([torch.randint(0, n, (1 << 16,), generator=g), torch.arange(n - 1024, n)])
    ref = oracle.sum([p[idx].contiguous() for p in inp.partials], "fp16")
    parts = [dev(p) for p in inp.partials]
    outs = []
    for strategy in STRATS:
        s = ar.ar_sum(parts, strategy=strategy)
        torch.cuda.synchronize()
        outs.append(s[idx.cuda()].cpu())
        del s
    for o in outs:
        tol.check_sum(o, ref, [p[idx] for p in inp.partials], "fp16", R=inp.R)
    assert all(torch.equal(bits(outs[0]), bits(o)) for o in outs[1:])


@pytest.mark.parametrize("strategy", STRATS)
def test_tp_prefill_sampled_rows(strategy):
    inp = _prefill_inputs()
    T, H = inp.tokens, inp.hidden
    g = torch.Generator().manual_seed(7)
    rows = sorted(set([0, 1, T // 2, T - 1] + torch.randint(0, T, (20,), generator=g).tolist()))
    parts = [dev(p) for p in inp.partials]
    out, res = ar.ar_residual_rmsnorm(parts, dev(inp.residual), dev(inp.weight), inp.eps,
                                      bias=dev(inp.bias), strategy=strategy)
    torch.cuda.synchronize()
    ridx = torch.tensor(rows)
    sub = workloads.FusedInputs(inp.R, len(rows), H, inp.dtype, inp.eps,
                                [p[ridx].contiguous() for p in inp.partials], inp.residual[ridx].contiguous(),
                                inp.weight, inp.bias)
    check_fused(sub, out[ridx.cuda()].cpu(), res[ridx.cuda()].cpu())


_PREFILL = {}


def _prefill_inputs():
    if "inp" not in _PREFILL:
        _PREFILL["inp"] = workloads.tp_prefill(seed=0)
    return _PREFILL["inp"]


def test_tp_prefill_residual_out_identical_across_strategies():
    inp = _prefill_inputs()
    parts = [dev(p) for p in inp.partials]
    res = []
    for strategy in STRATS:
        _, r = ar.ar_residual_rmsnorm(parts, dev(inp.residual), dev(inp.weight), inp.eps,
                                      bias=dev(inp.bias), strategy=strategy)
        res.append(r)
    torch.cuda.synchronize()
    assert all(torch.equal(bits(res[0]), bits(r)) for r in res[1:])
    _PREFILL.clear()


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("R", [1, 2, 3, 5, 8, 16])
def test_sum_ragged_sizes_and_rank_counts(dtype, R):
    for n in [1, 7, 8, 9, 31, 4095, 4097, 65537]:
        inp = workloads.sum_inputs(R, n, dtype, ("N", 0.0, 1.0), seed=n + R)
        ref = oracle.sum(inp.partials, dtype)
        outs = [ar.ar_sum([dev(p) for p in inp.partials], strategy=s).cpu() for s in STRATS]
        for o in outs:
            tol.check_sum(o, ref, inp.partials, dtype, R=R)
            assert torch.equal(bits(outs[0]), bits(o))


def test_empty_inputs_are_noops():
    e = torch.empty(0, dtype=torch.float16, device="cuda")
    out = ar.ar_sum([e, e.clone()])
    assert out.numel() == 0
    res = torch.empty(0, 64, dtype=torch.float16, device="cuda")
    w = torch.ones(64, dtype=torch.float16, device="cuda")
    for s in STRATS:
        o, r = ar.ar_residual_rmsnorm([res, res.clone()], res, w, 1e-6, strategy=s)
        assert o.numel() == 0 and r.numel() == 0


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_r1_passthrough_is_a_byte_copy(dtype):
    p = workloads.draw(("N", 0.0, 1.0), 100003, dtype, seed=1, k=0)
    p[:5] = -0.0
    pd = dev(p)
    for s in STRATS:
        out = ar.ar_sum([pd], strategy=s)
        assert torch.equal(bits(out.cpu()), bits(p))
    same = ar.ar_sum([pd], out=pd)           # in place: nothing launched, nothing changed
    assert torch.equal(bits(same.cpu()), bits(p))


def _offset_view(t, k=1):
    """t's values in a CUDA buffer that starts k elements past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device="cuda")
    v = buf[k:k + t.numel()].view(t.shape)
    v.copy_(t.cuda())
    return v


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_misaligned_pointers_take_the_elementwise_path(dtype):
    inp = workloads.sum_inputs(4, 10007, dtype, ("U", -1.0, 1.0), seed=3)
    ref = oracle.sum(inp.partials, dtype)
    parts = [_offset_view(p, 1 + r % 3) for r, p in enumerate(inp.partials)]
    out = _offset_view(torch.zeros(10007, dtype=TD[dtype]), 2)
    ar.ar_sum(parts, out=out)
    tol.check_sum(out.cpu(), ref, inp.partials, dtype, R=inp.R)

    f = workloads.fused_inputs(2, 9, 256, dtype, partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                               bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=4)
    for s in STRATS:
        o, r = ar.ar_residual_rmsnorm([_offset_view(p) for p in f.partials], _offset_view(f.residual),
                                      _offset_view(f.weight), f.eps, bias=_offset_view(f.bias), strategy=s)
        check_fused(f, o.cpu(), r.cpu())


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("H", [1, 3, 100, 4100])
def test_hidden_not_a_multiple_of_the_vector_width(dtype, H):
    f = workloads.fused_inputs(3, 5, H, dtype, partial_dist=("N", 0.0, 0.3), residual_dist=("N", 0.0, 4.0),
                               bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-5, seed=H)
    for s in STRATS:
        out, res = run_fused(f, s)
        check_fused(f, out, res)


@pytest.mark.parametrize("R", [1, 3, 5, 16])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_fused_generic_rank_counts(R, dtype):
    f = workloads.fused_inputs(R, 17, 2048, dtype, partial_dist=("N", 0.0, 1.0 / R),
                               residual_dist=("N", 0.0, 4.0), bias_dist=None,
                               weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=R)
    for s in STRATS:
        out, res = run_fused(f, s)
        check_fused(f, out, res)


def test_row_too_long_for_one_shot():
    """A 40960-wide bf16 row (5120 vectors): at 3 tokens the row-split cluster kernel holds it (one
    row over 8 blocks); at 16 tokens no one-shot kernel does, and only the two-shot path runs."""
    few = workloads.fused_inputs(2, 3, 40960, "bf16", partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                                 bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=9)
    assert ar.ar_query_launch(2, 40960, 3, ar.AR_BF16, "ONESHOT")["kernel_name"] == "k_fused_oneshot_cluster"
    for s in STRATS:
        out, res = run_fused(few, s)
        check_fused(few, out, res)
    many = workloads.fused_inputs(2, 16, 40960, "bf16", partial_dist=("N", 0.0, 0.5), residual_dist=("N", 0.0, 4.0),
                                  bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=10)
    with pytest.raises(ar.ARError) as e:
        run_fused(many, "ONESHOT")
    assert e.value.status == ar.AR_ERR_UNSUPPORTED
    for s in ["TWOSHOT", "AUTO"]:
        out, res = run_fused(many, s)
        check_fused(many, out, res)


@pytest.mark.parametrize("strategy", STRATS)
def test_aliasing_out_on_partial_and_residual_out_on_residual(strategy):
    f = workloads.decode_r8(8, seed=5)
    ref = oracle.residual_rmsnorm(f.partials, f.bias, f.residual, f.weight, f.eps, f.dtype)
    parts = [dev(p) for p in f.partials]
    resid = dev(f.residual)
    out, res = ar.ar_residual_rmsnorm(parts, resid, dev(f.weight), f.eps, out=parts[3], residual_out=resid,
                                      strategy=strategy)
    torch.cuda.synchronize()
    assert out.data_ptr() == parts[3].data_ptr() and res.data_ptr() == resid.data_ptr()
    check_fused(f, out.cpu(), res.cpu(), ref)
    s_in = workloads.reduce_only(4099, seed=2)
    ref_s = oracle.sum(s_in.partials, "fp16")
    sp = [dev(p) for p in s_in.partials]
    ar.ar_sum(sp, out=sp[0], strategy=strategy)
    tol.check_sum(sp[0].cpu(), ref_s, s_in.partials, "fp16", R=s_in.R)


def test_determinism_across_runs_and_strategies():
    f = workloads.decode_r8(64, seed=3)
    parts = [dev(p) for p in f.partials]
    by = {}
    for s in STRATS:
        runs = [ar.ar_residual_rmsnorm(parts, dev(f.residual), dev(f.weight), f.eps, strategy=s) for _ in range(3)]
        for o, r in runs[1:]:
            assert torch.equal(bits(o), bits(runs[0][0])) and torch.equal(bits(r), bits(runs[0][1]))
        by[s] = runs[0]
    assert torch.equal(bits(by["ONESHOT"][1]), bits(by["TWOSHOT"][1]))
    assert torch.equal(bits(by["AUTO"][1]), bits(by["ONESHOT"][1]))


def test_allreduce_dispatch_matches_direct_calls():
    f = workloads.tp_decode(7, seed=6)
    parts = [dev(p) for p in f.partials]
    direct = ar.ar_sum(parts)
    out = torch.empty_like(parts[0])
    ar.ar_allreduce(ar.make_params(parts, out), ar.AR_FUSION_NONE)
    assert torch.equal(bits(out), bits(direct))
    o1, r1 = ar.ar_residual_rmsnorm(parts, dev(f.residual), dev(f.weight), f.eps, bias=dev(f.bias), strategy="TWOSHOT")
    o2, r2 = torch.empty_like(o1), torch.empty_like(r1)
    ws = torch.empty(ar.ar_workspace_size(2, o1.numel(), ar.AR_FP16), dtype=torch.uint8, device="cuda")
    p = ar.make_params(parts, o2, bias=dev(f.bias), residual=dev(f.residual), weight=dev(f.weight), eps=f.eps,
                       hidden=f.hidden, residual_out=r2, workspace=ws)
    ar.ar_allreduce(p, ar.AR_FUSION_RESIDUAL_RMS_NORM, "TWOSHOT")
    torch.cuda.synchronize()
    assert torch.equal(bits(o1), bits(o2)) and torch.equal(bits(r1), bits(r2))


@pytest.mark.parametrize("strategy,R,T,H,kernel", [
    ("ONESHOT", 4, 33, 1000, None), ("TWOSHOT", 4, 33, 1000, None), ("AUTO", 4, 33, 1000, None),
    # the persistent bulk-copy-fed kernel (ragged last chunk: 1000 vectors in chunks of 512) and the
    # row-split cluster kernel (ragged slices: 1025 vectors over 8 blocks)
    ("AUTO", 8, 2100, 8000, "k_fused_oneshot_tma"), ("AUTO", 8, 3, 8200, "k_fused_oneshot_cluster")])
def test_guard_bands_untouched_and_inputs_unchanged(strategy, R, T, H, kernel):
    f = workloads.fused_inputs(R, T, H, "bf16", partial_dist=("N", 0.0, 0.25), residual_dist=("N", 0.0, 4.0),
                               bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=13)
    if kernel is not None:
        assert ar.ar_query_launch(R, H, T, ar.AR_BF16, strategy)["kernel_name"] == kernel
    n, G = f.tokens * f.hidden, 4096
    bufs = []
    views = []
    for _ in range(2):
        b = torch.full((n + 2 * G,), 0, dtype=torch.int16, device="cuda")
        b.fill_(-23131)                         # 0xA5A5 pattern
        bufs.append(b)
        views.append(b[G:G + n].view(torch.bfloat16).view(f.tokens, f.hidden))
    ws_need = ar.ar_workspace_size_rows(R, f.hidden, f.tokens, ar.AR_BF16)
    ws = torch.full((ws_need + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    parts = [dev(p) for p in f.partials]
    before = [p.clone() for p in parts] + [dev(f.residual)]
    resid = before[-1].clone()
    ar.ar_residual_rmsnorm(parts, resid, dev(f.weight), f.eps, bias=dev(f.bias), out=views[0],
                           residual_out=views[1], intermediate=ws[G:G + ws_need], strategy=strategy)
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.all(b[:G] == -23131) and torch.all(b[G + n:] == -23131)
    assert torch.all(ws[:G] == 0xA5) and torch.all(ws[G + ws_need:] == 0xA5)
    for p, q in zip(parts + [resid], before):
        assert torch.equal(bits(p), bits(q))
    check_fused(f, views[0].cpu(), views[1].cpu())


def test_rms_of_normalised_rows_on_gpu():
    T, H = 16, 4096
    f = workloads.fused_inputs(2, T, H, "fp32", partial_dist=("N", 0.0, 1e-7), residual_dist=("N", 0.0, 1e-6),
                               bias_dist=None, weight_dist=("N", 1.0, 0.0), eps=1e-6, seed=21)
    for s in STRATS:
        out, res = run_fused(f, s)
        x = res.double().numpy()
        ms = (x ** 2).mean(axis=1)
        want = ms / (ms + float(np.float32(1e-6)))
        got = (out.double().numpy() ** 2).mean(axis=1)
        assert np.allclose(got, want, rtol=1e-5, atol=0)


# ---------------------------------------------------------------- the norm on its own, and the unfused route

def _norm_rows(T, H, dtype, seed, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(T, H, generator=g, dtype=torch.float64) * scale).to(TD[dtype]).contiguous()
    w = (1.0 + 0.05 * torch.randn(H, generator=g, dtype=torch.float64)).to(TD[dtype]).contiguous()
    return x, w


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("T,H", [(1, 4096), (7, 8192), (300, 64), (33, 16384), (5, 100), (3, 3), (129, 1024),
                                 # 1024 rows or more, ragged rows (H=8000), and rows of under a warp (H=64)
                                 (1500, 8192), (1024, 8000), (1100, 1000), (1030, 64), (1024, 16384)])
def test_rmsnorm_matches_oracle(dtype, T, H):
    x, w = _norm_rows(T, H, dtype, seed=T * 7 + H)
    eps = 1e-5
    out = ar.ar_rmsnorm(x.cuda(), w.cuda(), eps)
    torch.cuda.synchronize()
    ref, inv = oracle.rmsnorm(x, w, eps, dtype)
    tol.check_fused_out(out.cpu(), ref, [x], w, inv, dtype, H, "rmsnorm out", R=1)


def test_rmsnorm_in_place_and_limits():
    x, w = _norm_rows(17, 8192, "bf16", seed=3)
    ref, _ = oracle.rmsnorm(x, w, 1e-6, "bf16")
    xd = x.cuda()
    ar.ar_rmsnorm(xd, w.cuda(), 1e-6, out=xd)
    torch.cuda.synchronize()
    assert torch.equal(xd.cpu().view(torch.int16), ar.ar_rmsnorm(x.cuda(), w.cuda(), 1e-6).cpu().view(torch.int16))
    tol.check_fused_out(xd.cpu(), ref, [x], w, oracle.rmsnorm(x, w, 1e-6, "bf16")[1], "bf16", 8192, "in place",
                        R=1)
    big = torch.zeros(1, 16385, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ar.ARError) as e:
        ar.ar_rmsnorm(big, torch.ones(16385, dtype=torch.bfloat16, device="cuda"), 1e-6)
    assert e.value.status == ar.AR_ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype,R,T,H,has_bias", [("bf16", 8, 40, 8192, True), ("fp16", 2, 9, 4096, True),
                                                  ("fp32", 2, 4, 64, False)])
def test_unfused_route_matches_oracle_composition(dtype, R, T, H, has_bias):
    """ar_sum, then ar_residual_rmsnorm with the rounded sum as its one partial: the oracle composed the same way."""
    inp = workloads.fused_inputs(R, T, H, dtype, partial_dist=("N", 0.0, 1.0 / R), residual_dist=("N", 0.0, 4.0),
                                 bias_dist=("N", 0.0, 0.02) if has_bias else None, weight_dist=("N", 1.0, 0.05),
                                 eps=1e-6, seed=T)
    s = ar.ar_sum([dev(p) for p in inp.partials])
    out, res = ar.ar_residual_rmsnorm([s], dev(inp.residual), dev(inp.weight), inp.eps, bias=dev(inp.bias))
    torch.cuda.synchronize()
    s_ref = oracle.sum(inp.partials, dtype)
    tol.check_sum(s.cpu(), s_ref, [p.reshape(T, H) for p in inp.partials], dtype, "sum", R=R)
    step2 = workloads.FusedInputs(1, T, H, dtype, inp.eps, [s_ref.reshape(T, H)], inp.residual, inp.weight, inp.bias)
    check_fused(step2, out.cpu(), res.cpu())


@pytest.mark.parametrize("config", [ar.AR_CONFIG_USE_MEMCPY, ar.AR_CONFIG_RESIDUAL_RMS_NORM,
                                    ar.AR_CONFIG_USE_MEMCPY | ar.AR_CONFIG_RESIDUAL_RMS_NORM])
@pytest.mark.parametrize("strategy", ["ONESHOT", "TWOSHOT"])
def test_allreduce_config_flags_match_allreduce(config, strategy):
    """USE_MEMCPY (stage the partials in the registered workspace first) and the RESIDUAL_RMS_NORM
    flag give the same bits as ar_allreduce with the matching fusion op."""
    f = workloads.fused_inputs(8, 33, 8192, "bf16", partial_dist=("N", 0.0, 0.125), residual_dist=("N", 0.0, 4.0),
                               bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=config)
    parts = [dev(p) for p in f.partials]
    fused = bool(config & ar.AR_CONFIG_RESIDUAL_RMS_NORM)
    outs = []
    for cfg in (None, config):
        out, rout = torch.empty_like(parts[0]), torch.empty_like(parts[0])
        ws = torch.empty(ar.ar_config_workspace_size(8, out.numel(), 8192, ar.AR_BF16), dtype=torch.uint8,
                         device="cuda")
        p = ar.make_params(parts, out, bias=dev(f.bias), residual=dev(f.residual), weight=dev(f.weight), eps=f.eps,
                           hidden=8192, residual_out=rout, workspace=ws)
        op = ar.AR_FUSION_RESIDUAL_RMS_NORM if fused else ar.AR_FUSION_NONE
        if cfg is None:
            ar.ar_allreduce(p, op, strategy)
        else:
            ar.ar_allreduce_config(p, ar.AR_FUSION_NONE, strategy, cfg)
        torch.cuda.synchronize()
        outs.append((out.cpu(), rout.cpu() if fused else None))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    if fused:
        assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))
    if fused:
        check_fused(f, *outs[1])
    else:
        tol.check_sum(outs[1][0], oracle.sum(f.partials, "bf16"), [q.reshape(33, 8192) for q in f.partials], "bf16",
                      R=f.R)


@pytest.mark.parametrize("R,dtype,H,T", [(16, "bf16", 8192, 5), (16, "bf16", 8192, 64), (16, "bf16", 8192, 300),
                                         (3, "fp16", 4096, 64), (3, "fp16", 4096, 2100),
                                         (4, "fp16", 8192, 100), (4, "fp16", 8192, 700)])
def test_measured_rank_counts_through_auto(R, dtype, H, T):
    """R=16 and R=3 rows through the kernels the measured table picks for them (row-split cluster
    kernel at few tokens, bulk-copy-fed persistent kernel with R outside the compiled rank counts),
    and R=4 fp16 rows of 8192 through the table's register shapes on both sides of 512 tokens."""
    f = workloads.fused_inputs(R, T, H, dtype, partial_dist=("N", 0.0, 1.0 / R), residual_dist=("N", 0.0, 4.0),
                               bias_dist=("N", 0.0, 0.02), weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=R * T)
    kernel = ar.ar_query_launch(R, H, T, ar.dtype_code(TD[dtype]))["kernel_name"]
    assert kernel in ("k_fused_oneshot_cluster", "k_fused_oneshot_tma", "k_fused_oneshot"), kernel
    out, res = run_fused(f, "AUTO")
    check_fused(f, out, res)


@pytest.mark.parametrize("strategy", STRATS)
def test_permuted_partials_stay_within_tolerance(strategy):
    """The sum is accumulated in rank order, so permuting the partials changes the fp32 rounding, but
    never beyond the tolerance around the (permutation-invariant) exact result; residual_out and out
    of the permuted call are checked against the oracle of the original order."""
    f = workloads.decode_r8(64, seed=12)
    ref = oracle.residual_rmsnorm(f.partials, f.bias, f.residual, f.weight, f.eps, f.dtype)
    for perm in ([7, 6, 5, 4, 3, 2, 1, 0], [3, 0, 6, 1, 7, 4, 2, 5]):
        g = workloads.FusedInputs(f.R, f.tokens, f.hidden, f.dtype, f.eps, [f.partials[k] for k in perm],
                                  f.residual, f.weight, f.bias)
        out, res = run_fused(g, strategy)
        check_fused(f, out, res, ref)
