"""Parity of the Lamport-style fused call (ar_residual_rmsnorm_lamport) with
the CPU oracle, and the protocol's own properties:

- the buffer is left holding the empty marker after every call, so one
  buffer serves a sequence of calls;
- partials full of -0.0 (the marker's value) still arrive;
- residual_out equals the other strategies' bit for bit, up to the sign of
  exact zeros;
- aliasing, guard bands and unmodified inputs;
- the full-size prefill workload, checked on sampled rows.

The bounded waits are covered by test_lamport_timeout (a child process).
"""
import os
import subprocess
import sys

import pytest
import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tensor_allreduce_residual_gb300 import _build
from tests import tolerance as tol

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MARKER = {"fp32": (torch.int32, -(1 << 31)), "fp16": (torch.int16, -(1 << 15)), "bf16": (torch.int16, -(1 << 15))}


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    assert torch.cuda.is_available()
    _build.build()
    ar.lib()


def dev(t):
    return None if t is None else t.cuda()


def terms_of(inp):
    T, H = inp.tokens, inp.hidden
    t = [p.reshape(T, H) for p in inp.partials]
    if inp.bias is not None:
        t.append(inp.bias.expand(T, H).contiguous())
    t.append(inp.residual)
    return t


def check(inp, out, res, what=""):
    o_out, o_res, inv = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, inp.eps,
                                                inp.dtype)
    terms = terms_of(inp)
    tol.check_sum(res, o_res, terms, inp.dtype, "residual_out " + what, R=inp.R, hidden=inp.hidden)
    tol.check_fused_out(out, o_out, terms, inp.weight, inv, inp.dtype, inp.hidden, "out " + what, R=inp.R)


def all_marker(buf, dtype, nbytes):
    it, m = MARKER[dtype]
    v = buf[:nbytes].view(it)
    return bool(torch.all(v == m))


PROGRESS = 4096   # the buffer starts with the blocks' progress words


def slots_empty(buf, dtype):
    """The slots and the exchange area (everything after the progress words) hold the marker."""
    return all_marker(buf[PROGRESS:], dtype, buf.numel() - PROGRESS)


def run(inp, buf=None, **kw):
    out, res = ar.ar_residual_rmsnorm_lamport([dev(p) for p in inp.partials], dev(inp.residual), dev(inp.weight),
                                              inp.eps, bias=dev(inp.bias), buffer=buf, **kw)
    torch.cuda.synchronize()
    return out, res


def _inputs(R, T, H, dtype, bias=True, seed=0):
    return workloads.fused_inputs(R, T, H, dtype, partial_dist=("N", 0.0, 1.0 / R), residual_dist=("N", 0.0, 4.0),
                                  bias_dist=("N", 0.0, 0.02) if bias else None, weight_dist=("N", 1.0, 0.05),
                                  eps=1e-6, seed=seed)


@pytest.mark.parametrize("R,T,H,dtype,bias", [
    (2, 4, 64, "fp32", True),          # PR1's shape
    (2, 1, 4096, "fp16", True), (2, 7, 4096, "fp16", True), (2, 32, 4096, "fp16", True),   # TP decode
    (8, 1, 8192, "bf16", False), (8, 8, 8192, "bf16", False), (8, 64, 8192, "bf16", False),
    (8, 256, 8192, "bf16", False),     # R=8 decode / small prefill
    (3, 5, 1000, "fp32", True),        # runtime rank count, ragged row (250 vectors)
    (16, 3, 2048, "bf16", True), (1, 9, 512, "fp16", False), (4, 33, 8200, "bf16", True),
    (2, 2, 16384, "bf16", True),       # the longest row class (8 vectors a thread)
    (5, 300, 768, "fp16", True),       # rows in groups of several per block, blocks striding
    (4, 3000, 1024, "bf16", True),     # more rows than the ring holds: ring rows reused within the call
    (2, 20000, 64, "fp32", True),      # the same with 8 rows a group
    # separate push and reduce warps in blocks of 1024 threads (two vectors a thread, 512 a row):
    (3, 1100, 8192, "fp16", True),     # runtime rank count
    (4, 1500, 4096, "fp32", True),     # fp32 rows
    (8, 1200, 6000, "bf16", False),    # ragged row: 750 vectors over 512 threads
])
def test_parity_with_oracle(R, T, H, dtype, bias):
    inp = _inputs(R, T, H, dtype, bias, seed=R * 100 + T)
    buf = ar.lamport_buffer(R, H, T, workloads.DTYPES[dtype])
    out, res = run(inp, buf)
    check(inp, out.cpu(), res.cpu(), f"R{R} T{T} H{H} {dtype}")
    assert slots_empty(buf, dtype)
    assert ar.ar_device_status() == ar.AR_OK


def test_one_buffer_serves_a_sequence_of_calls():
    """The buffer is emptied by every call: three calls on different inputs, one buffer, all correct."""
    R, T, H = 8, 64, 8192
    buf = ar.lamport_buffer(R, H, T, torch.bfloat16)
    for seed in (1, 2, 3):
        inp = _inputs(R, T, H, "bf16", bias=False, seed=seed)
        out, res = run(inp, buf)
        check(inp, out.cpu(), res.cpu(), f"call {seed}")
        assert slots_empty(buf, "bf16")
    # a smaller call on the same (larger) buffer uses its front part only
    inp = _inputs(R, 3, H, "bf16", bias=False, seed=4)
    out, res = run(inp, buf)
    check(inp, out.cpu(), res.cpu(), "smaller call")
    assert slots_empty(buf, "bf16")


def test_ring_reuse_over_a_sequence_of_calls():
    """Rows beyond the ring reuse its rows within a call (each push waits for its row to be empty
    again); three such calls in a row on one buffer, all correct, the buffer left empty after each."""
    R, T, H = 8, 2500, 2048
    buf = ar.lamport_buffer(R, H, T, torch.bfloat16)
    assert buf.numel() < R * T * H * 2          # the slots hold fewer rows than the call
    for seed in (5, 6, 7):
        inp = _inputs(R, T, H, "bf16", bias=seed != 6, seed=seed)
        out, res = run(inp, buf)
        check(inp, out.cpu(), res.cpu(), f"ring call {seed}")
        assert slots_empty(buf, "bf16")
    assert ar.ar_device_status() == ar.AR_OK


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_negative_zero_partials_arrive(dtype):
    """Elements equal to the marker's value (-0.0) are pushed as +0.0: the call completes and
    only the sign of exact-zero results can differ."""
    R, T, H = 4, 6, 1024
    inp = _inputs(R, T, H, dtype, seed=9)
    neg0 = torch.tensor(-0.0, dtype=workloads.DTYPES[dtype])
    for r in range(R):
        inp.partials[r][0].fill_(neg0)              # a whole row of -0.0 in every partial
        inp.partials[r][2, ::3] = neg0               # scattered lanes
    inp.residual[0, :16] = neg0                      # x = bias + (-0.0) in the first lanes of row 0
    out, res = run(inp)
    check(inp, out.cpu(), res.cpu(), "with -0.0 partials")
    assert ar.ar_device_status() == ar.AR_OK


def test_residual_out_matches_other_strategies():
    R, T, H = 8, 256, 8192
    inp = _inputs(R, T, H, "bf16", bias=True, seed=21)
    parts = [dev(p) for p in inp.partials]
    _, r_lam = ar.ar_residual_rmsnorm_lamport(parts, dev(inp.residual), dev(inp.weight), inp.eps,
                                              bias=dev(inp.bias))
    for s in ("ONESHOT", "TWOSHOT", "AUTO"):
        _, r = ar.ar_residual_rmsnorm(parts, dev(inp.residual), dev(inp.weight), inp.eps, bias=dev(inp.bias),
                                      strategy=s)
        torch.cuda.synchronize()
        assert torch.equal(r, r_lam)        # value equality: +0.0 == -0.0


def test_determinism_across_runs():
    inp = _inputs(8, 64, 8192, "bf16", bias=False, seed=5)
    buf = ar.lamport_buffer(8, 8192, 64, torch.bfloat16)
    runs = [tuple(t.clone() for t in run(inp, buf)) for _ in range(3)]
    for o, r in runs[1:]:
        assert torch.equal(o.view(torch.int16), runs[0][0].view(torch.int16))
        assert torch.equal(r.view(torch.int16), runs[0][1].view(torch.int16))


def test_aliasing_out_on_partial_and_residual_out_on_residual():
    f = workloads.decode_r8(8, seed=5)
    parts = [dev(p) for p in f.partials]
    resid = dev(f.residual)
    out, res = ar.ar_residual_rmsnorm_lamport(parts, resid, dev(f.weight), f.eps, out=parts[3], residual_out=resid)
    torch.cuda.synchronize()
    assert out.data_ptr() == parts[3].data_ptr() and res.data_ptr() == resid.data_ptr()
    check(f, out.cpu(), res.cpu(), "aliased")


def test_guard_bands_untouched_and_inputs_unchanged():
    R, T, H, G = 4, 33, 1000, 4096
    f = _inputs(R, T, H, "bf16", seed=13)
    n = T * H
    bufs, views = [], []
    for _ in range(2):
        b = torch.full((n + 2 * G,), -23131, dtype=torch.int16, device="cuda")   # 0xA5A5 pattern
        bufs.append(b)
        views.append(b[G:G + n].view(torch.bfloat16).view(T, H))
    need = ar.ar_lamport_buffer_size(R, H, T, torch.bfloat16)
    lam = torch.full((need + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    ar.ar_lamport_init(lam[G:G + need], torch.bfloat16)
    parts = [dev(p) for p in f.partials]
    before = [p.clone() for p in parts] + [dev(f.residual)]
    resid = before[-1].clone()
    ar.ar_residual_rmsnorm_lamport(parts, resid, dev(f.weight), f.eps, bias=dev(f.bias), out=views[0],
                                   residual_out=views[1], buffer=lam[G:G + need])
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.all(b[:G] == -23131) and torch.all(b[G + n:] == -23131)
    assert torch.all(lam[:G] == 0xA5) and torch.all(lam[G + need:] == 0xA5)
    for p, q in zip(parts + [resid], before):
        assert torch.equal(p.view(torch.int16), q.view(torch.int16))
    check(f, views[0].cpu(), views[1].cpu(), "guard bands")


def test_init_fills_ragged_sizes():
    for nbytes in (2, 14, 16, 18, 4096 + 6):
        for dtype, code in (("fp32", torch.float32), ("bf16", torch.bfloat16)):
            b = torch.full((nbytes + 32,), 0x11, dtype=torch.uint8, device="cuda")
            ar.ar_lamport_init(b[:nbytes], code)
            torch.cuda.synchronize()
            assert torch.all(b[nbytes:] == 0x11)
            whole = nbytes // 4 * 4 if dtype == "fp32" else nbytes
            if whole:
                assert all_marker(b, dtype, whole)
            if dtype == "fp32" and nbytes % 4:
                assert b[nbytes - 2].item() == 0 and b[nbytes - 1].item() == 0   # low half of -0.0f


def test_errors_raise():
    f = _inputs(2, 4, 1024, "bf16")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ar.ARError) as e:
        run(f, small)
    assert e.value.status == ar.AR_ERR_WORKSPACE
    x = torch.empty(4 * 1024 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(4, 1024)   # misaligned
    x.copy_(f.residual.cuda())
    with pytest.raises(ar.ARError) as e:
        ar.ar_residual_rmsnorm_lamport([dev(p) for p in f.partials], x, dev(f.weight), f.eps)
    assert e.value.status == ar.AR_ERR_UNSUPPORTED


def test_full_size_prefill_sampled_rows():
    """The 8192 x 8192 R=8 bf16 prefill, the bench's launch, checked on sampled rows."""
    inp = workloads.tp_prefill(seed=0)
    T, H = inp.tokens, inp.hidden
    buf = ar.lamport_buffer(inp.R, H, T, torch.bfloat16)
    out, res = run(inp, buf)
    g = torch.Generator().manual_seed(11)
    rows = sorted(set([0, 1, T // 2, T - 1] + torch.randint(0, T, (20,), generator=g).tolist()))
    ridx = torch.tensor(rows)
    sub = workloads.FusedInputs(inp.R, len(rows), H, inp.dtype, inp.eps,
                                [p[ridx].contiguous() for p in inp.partials], inp.residual[ridx].contiguous(),
                                inp.weight, inp.bias)
    check(sub, out[ridx.cuda()].cpu(), res[ridx.cuda()].cpu(), "prefill")
    assert slots_empty(buf, "bf16")
    assert ar.ar_device_status() == ar.AR_OK


@pytest.mark.parametrize("shape", ["1:0", "2:0", "4:0", "8:0", "1:4:0:2", "1:4:0:4", "1:4:0:8", "2:4:0:8",
                                   "1:0:1", "2:0:1", "4:0:1"])
def test_lamport_shape_parity(shape):
    """Every launch shape the call can take, forced through the shape override in a child process
    (third field 1: separate push and reduce warps, where the row fits them)."""
    env = dict(os.environ, AR_ONESHOT_SHAPE=shape)
    res = subprocess.run([sys.executable, "-m", "tests.lamport_shape_child"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and "lamport shape ok" in res.stdout, res.stdout[-3000:] + res.stderr[-3000:]


def test_lamport_timeout():
    """A rank whose pushes never come: every poll of its slot gives up after about a second,
    the call returns, ar_device_status reports it, and the context stays usable."""
    env = dict(os.environ, AR_TEST_LAMPORT_SKIP_RANK="1")
    res = subprocess.run([sys.executable, "-m", "tests.lamport_timeout_child"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and "lamport timeout ok" in res.stdout, res.stdout[-3000:] + res.stderr[-3000:]
