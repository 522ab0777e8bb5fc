"""Pins for the CPU oracle: each test ties it to something other than itself.

- rounding: numpy's direct binary64 -> binary16 / binary32 conversions, and a
  brute-force nearest-value search over every bf16 / fp16 pattern;
- decoding: numpy / torch views of all 65536 16-bit patterns;
- the sum: math.fsum (exact) followed by brute-force rounding;
- the fused op: a hand-computed worked example (tests/golden/hand_h8.json),
  closed forms (H=1 and H=2 rows), the RMS invariant, scale invariance,
  row independence, bias placement, permutation invariance, R=1 identity and
  the eps=0 special case against numpy's vector norm;
- the norm on its own (or_rmsnorm): the same worked example, the RMS closed
  form, numpy's vector norm at eps=0, scale invariance and row permutation.
"""
import json
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.bruteforce import nearest, table16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_h8.json")
TD = workloads.DTYPES


def _t(vals, dtype):
    return torch.tensor(vals, dtype=torch.float64).to(TD[dtype]).contiguous()


# ---------------------------------------------------------------- rounding

def _sample_doubles(rng, lo_exp, hi_exp, count):
    out = []
    for _ in range(count):
        e = rng.uniform(lo_exp, hi_exp)
        out.append(rng.choice((-1.0, 1.0)) * 2.0 ** e)
    return out


def test_round_fp16_matches_numpy_direct_conversion():
    rng = random.Random(1)
    xs = _sample_doubles(rng, -30, 17, 6000)
    vals, _, _ = table16("fp16")
    for _ in range(3000):                      # exact midpoints and their neighbours
        j = rng.randrange(len(vals) - 1)
        mid = (vals[j] + vals[j + 1]) / 2
        xs += [mid, math.nextafter(mid, math.inf), math.nextafter(mid, -math.inf)]
    xs += [65504.0, 65519.999, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -24, -0.0, 1e-300]
    got = np.array([oracle.round_bits(x, "fp16") for x in xs], dtype=np.uint32)
    with np.errstate(over="ignore"):             # 65520 and up round to infinity, as intended
        want = np.array(xs, dtype=np.float64).astype(np.float16).view(np.uint16).astype(np.uint32)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(xs[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_round_fp32_matches_numpy_cast():
    rng = random.Random(2)
    xs = _sample_doubles(rng, -152, 129, 6000)
    f = np.array(_sample_doubles(rng, -149, 127, 3000), dtype=np.float32)
    g = np.nextafter(f, np.float32(np.inf))
    mids = (f.astype(np.float64) + g.astype(np.float64)) / 2
    xs += mids.tolist() + [math.nextafter(m, math.inf) for m in mids.tolist()]
    got = np.array([oracle.round_bits(x, "fp32") for x in xs], dtype=np.uint32)
    with np.errstate(over="ignore"):
        want = np.array(xs, dtype=np.float64).astype(np.float32).view(np.uint32)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(xs[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_round_16bit_matches_bruteforce_nearest(dtype):
    rng = random.Random(3)
    lo, hi = (-136, 129) if dtype == "bf16" else (-26, 17)
    xs = _sample_doubles(rng, lo, hi, 1500)
    vals, _, _ = table16(dtype)
    for _ in range(700):
        j = rng.randrange(len(vals) - 1)
        mid = (vals[j] + vals[j + 1]) / 2
        xs += [mid, math.nextafter(mid, math.inf)]
    for x in xs:
        assert oracle.round_value(x, dtype) == nearest(x, dtype), x


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_decode_all_16bit_patterns(dtype):
    pats = np.arange(65536, dtype=np.uint16)
    if dtype == "fp16":
        want = pats.view(np.float16).astype(np.float64)
    else:
        want = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_bits(int(b), dtype) for b in pats])
    both_nan = np.isnan(got) & np.isnan(want)
    assert np.all((got == want) | both_nan)
    assert np.all(np.signbit(got[~both_nan]) == np.signbit(want[~both_nan]))


# ---------------------------------------------------------------- the sum

@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("R", [1, 2, 3, 8, 16])
def test_sum_is_exact_sum_rounded_once(dtype, R):
    n = 300
    g = torch.Generator().manual_seed(R * 7 + len(dtype))
    parts = []
    for r in range(R):
        scale = 10.0 ** (r % 4 - 2)            # mixed magnitudes: exposes order/rounding errors
        parts.append((torch.randn(n, generator=g, dtype=torch.float64) * scale).to(TD[dtype]).contiguous())
    if R >= 2:                                 # exact cancellation in a few places
        parts[1][:10] = -parts[0][:10]
    out = oracle.sum(parts, dtype).to(torch.float64).numpy()
    cols = [p.to(torch.float64).numpy() for p in parts]
    for i in range(n):
        exact = sum((Fraction(c[i]) for c in cols), Fraction(0))
        assert out[i] == nearest(exact, dtype), (i, out[i], float(exact))
    fs = np.array([math.fsum(c[i] for c in cols) for i in range(n)])
    assert np.allclose(out, fs, rtol=2.0 ** -7, atol=0)


def test_sum_R1_is_identity_bytes():
    for dtype in ("fp32", "fp16", "bf16"):
        p = workloads.draw(("N", 0.0, 1.0), 1000, dtype, seed=5, k=0)
        out = oracle.sum([p], dtype)
        assert torch.equal(out.view(torch.uint8 if dtype == "fp32" else torch.int16),
                           p.view(torch.uint8 if dtype == "fp32" else torch.int16))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_sum_permutation_invariant(dtype):
    inp = workloads.sum_inputs(8, 4096, dtype, ("N", 0.0, 1.0 / 8), seed=3)
    a = oracle.sum(inp.partials, dtype)
    perm = [inp.partials[i] for i in (5, 2, 7, 0, 1, 6, 3, 4)]
    b = oracle.sum(perm, dtype)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------- fused op

def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_hand_worked_example_exact(dtype):
    d = _golden()
    p0, p1 = _t(d["p0"], dtype), _t(d["p1"], dtype)
    out, res_out, inv = oracle.residual_rmsnorm(
        [p0, p1], _t(d["bias"], dtype), _t(d["residual"], dtype), _t(d["weight"], dtype),
        d["eps"], dtype)
    assert out.to(torch.float64).tolist() == d["expected_out"]
    assert res_out.to(torch.float64).tolist() == d["expected_residual_out"]
    assert inv.tolist() == [0.5, 0.25]
    s = oracle.sum([p0, p1], dtype)
    assert s.to(torch.float64).tolist() == d["expected_sum"]


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_hand_worked_example_small_eps(dtype):
    """Same rows with eps = float(1e-6): out = x*w/sqrt(mean_sq + eps), mean_sq = 3 and 15 by hand."""
    d = _golden()
    eps_f = float(np.float32(1e-6))
    out, res_out, _ = oracle.residual_rmsnorm(
        [_t(d["p0"], dtype), _t(d["p1"], dtype)], _t(d["bias"], dtype),
        _t(d["residual"], dtype), _t(d["weight"], dtype), 1e-6, dtype)
    import decimal
    decimal.getcontext().prec = 60
    for t, ms in enumerate(d["expected_mean_sq"]):
        root = (decimal.Decimal(ms) + decimal.Decimal(eps_f)).sqrt()
        for j in range(8):
            xw = decimal.Decimal(d["expected_residual_out"][t][j]) * decimal.Decimal(d["weight"][j])
            y = Fraction(xw / root)
            assert rounded_within_binary64(out[t, j].item(), y, dtype), (t, j)
    assert res_out.to(torch.float64).tolist() == d["expected_residual_out"]


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_single_element_rows_give_sign_times_weight(dtype):
    """H=1, eps=0: out = x / |x| * w = sign(x) * w, exactly."""
    inp = workloads.fused_inputs(3, 64, 1, dtype, partial_dist=("N", 0.0, 1.0),
                                 residual_dist=("N", 0.0, 1.0), bias_dist=("N", 0.0, 1.0),
                                 weight_dist=("N", 1.0, 1.0), eps=0.0, seed=11)
    out, res_out, _ = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, 0.0, dtype)
    x = res_out.to(torch.float64).flatten()
    w = inp.weight.to(torch.float64).item()
    for t in range(64):
        if x[t] != 0:
            assert out[t, 0].item() == math.copysign(1.0, x[t].item()) * w


def rounded_within_binary64(got: float, exact: Fraction, dtype: str) -> bool:
    """got is the correctly rounded value of `exact`, or -- only when `exact`
    lies within binary64 error (2^-50 relative: three binary64 roundings) of a
    rounding boundary -- the neighbour on the other side of that boundary."""
    want = nearest(exact, dtype)
    if got == want:
        return True
    lo, hi = sorted((Fraction(got), Fraction(want)))
    mid = (lo + hi) / 2
    return abs(exact - mid) <= abs(exact) * Fraction(1, 2 ** 50) and nearest(mid, dtype) in (got, want)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_two_element_closed_form(dtype):
    """x = (c, 7c), eps=0: mean square 25c^2, so out = sign(c) * (w0/5, 7*w1/5),
    correctly rounded (checked for many random weights)."""
    rows = [0.5, -3.0, 0.125, 96.0]
    res = _t([[c, 7 * c] for c in rows], dtype)
    zero = torch.zeros_like(res)
    g = torch.Generator().manual_seed(31)
    for trial in range(60):
        w = (torch.randn(2, generator=g, dtype=torch.float64) * 2).to(TD[dtype]).contiguous()
        w0, w1 = (Fraction(v) for v in w.to(torch.float64).tolist())
        out, _, _ = oracle.residual_rmsnorm([zero], None, res, w, 0.0, dtype)
        for t, c in enumerate(rows):
            s = 1 if c > 0 else -1
            assert rounded_within_binary64(out[t, 0].item(), s * w0 / 5, dtype), (trial, t)
            assert rounded_within_binary64(out[t, 1].item(), s * w1 * 7 / 5, dtype), (trial, t)


def test_rms_of_normalised_rows_closed_form():
    """weight=1: mean(out^2) = ms/(ms+eps).  Rows scaled so that ms is near eps."""
    T, H, eps = 6, 256, 1e-6
    g = torch.Generator().manual_seed(9)
    scales = torch.tensor([1e-4, 3e-4, 1e-3, 1e-2, 1.0, 30.0], dtype=torch.float64)
    res = (torch.randn(T, H, generator=g, dtype=torch.float64) * scales[:, None]).float().contiguous()
    zero = torch.zeros_like(res)
    w = torch.ones(H, dtype=torch.float32)
    out, res_out, _ = oracle.residual_rmsnorm([zero], None, res, w, eps, "fp32")
    x = res_out.double().numpy()
    y = out.double().numpy()
    ms = (x ** 2).mean(axis=1)
    ratio = ms / (ms + float(np.float32(eps)))
    got = (y ** 2).mean(axis=1)
    assert np.allclose(got, ratio, rtol=1e-6, atol=0), (got, ratio)
    assert ratio.min() < 0.1 and ratio.max() > 0.999     # eps matters in some rows, not in others


def test_eps_zero_unit_weight_is_vector_normalisation():
    """eps=0, w=1: out = x / ||x||_2 * sqrt(H) (numpy's norm)."""
    inp = workloads.pr1(seed=4)
    w = torch.ones(64, dtype=torch.float32)
    out, res_out, _ = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, w, 0.0, "fp32")
    x = res_out.double().numpy()
    want = x / np.linalg.norm(x, axis=1, keepdims=True) * math.sqrt(64)
    assert np.allclose(out.double().numpy(), want, rtol=2.0 ** -22, atol=0)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_scale_invariance(dtype):
    """All additive inputs * 2^k and eps * 4^k: out unchanged, residual_out * 2^k (exact)."""
    inp = workloads.fused_inputs(4, 5, 48, dtype, partial_dist=("N", 0.0, 0.25),
                                 residual_dist=("N", 0.0, 1.0), bias_dist=("N", 0.0, 0.1),
                                 weight_dist=("N", 1.0, 0.1), eps=1e-3, seed=21)
    k = 3
    eps = float(np.float32(1e-3))
    o1, r1, _ = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, eps, dtype)
    sc = lambda t: (t.to(torch.float64) * 2 ** k).to(TD[dtype]).contiguous()  # noqa: E731 (exact)
    o2, r2, _ = oracle.residual_rmsnorm([sc(p) for p in inp.partials], sc(inp.bias), sc(inp.residual),
                                        inp.weight, eps * 4 ** k, dtype)
    assert torch.equal(o1, o2)
    assert torch.equal(r1.to(torch.float64) * 2 ** k, r2.to(torch.float64))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_rows_are_independent(dtype):
    inp = workloads.fused_inputs(3, 7, 40, dtype, partial_dist=("N", 0.0, 1.0),
                                 residual_dist=("N", 0.0, 1.0), bias_dist=("N", 0.0, 0.1),
                                 weight_dist=("N", 1.0, 0.1), eps=1e-5, seed=8)
    out, res_out, inv = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, 1e-5, dtype)
    for t in range(7):
        o, r, i1 = oracle.residual_rmsnorm([p[t:t + 1].contiguous() for p in inp.partials], inp.bias,
                                           inp.residual[t:t + 1].contiguous(), inp.weight, 1e-5, dtype)
        assert torch.equal(o[0], out[t]) and torch.equal(r[0], res_out[t]) and i1[0] == inv[t]


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_residual_out_is_sum_of_all_terms(dtype):
    """residual_out = sum(partials, bias broadcast once, residual) = the plain sum of R+2 terms."""
    inp = workloads.fused_inputs(4, 6, 32, dtype, partial_dist=("N", 0.0, 0.25),
                                 residual_dist=("N", 0.0, 4.0), bias_dist=("N", 0.0, 0.02),
                                 weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=12)
    _, res_out, _ = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, 1e-6, dtype)
    terms = [p.contiguous() for p in inp.partials] + [inp.bias.expand(6, 32).contiguous(), inp.residual]
    assert torch.equal(res_out, oracle.sum(terms, dtype))
    _, no_bias, _ = oracle.residual_rmsnorm(inp.partials, None, inp.residual, inp.weight, 1e-6, dtype)
    zero_bias = torch.zeros_like(inp.bias)
    _, zb, _ = oracle.residual_rmsnorm(inp.partials, zero_bias, inp.residual, inp.weight, 1e-6, dtype)
    assert torch.equal(no_bias, zb)
    assert not torch.equal(no_bias, res_out)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_fused_permutation_invariant(dtype):
    inp = workloads.decode_r8(3, seed=2) if dtype == "bf16" else workloads.tp_decode(3, seed=2)
    a = oracle.residual_rmsnorm(inp.partials, inp.bias, inp.residual, inp.weight, inp.eps, dtype)
    b = oracle.residual_rmsnorm(inp.partials[::-1], inp.bias, inp.residual, inp.weight, inp.eps, dtype)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_sum_signed_zero_passthrough(dtype):
    """tpSize=1 is a passthrough, so a lone -0 stays -0; -0 + -0 is -0 (IEEE)."""
    neg = torch.full((16,), -0.0, dtype=TD[dtype])
    one = oracle.sum([neg], dtype)
    two = oracle.sum([neg, neg.clone()], dtype)
    assert torch.all(torch.signbit(one)) and torch.all(torch.signbit(two))
    mixed = oracle.sum([neg, torch.zeros(16, dtype=TD[dtype])], dtype)
    assert not torch.any(torch.signbit(mixed))        # -0 + +0 = +0 (round to nearest)


# ---------------------------------------------------------------- the norm on its own

@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_rmsnorm_hand_worked_example_exact(dtype):
    """The golden rows x (already summed by hand), eps = 1: out and the per-row factor are exact."""
    d = _golden()
    out, inv = oracle.rmsnorm(_t(d["expected_residual_out"], dtype), _t(d["weight"], dtype), d["eps"], dtype)
    assert out.to(torch.float64).tolist() == d["expected_out"]
    assert inv.tolist() == [0.5, 0.25]


def test_rmsnorm_rms_closed_form():
    """weight = 1: mean(out^2) = ms / (ms + eps) for every row, from tiny to large rows."""
    T, H, eps = 6, 512, 1e-6
    g = torch.Generator().manual_seed(31)
    scales = torch.tensor([1e-4, 3e-4, 1e-3, 1e-2, 1.0, 30.0], dtype=torch.float64)
    x = (torch.randn(T, H, generator=g, dtype=torch.float64) * scales[:, None]).float().contiguous()
    out, _ = oracle.rmsnorm(x, torch.ones(H, dtype=torch.float32), eps, "fp32")
    xv, yv = x.double().numpy(), out.double().numpy()
    ms = (xv ** 2).mean(axis=1)
    ratio = ms / (ms + float(np.float32(eps)))
    assert np.allclose((yv ** 2).mean(axis=1), ratio, rtol=1e-6, atol=0)
    assert ratio.min() < 0.1 and ratio.max() > 0.999


def test_rmsnorm_eps_zero_is_vector_normalisation():
    """eps = 0, weight = 1: out = x / ||x||_2 * sqrt(H), with numpy's norm."""
    g = torch.Generator().manual_seed(32)
    x = torch.randn(7, 96, generator=g).contiguous()
    out, _ = oracle.rmsnorm(x, torch.ones(96), 0.0, "fp32")
    xv = x.double().numpy()
    want = xv / np.linalg.norm(xv, axis=1, keepdims=True) * math.sqrt(96)
    assert np.allclose(out.double().numpy(), want, rtol=2.0 ** -22, atol=0)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_rmsnorm_scale_and_row_permutation(dtype):
    """x * 2^k with eps * 4^k leaves out unchanged; permuting rows permutes out."""
    g = torch.Generator().manual_seed(33)
    x = torch.randn(9, 40, generator=g, dtype=torch.float64).to(TD[dtype]).contiguous()
    w = (1.0 + 0.1 * torch.randn(40, generator=g, dtype=torch.float64)).to(TD[dtype]).contiguous()
    eps = float(np.float32(1e-3))
    o1, _ = oracle.rmsnorm(x, w, eps, dtype)
    o2, _ = oracle.rmsnorm((x.to(torch.float64) * 8).to(TD[dtype]).contiguous(), w, eps * 64, dtype)
    assert torch.equal(o1.view(torch.uint8), o2.view(torch.uint8))
    perm = torch.tensor([4, 0, 8, 2, 6, 1, 7, 3, 5])
    o3, _ = oracle.rmsnorm(x[perm].contiguous(), w, eps, dtype)
    assert torch.equal(o3.view(torch.uint8), o1[perm].contiguous().view(torch.uint8))
