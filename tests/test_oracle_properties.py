"""Property searches over the CPU oracle's rounding and sum (hypothesis; skipped where it is absent).

Where the fixed pins sample inputs, these let hypothesis hunt for the edge cases of rounding straight
from binary64: subnormals, the overflow threshold, exact ties between neighbours, signed zeros, and sums
that cancel.  The sums are checked against their definition: the binary64 sum in rank order, rounded
once (the exact sum rounded once wherever the binary64 sum is exact).  The references are the same independent ones as in the pins: numpy's direct binary64 ->
binary16 conversion, and a brute-force nearest-value search over every 16-bit pattern (ties to even).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.bruteforce import nearest, table16

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings

TD = workloads.DTYPES
FINITE = st.floats(allow_nan=False, allow_infinity=False, width=64)


def _ties(dtype):
    """Exact midpoints between neighbouring finite values of a 16-bit type, and their neighbours."""
    vals, _, _ = table16(dtype)
    return st.integers(0, len(vals) - 2).flatmap(
        lambda j: st.sampled_from([(vals[j] + vals[j + 1]) / 2,
                                   math.nextafter((vals[j] + vals[j + 1]) / 2, math.inf),
                                   math.nextafter((vals[j] + vals[j + 1]) / 2, -math.inf)]))


@settings(max_examples=400, deadline=None)
@given(x=FINITE | _ties("fp16"))
def test_fp16_rounding_matches_numpy(x):
    with np.errstate(over="ignore"):
        want = int(np.array([x], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
    assert oracle.round_bits(x, "fp16") == want


@settings(max_examples=400, deadline=None)
@given(x=st.floats(min_value=-3.3e38, max_value=3.3e38, allow_nan=False, width=64) | _ties("bf16"))
def test_bf16_rounding_matches_bruteforce_nearest(x):
    assert oracle.round_value(x, "bf16") == nearest(x, "bf16")


@settings(max_examples=200, deadline=None)
@given(bits=st.lists(st.integers(0, 0xFFFF), min_size=1, max_size=16), dtype=st.sampled_from(["fp16", "bf16"]))
def test_sum_of_16bit_values_is_the_binary64_sum_rounded_once(bits, dtype):
    """The oracle's sum is the binary64 sum in rank order, rounded once.  Wherever that binary64 sum is
    exact (always for fp16: every value is a multiple of 2^-24 below 2^16), it is the exact sum rounded
    once.  A bf16 sum spanning more than 53 bits of range (a subnormal beside values near 2^15) is not
    exact in binary64: there the oracle keeps its binary64 sum, which can sit on a rounding tie that the
    exact sum does not (2^-133 + 16384 + 23680 is above the tie between 39936 and 40192)."""
    vals = [oracle.decode_bits(b, dtype) for b in bits]
    if any(not math.isfinite(v) for v in vals):
        return
    parts = [torch.tensor([v], dtype=torch.float64).to(TD[dtype]) for v in vals]
    got = float(oracle.sum(parts, dtype).to(torch.float64)[0])
    acc = 0.0
    for v in vals:      # binary64, rank order
        acc += v
    exact = sum((Fraction(v) for v in vals), Fraction(0))
    want = nearest(Fraction(acc), dtype)
    assert got == want or (math.isinf(got) and math.isinf(want) and (got > 0) == (want > 0))
    if Fraction(acc) == exact:
        assert want == nearest(exact, dtype) or math.isinf(want)
    if dtype == "fp16":
        assert Fraction(acc) == exact


@settings(max_examples=200, deadline=None)
@given(x=st.floats(min_value=-60000, max_value=60000, allow_nan=False, width=16))
def test_a_value_and_its_negation_sum_to_zero(x):
    a = torch.tensor([x], dtype=torch.float16)
    assert float(oracle.sum([a, -a], "fp16")[0]) == 0.0
    assert float(oracle.sum([a], "fp16")[0]) == float(a[0])
