"""Brute-force helpers that pin the oracle without sharing its code.

Rounding here is done by enumerating every finite value of the 16-bit formats
(decoded by numpy / torch, not by the oracle) and picking the nearest one with
exact rational arithmetic; ties go to the value with an even bit pattern.
"""
from __future__ import annotations

import bisect
import math
from fractions import Fraction
from functools import lru_cache

import numpy as np
import torch


@lru_cache(maxsize=None)
def table16(dtype: str):
    """Sorted finite values of fp16 or bf16, their bit patterns, and the
    overflow sentinel 2^(emax+1) standing for +inf."""
    pats = np.arange(65536, dtype=np.uint16)
    if dtype == "fp16":
        vals = pats.view(np.float16).astype(np.float64)
        inf_at = 2.0 ** 16
    elif dtype == "bf16":
        vals = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
        inf_at = 2.0 ** 128
    else:
        raise ValueError(dtype)
    keep = {}
    for v, b in zip(vals.tolist(), pats.tolist()):
        if math.isfinite(v) and v not in keep:   # +0 first; -0 maps to the same key
            keep[v] = b
    order = sorted(keep)
    return order, [keep[v] for v in order], inf_at


def nearest16(x, dtype: str) -> float:
    """Nearest fp16/bf16 value to the real number x (float or Fraction), ties to even."""
    xf = Fraction(x)
    if xf < 0:
        return -nearest16(-xf, dtype) if xf != 0 else 0.0
    vals, bits, inf_at = table16(dtype)
    top = vals[-1]
    if xf >= Fraction(top):
        half = (Fraction(inf_at) - Fraction(top)) / 2
        if xf - Fraction(top) < half:
            return top
        return math.inf                   # the tie goes to the even pattern (inf)
    i = bisect.bisect_left(vals, float(xf))
    cands = [j for j in (i - 1, i, i + 1) if 0 <= j < len(vals)]
    best = min(cands, key=lambda j: (abs(Fraction(vals[j]) - xf), bits[j] & 1))
    return vals[best]


def nearest32(x) -> float:
    """Nearest binary32 value to the real number x, ties to even (three candidates)."""
    xf = Fraction(x)
    f = np.float32(float(xf))
    cands = {float(f), float(np.nextafter(f, np.float32(np.inf))), float(np.nextafter(f, np.float32(-np.inf)))}
    cands = [c for c in cands if math.isfinite(c)]

    def key(c):
        bits = int(np.float32(c).view(np.uint32))
        return (abs(Fraction(c) - xf), bits & 1)
    return min(cands, key=key)


def nearest(x, dtype: str) -> float:
    return nearest32(x) if dtype == "fp32" else nearest16(x, dtype)
