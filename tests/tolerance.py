"""GPU-vs-oracle comparison rules.

fp32 outputs: |gpu - oracle| <= 1e-5 * row scale, the scale being the largest
|oracle| value of the row.  A flat reduce-only tensor is one row; a [T, H]
output (residual_out, out) is T rows of `hidden` values.

fp16 / bf16 outputs: |gpu - oracle| <= 2 ulp(oracle) + floor, where the floor
is what fp32 accumulation in a fixed order may lose before the one rounding,
with R the number of partials:
    floor(sum, residual_out) = (R + 2) * 2^-24 * sum of |terms|
    floor(out)               = floor(residual_out) * |w| * inv_rms
(terms = the R partials, plus bias and residual for the fused call).  The
fp32 sum of R + 2 terms in a fixed order is off the exact sum by at most
(R + 1) * 2^-24 * sum |terms|, so R + 2 bounds it with room to spare.  Away
from cancellation the floor is far below an ulp; near cancellation it is
what lets a correct fp32 result differ from the exactly rounded one.

Strict 2-ulp report.  Every check counts the elements beyond a strict 2 ulp
and records them in REPORT (printed at the end of the pytest run).  Such an
element must be explained by the floor: with x' the fp32 sum and x the exact
one, |rnd(x') - rnd(x)| <= ulp + |x' - x| (the two half-ulp roundings, one
binade apart at most), so beyond 2 ulp the accumulation error |x' - x| is
above half an ulp.  The checks assert that the floor is above 0.45 ulp at
every such element (0.5 for sums; for `out` the products and the inverse
RMS add a relative error below 1e-5, about 0.05 ulp at most): a strict
violation anywhere else is a failure even when it is within the bound.
"""
from __future__ import annotations

import numpy as np
import torch

_FMT = {"fp16": (11, -14), "bf16": (8, -126)}
U32 = 2.0 ** -24

# One record per check: what was compared and how many elements exceeded a
# strict 2 ulp.  The test that made the check is named by CURRENT_TEST,
# which tests/conftest.py sets for every test.
REPORT: list = []
CURRENT_TEST = ""


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of ``dtype`` at |v| (the subnormal quantum near zero)."""
    p, emin = _FMT[dtype]
    _, e = np.frexp(np.abs(v))
    lead = np.maximum(e.astype(np.int64) - 1, emin)
    return np.ldexp(1.0, (lead - (p - 1)).astype(np.int64))


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy().reshape(-1)


def _kind(what: str, fused_out: bool) -> str:
    return "out" if fused_out else ("residual_out" if "residual_out" in what else "sum")


def _record(what: str, kind: str, dtype: str, n: int, err: np.ndarray, u: np.ndarray, floor: np.ndarray,
            explained: float) -> dict:
    """Counts strict 2-ulp violations, checks each lies where the floor is above `explained` ulp, records."""
    strict = err > 2 * u
    n_strict = int(strict.sum())
    ratio = floor[strict] / u[strict] if n_strict else np.zeros(0)
    rec = {"test": CURRENT_TEST, "what": what, "kind": kind, "dtype": dtype, "elements": int(n),
           "strict_violations": n_strict, "max_err_ulp": float((err / u).max(initial=0.0)),
           "min_floor_ulp_at_violations": float(ratio.min()) if n_strict else None}
    REPORT.append(rec)
    assert np.all(ratio > explained), (
        f"{what}: {int((ratio <= explained).sum())} elements beyond a strict 2 ulp where the fp32 "
        f"accumulation floor is below {explained} ulp (not explained by cancellation)")
    return rec


def check_sum(gpu: torch.Tensor, ref: torch.Tensor, terms, dtype: str, what: str = "sum", *, R: int,
              hidden: int | None = None):
    """Checks an R-way sum, or a residual_out (terms: the R partials, bias and residual).

    `hidden` makes the fp32 row scale per row of that many values (a [T, H]
    residual_out); without it the tensor is one row (a flat sum).
    """
    g, o = _f64(gpu), _f64(ref)
    assert g.shape == o.shape, (g.shape, o.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = np.abs(g - o)
    if dtype == "fp32":
        if hidden is not None:
            scale = np.repeat(np.abs(o).reshape(-1, hidden).max(axis=1), hidden) if o.size else o
        else:
            scale = np.max(np.abs(o)) if o.size else 0.0
        bad = err > 1e-5 * scale
        assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1e-5*row scale, max err {err.max()}"
        rec = {"test": CURRENT_TEST, "what": what, "kind": _kind(what, False), "dtype": dtype,
               "elements": int(o.size), "max_err": float(err.max(initial=0.0)), "strict_violations": 0}
        REPORT.append(rec)
        return rec
    abs_sum = np.zeros_like(o)
    for t in terms:
        abs_sum += np.abs(_f64(t))
    floor = (R + 2) * U32 * abs_sum
    u = ulp(o, dtype)
    bad = err > 2 * u + floor
    assert not bad.any(), (f"{what}: {bad.sum()} elements beyond 2 ulp + floor; first at "
                           f"{np.nonzero(bad)[0][:5]}, gpu {g[bad][:5]}, oracle {o[bad][:5]}")
    return _record(what, _kind(what, False), dtype, o.size, err, u, floor, 0.5)


def check_fused_out(gpu: torch.Tensor, ref: torch.Tensor, terms, weight: torch.Tensor,
                    inv_rms: np.ndarray, dtype: str, hidden: int, what: str = "out", *, R: int):
    """Checks the normalised output against the oracle, row by row (R: the number of partials)."""
    g, o = _f64(gpu).reshape(-1, hidden), _f64(ref).reshape(-1, hidden)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = np.abs(g - o)
    if dtype == "fp32":
        scale = np.max(np.abs(o), axis=1, keepdims=True)
        bad = err > 1e-5 * scale
        assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1e-5*row scale, max err {err.max()}"
        rec = {"test": CURRENT_TEST, "what": what, "kind": "out", "dtype": dtype, "elements": int(o.size),
               "max_err": float(err.max(initial=0.0)), "strict_violations": 0}
        REPORT.append(rec)
        return rec
    abs_sum = np.zeros_like(o)
    for t in terms:
        a = np.abs(_f64(t))
        abs_sum += a.reshape(-1, hidden) if a.size == o.size else a.reshape(1, hidden)
    w = np.abs(_f64(weight)).reshape(1, hidden)
    floor = (R + 2) * U32 * abs_sum * w * inv_rms.reshape(-1, 1)
    u = ulp(o, dtype)
    bad = err > 2 * u + floor
    assert not bad.any(), (f"{what}: {bad.sum()} elements beyond 2 ulp + floor; rows "
                           f"{np.nonzero(bad)[0][:5]}, gpu {g[bad][:5]}, oracle {o[bad][:5]}")
    return _record(what, "out", dtype, o.size, err.reshape(-1), u.reshape(-1), floor.reshape(-1), 0.45)


def summary() -> dict:
    """Totals of REPORT per (dtype, output): elements checked and strict 2-ulp violations."""
    tot: dict = {}
    for r in REPORT:
        k = f"{r['dtype']} {r['kind']}"
        t = tot.setdefault(k, {"checks": 0, "elements": 0, "strict_violations": 0, "max_err_ulp": 0.0,
                               "min_floor_ulp_at_violations": None})
        t["checks"] += 1
        t["elements"] += r["elements"]
        t["strict_violations"] += r["strict_violations"]
        if "max_err_ulp" in r:
            t["max_err_ulp"] = max(t["max_err_ulp"], r["max_err_ulp"])
        m = r.get("min_floor_ulp_at_violations")
        if m is not None:
            cur = t["min_floor_ulp_at_violations"]
            t["min_floor_ulp_at_violations"] = m if cur is None else min(cur, m)
    return tot
