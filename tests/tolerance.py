"""GPU-vs-oracle comparison rules.

fp32 outputs: |gpu - oracle| <= 1e-5 * row scale, the scale being the largest
|oracle| value of the row (a flat reduce-only tensor is one row).

fp16 / bf16 outputs: |gpu - oracle| <= 2 ulp(oracle) + floor, where the floor
is what fp32 accumulation in a fixed order may lose before the one rounding:
    floor(residual_out) = (R + 2) * 2^-24 * sum of |terms|
    floor(out)          = floor(residual_out) * |w| * inv_rms
Away from cancellation the floor is far below an ulp; near cancellation it is
what makes a correct fp32 result legitimately differ from the exact one.
"""
from __future__ import annotations

import numpy as np
import torch

_FMT = {"fp16": (11, -14), "bf16": (8, -126)}


def ulp(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of ``dtype`` at |v| (the subnormal quantum near zero)."""
    p, emin = _FMT[dtype]
    _, e = np.frexp(np.abs(v))
    lead = np.maximum(e.astype(np.int64) - 1, emin)
    return np.ldexp(1.0, (lead - (p - 1)).astype(np.int64))


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy().reshape(-1)


def check_sum(gpu: torch.Tensor, ref: torch.Tensor, terms, dtype: str, what: str = "sum"):
    """Checks an R-way sum (or a residual_out, with its R+2 terms)."""
    g, o = _f64(gpu), _f64(ref)
    assert g.shape == o.shape, (g.shape, o.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = np.abs(g - o)
    if dtype == "fp32":
        scale = np.max(np.abs(o)) if o.size else 0.0
        bad = err > 1e-5 * scale
        assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1e-5*scale, max err {err.max()}"
        return {"max_err": float(err.max(initial=0.0)), "strict_violations": 0}
    abs_sum = np.zeros_like(o)
    for t in terms:
        abs_sum += np.abs(_f64(t))
    floor = (len(terms) + 2) * 2.0 ** -24 * abs_sum
    tol = 2 * ulp(o, dtype) + floor
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements beyond 2 ulp + floor; first at "
                           f"{np.nonzero(bad)[0][:5]}, gpu {g[bad][:5]}, oracle {o[bad][:5]}")
    strict = int((err > 2 * ulp(o, dtype)).sum())
    return {"max_err_ulp": float((err / ulp(o, dtype)).max(initial=0.0)), "strict_violations": strict}


def check_fused_out(gpu: torch.Tensor, ref: torch.Tensor, terms, weight: torch.Tensor,
                    inv_rms: np.ndarray, dtype: str, hidden: int, what: str = "out"):
    """Checks the normalised output against the oracle, row by row."""
    g, o = _f64(gpu).reshape(-1, hidden), _f64(ref).reshape(-1, hidden)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = np.abs(g - o)
    if dtype == "fp32":
        scale = np.max(np.abs(o), axis=1, keepdims=True)
        bad = err > 1e-5 * scale
        assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1e-5*row scale, max err {err.max()}"
        return {"max_err": float(err.max(initial=0.0)), "strict_violations": 0}
    abs_sum = np.zeros_like(o)
    for t in terms:
        a = np.abs(_f64(t))
        abs_sum += a.reshape(-1, hidden) if a.size == o.size else a.reshape(1, hidden)
    w = np.abs(_f64(weight)).reshape(1, hidden)
    floor = (len(terms) + 2) * 2.0 ** -24 * abs_sum * w * inv_rms.reshape(-1, 1)
    tol = 2 * ulp(o, dtype) + floor
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements beyond 2 ulp + floor; rows "
                           f"{np.nonzero(bad)[0][:5]}, gpu {g[bad][:5]}, oracle {o[bad][:5]}")
    strict = int((err > 2 * ulp(o, dtype)).sum())
    return {"max_err_ulp": float((err / ulp(o, dtype)).max(initial=0.0)), "strict_violations": strict}
