"""Seeded random shapes through every strategy, against the oracle.

The fixed workloads cover the measured configurations; this draws rank
counts 1..16, all three element types, rows from 1 to 16384 elements (packed
and element-wise), 1 to 3000 rows (enough to reach the bulk-copy-fed kernel
by rule) and optional bias, and checks out and residual_out of each call
(and of the Lamport-style call, where it takes the shape) against the oracle
with the usual tolerance.  Sizes are bounded so the oracle
stays within seconds."""
import random

import pytest
import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
import workloads
from tests import tolerance as tol

pytestmark = pytest.mark.gpu


def _cases(count=32, seed=2024):
    rng = random.Random(seed)
    out = []
    while len(out) < count:
        R = rng.choice([1, 2, 3, 4, 5, 8, 12, 16])
        dt = rng.choice(["fp32", "fp16", "bf16"])
        H = rng.choice([rng.randint(1, 200), 8 * rng.randint(1, 2048), rng.randint(1, 16384)])
        T = rng.choice([rng.randint(1, 8), rng.randint(1, 300), rng.randint(2048, 3000)])
        if R * T * H > 24_000_000:
            continue
        out.append((R, dt, H, T, rng.random() < 0.6, rng.choice(["ONESHOT", "TWOSHOT", "AUTO"]), rng.randint(0, 9999)))
    return out


def _kernel_cases(count=10, seed=77):
    """Draws aimed at the persistent bulk-copy-fed kernel (packed rows, 2048+ rows) and the row-split
    cluster kernel (packed rows of 1024+ vectors, a few rows)."""
    rng = random.Random(seed)
    out = []
    while len(out) < 2 * count:
        R = rng.choice([1, 2, 3, 4, 6, 8, 16])
        dt = rng.choice(["fp32", "fp16", "bf16"])
        lanes = 4 if dt == "fp32" else 8
        if len(out) % 2 == 0:
            H, T = lanes * rng.randint(4, 1024), rng.randint(2048, 3000)
        else:
            H, T = lanes * rng.randint(1024, 2048), rng.randint(1, 8)
        if R * T * H > 24_000_000:
            continue
        out.append((R, dt, H, T, rng.random() < 0.5, rng.choice(["ONESHOT", "AUTO"]), rng.randint(0, 9999)))
    return out


@pytest.mark.parametrize("R,dt,H,T,has_bias,strategy,seed", _cases() + _kernel_cases())
def test_random_shape_matches_oracle(R, dt, H, T, has_bias, strategy, seed):
    f = workloads.fused_inputs(R, T, H, dt, partial_dist=("N", 0.0, 1.0 / R), residual_dist=("N", 0.0, 4.0),
                               bias_dist=("N", 0.0, 0.02) if has_bias else None, weight_dist=("N", 1.0, 0.05),
                               eps=1e-6, seed=seed)
    parts = [p.cuda() for p in f.partials]
    try:
        out, res = ar.ar_residual_rmsnorm(parts, f.residual.cuda(), f.weight.cuda(), f.eps,
                                          bias=None if f.bias is None else f.bias.cuda(), strategy=strategy)
    except ar.ARError as e:   # only a forced ONESHOT on a row no one-shot kernel holds may be refused
        assert strategy == "ONESHOT" and e.status == ar.AR_ERR_UNSUPPORTED
        return
    torch.cuda.synchronize()
    ref_out, ref_res, inv = oracle.residual_rmsnorm(f.partials, f.bias, f.residual, f.weight, f.eps, dt)
    terms = [p.reshape(T, H) for p in f.partials]
    if f.bias is not None:
        terms.append(f.bias.expand(T, H).contiguous())
    terms.append(f.residual)
    tol.check_sum(res.cpu(), ref_res, terms, dt, "residual_out", R=R, hidden=H)
    tol.check_fused_out(out.cpu(), ref_out, terms, f.weight, inv, dt, H, "out", R=R)
    # and the plain sum of the same partials
    s = ar.ar_sum(parts, strategy="TWOSHOT" if strategy == "TWOSHOT" else "ONESHOT")
    torch.cuda.synchronize()
    tol.check_sum(s.cpu(), oracle.sum(f.partials, dt), f.partials, dt, "sum", R=R)
    # and the Lamport-style call, wherever it takes the shape
    if ar.ar_lamport_supported(R, H, T, workloads.DTYPES[dt]) is not None:
        lo, lr = ar.ar_residual_rmsnorm_lamport(parts, f.residual.cuda(), f.weight.cuda(), f.eps,
                                                bias=None if f.bias is None else f.bias.cuda())
        torch.cuda.synchronize()
        tol.check_sum(lr.cpu(), ref_res, terms, dt, "Lamport residual_out", R=R, hidden=H)
        tol.check_fused_out(lo.cpu(), ref_out, terms, f.weight, inv, dt, H, "Lamport out", R=R)
        assert ar.ar_device_status() == ar.AR_OK
