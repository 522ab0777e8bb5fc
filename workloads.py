"""Seeded synthetic inputs for the R-way reduce (+ bias + residual + RMSNorm) path.

This module is shared by the tests, the benchmark and the smoke check. It only
draws random numbers and lays them out; it holds none of the method's
arithmetic (no sums, no norms, no rounding logic of its own: the one rounding
step is torch's own dtype conversion of the drawn values, and both the CUDA
path and the oracle then read the same dtype-valued tensors).

Workload shapes follow the five configurations the method is measured on:
  * ``pr1``          R=2 fp32, T=4, H=64, U(-1,1) partials and residual.
  * ``tp_decode``    R=2 fp16, T=1..32, H=4096, N(0,1/R) partials.
  * ``decode_r8``    R=8 bf16, T in {1,8,64,256}, H=8192, no bias.
  * ``reduce_only``  R=4 fp16 U(-1,1), flat n = 2^9 .. 2^27.
  * ``tp_prefill``   R=8 bf16, T=8192, H=8192 (1 GiB of partials).

Reading of "N(a, b)": the second argument is the variance (textbook
N(mu, sigma^2)), so N(0, 1/R) partials give a unit-variance reduced sum.

Seeds: tensor k of a workload draws from ``torch.Generator().manual_seed(
seed*1000 + k)`` with k = r for partial r, 100 for the residual, 200 for the
bias and 300 for the weight.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}
# Same numeric codes as the C ABI's ar_dtype (AR_FP32=0, AR_FP16=1, AR_BF16=2).
DTYPE_CODE = {"fp32": 0, "fp16": 1, "bf16": 2}
ELEM_SIZE = {"fp32": 4, "fp16": 2, "bf16": 2}

K_RESIDUAL, K_BIAS, K_WEIGHT = 100, 200, 300


def _gen(seed: int, k: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + k)
    return g


def draw(dist: tuple, numel: int, dtype: str, seed: int, k: int, device: str = "cpu") -> torch.Tensor:
    """Draw ``numel`` values from ``dist`` and convert them to ``dtype``.

    ``dist`` is ("U", lo, hi) or ("N", mean, variance).  With device="cuda"
    the values come from torch's CUDA generator (same recipe and seeds, a
    different random stream than the CPU one); the benchmark uses it to make
    its 1.5 GB inputs quickly.
    """
    g = _gen(seed, k, device)
    kind, a, b = dist
    if kind == "U":
        v = torch.rand(numel, generator=g, dtype=torch.float32, device=device)
        v.mul_(b - a).add_(a)
    elif kind == "N":
        v = torch.randn(numel, generator=g, dtype=torch.float32, device=device)
        v.mul_(math.sqrt(b)).add_(a)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return v.to(DTYPES[dtype]).contiguous()


@dataclass
class SumInputs:
    R: int
    n: int
    dtype: str
    partials: list


@dataclass
class FusedInputs:
    R: int
    tokens: int
    hidden: int
    dtype: str
    eps: float
    partials: list           # R tensors of shape [tokens, hidden]
    residual: torch.Tensor   # [tokens, hidden]
    weight: torch.Tensor     # [hidden]
    bias: torch.Tensor | None = None  # [hidden] or None
    extra: dict = field(default_factory=dict)


def sum_inputs(R: int, n: int, dtype: str, dist=("U", -1.0, 1.0), seed: int = 0,
               device: str = "cpu") -> SumInputs:
    parts = [draw(dist, n, dtype, seed, r, device) for r in range(R)]
    return SumInputs(R, n, dtype, parts)


def fused_inputs(R: int, tokens: int, hidden: int, dtype: str, *,
                 partial_dist, residual_dist, weight_dist, bias_dist=None,
                 eps: float, seed: int = 0, device: str = "cpu") -> FusedInputs:
    n = tokens * hidden
    parts = [draw(partial_dist, n, dtype, seed, r, device).view(tokens, hidden) for r in range(R)]
    residual = draw(residual_dist, n, dtype, seed, K_RESIDUAL, device).view(tokens, hidden)
    weight = draw(weight_dist, hidden, dtype, seed, K_WEIGHT, device)
    bias = None if bias_dist is None else draw(bias_dist, hidden, dtype, seed, K_BIAS, device)
    return FusedInputs(R, tokens, hidden, dtype, eps, parts, residual, weight, bias)


# --------------------------------------------------------------------------
# The five measured configurations.
# --------------------------------------------------------------------------

def pr1(seed: int = 0) -> FusedInputs:
    """R=2 fp32, T=4, H=64; partials/residual U(-1,1), bias U(-0.1,0.1), w N(1,0.1), eps=1e-6."""
    return fused_inputs(2, 4, 64, "fp32", partial_dist=("U", -1.0, 1.0),
                        residual_dist=("U", -1.0, 1.0), bias_dist=("U", -0.1, 0.1),
                        weight_dist=("N", 1.0, 0.1), eps=1e-6, seed=seed)


def tp_decode(tokens: int, seed: int = 0, device: str = "cpu") -> FusedInputs:
    """R=2 fp16, H=4096; partials N(0,1/2), residual N(0,4), bias N(0,0.02), w N(1,0.05), eps=1e-5."""
    R = 2
    return fused_inputs(R, tokens, 4096, "fp16", partial_dist=("N", 0.0, 1.0 / R),
                        residual_dist=("N", 0.0, 4.0), bias_dist=("N", 0.0, 0.02),
                        weight_dist=("N", 1.0, 0.05), eps=1e-5, seed=seed, device=device)


def decode_r8(tokens: int, seed: int = 0, device: str = "cpu") -> FusedInputs:
    """R=8 bf16, H=8192; partials N(0,1/8), residual N(0,4), no bias, w N(1,0.05), eps=1e-6."""
    R = 8
    return fused_inputs(R, tokens, 8192, "bf16", partial_dist=("N", 0.0, 1.0 / R),
                        residual_dist=("N", 0.0, 4.0), bias_dist=None,
                        weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=seed, device=device)


def reduce_only(n: int, seed: int = 0, device: str = "cpu") -> SumInputs:
    """R=4 fp16, flat n elements, partials U(-1,1)."""
    return sum_inputs(4, n, "fp16", ("U", -1.0, 1.0), seed, device)


def tp_prefill(tokens: int = 8192, hidden: int = 8192, seed: int = 0, device: str = "cpu") -> FusedInputs:
    """R=8 bf16, T=8192, H=8192; partials N(0,1/8), residual N(0,4), bias N(0,0.02), w N(1,0.05), eps=1e-6."""
    R = 8
    return fused_inputs(R, tokens, hidden, "bf16", partial_dist=("N", 0.0, 1.0 / R),
                        residual_dist=("N", 0.0, 4.0), bias_dist=("N", 0.0, 0.02),
                        weight_dist=("N", 1.0, 0.05), eps=1e-6, seed=seed, device=device)


TP_DECODE_TOKENS = list(range(1, 33))
DECODE_R8_TOKENS = [1, 8, 64, 256]
REDUCE_ONLY_N = [2 ** k for k in range(9, 28)]


def fused_algorithmic_bytes(R: int, tokens: int, hidden: int, dtype: str, has_bias: bool) -> int:
    """Bytes one fused call must move: R partials + residual + bias + weight + two outputs."""
    s = ELEM_SIZE[dtype]
    n = tokens * hidden
    return R * n * s + n * s + (hidden * s if has_bias else 0) + hidden * s + 2 * n * s


def sum_algorithmic_bytes(R: int, n: int, dtype: str) -> int:
    """Bytes one reduce-only call must move: R partials read, one output written."""
    return (R + 1) * n * ELEM_SIZE[dtype]
