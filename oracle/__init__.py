"""CPU oracle for the R-way reduce and the fused reduce + residual + RMSNorm.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path
(``tensor_allreduce_residual_gb300``) never imports this package, and this
package never imports the product path.

The arithmetic lives in ``ar_oracle.c`` (plain C, binary64, one rounding to
the output format, single-threaded).  This module builds it with gcc and
marshals torch CPU tensors to it; it does no arithmetic of its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ar_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libar_oracle.so")

_CODES = {"fp32": 0, "fp16": 1, "bf16": 2}
_TORCH = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}

_lib = None


def build(force: bool = False) -> str:
    """Compile ar_oracle.c into a shared library next to it (host gcc, no ISA flags)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
                    "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        lib.or_round_value.argtypes = [ctypes.c_double, ctypes.c_int]
        lib.or_round_value.restype = ctypes.c_double
        lib.or_round_bits.argtypes = [ctypes.c_double, ctypes.c_int]
        lib.or_round_bits.restype = ctypes.c_uint32
        lib.or_decode_bits.argtypes = [ctypes.c_uint32, ctypes.c_int]
        lib.or_decode_bits.restype = ctypes.c_double
        lib.or_sum.argtypes = [ctypes.POINTER(vp), ctypes.c_int, sz, ctypes.c_int, vp]
        lib.or_sum.restype = None
        lib.or_residual_rmsnorm.argtypes = [
            ctypes.POINTER(vp), ctypes.c_int, vp, vp, vp, ctypes.c_float,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
        lib.or_residual_rmsnorm.restype = None
        lib.or_rmsnorm.argtypes = [vp, vp, ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
        lib.or_rmsnorm.restype = None
        _lib = lib
    return _lib


def _check(t: torch.Tensor, dtype: str, numel: int, what: str):
    if t.device.type != "cpu" or not t.is_contiguous():
        raise ValueError(f"oracle: {what} must be a contiguous CPU tensor")
    if t.dtype != _TORCH[dtype]:
        raise ValueError(f"oracle: {what} has dtype {t.dtype}, expected {dtype}")
    if t.numel() != numel:
        raise ValueError(f"oracle: {what} has {t.numel()} elements, expected {numel}")


def _ptrs(tensors):
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = t.data_ptr()
    return arr


def round_value(v: float, dtype: str) -> float:
    """v rounded to the nearest ``dtype`` value (ties to even), as a float."""
    return _load().or_round_value(float(v), _CODES[dtype])


def round_bits(v: float, dtype: str) -> int:
    """Bit pattern of v rounded to ``dtype``."""
    return int(_load().or_round_bits(float(v), _CODES[dtype]))


def decode_bits(bits: int, dtype: str) -> float:
    """Exact value of a ``dtype`` bit pattern."""
    return _load().or_decode_bits(int(bits), _CODES[dtype])


def sum(partials, dtype: str) -> torch.Tensor:  # noqa: A001 - the op is a sum
    """out = sum_r partials[r], binary64 in rank order, rounded once to dtype."""
    R = len(partials)
    n = partials[0].numel()
    for r, p in enumerate(partials):
        _check(p, dtype, n, f"partials[{r}]")
    out = torch.empty(n, dtype=_TORCH[dtype])
    _load().or_sum(_ptrs(partials), R, n, _CODES[dtype], out.data_ptr())
    return out.view(partials[0].shape)


def residual_rmsnorm(partials, bias, residual, weight, eps: float, dtype: str):
    """Fused sum + bias + residual + RMSNorm over [tokens, hidden] rows.

    Returns (out, residual_out, inv_rms) where inv_rms is a float64 numpy
    array holding 1/sqrt(mean(x^2)+eps) per row.
    """
    R = len(partials)
    tokens, hidden = residual.shape
    n = tokens * hidden
    for r, p in enumerate(partials):
        _check(p, dtype, n, f"partials[{r}]")
    _check(residual, dtype, n, "residual")
    _check(weight, dtype, hidden, "weight")
    if bias is not None:
        _check(bias, dtype, hidden, "bias")
    out = torch.empty((tokens, hidden), dtype=_TORCH[dtype])
    res_out = torch.empty((tokens, hidden), dtype=_TORCH[dtype])
    inv = np.zeros(max(tokens, 1), dtype=np.float64)
    xrow = np.zeros(max(hidden, 1), dtype=np.float64)
    _load().or_residual_rmsnorm(
        _ptrs(partials), R, None if bias is None else bias.data_ptr(),
        residual.data_ptr(), weight.data_ptr(), ctypes.c_float(eps),
        hidden, tokens, _CODES[dtype], out.data_ptr(), res_out.data_ptr(),
        inv.ctypes.data, xrow.ctypes.data)
    return out, res_out, inv[:tokens]


def rmsnorm(x, weight, eps: float, dtype: str):
    """RMSNorm of [tokens, hidden] rows on their own: (out, inv_rms per row as float64 numpy)."""
    tokens, hidden = x.shape
    _check(x, dtype, tokens * hidden, "x")
    _check(weight, dtype, hidden, "weight")
    out = torch.empty((tokens, hidden), dtype=_TORCH[dtype])
    inv = np.zeros(max(tokens, 1), dtype=np.float64)
    _load().or_rmsnorm(x.data_ptr(), weight.data_ptr(), ctypes.c_float(eps), hidden, tokens, _CODES[dtype],
                       out.data_ptr(), inv.ctypes.data)
    return out, inv[:tokens]
