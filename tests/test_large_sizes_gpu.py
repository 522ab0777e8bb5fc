"""Sizes past 2^31 elements: no 32-bit index may wrap.

ar_sum on n = 2^31 + 13 fp16 elements (R = 2), and the fused call on
262,145 rows of hidden 8192 (R = 1, 2^31 + 8192 elements per tensor, bf16),
with the inputs built on the device from integer patterns that are exact in
the element type.  The oracle checks sampled positions on both sides of the
2^31 boundary and at the very end.  About 13 GB and 17 GB of device memory.
"""
import pytest
import torch

import oracle
import tensor_allreduce_residual_gb300 as ar
from tests import tolerance as tol

pytestmark = pytest.mark.gpu

N31 = 1 << 31


def _pattern(n, mod, off, scale, dtype):
    """((i mod `mod`) - off) / scale for i < n, exact in fp16 / bf16 for the values used here."""
    i = torch.arange(n, device="cuda", dtype=torch.int64)
    return ((i % mod) - off).to(torch.float32).div_(scale).to(dtype)


def _free_bytes():
    free, _ = torch.cuda.mem_get_info()
    return free


def test_sum_past_2_31_elements():
    n = N31 + 13
    if _free_bytes() < 3 * 2 * n + (4 << 30):
        pytest.skip("not enough free device memory")
    p0 = _pattern(n, 1021, 510, 512.0, torch.float16)
    p1 = _pattern(n, 977, 488, 256.0, torch.float16)
    out = ar.ar_sum([p0, p1])
    torch.cuda.synchronize()
    idx = torch.tensor([0, 1, N31 - 9, N31 - 1, N31, N31 + 1, N31 + 7, n - 8, n - 1], device="cuda")
    got = out[idx].cpu()
    want = oracle.sum([p0[idx].cpu().contiguous(), p1[idx].cpu().contiguous()], "fp16")
    tol.check_sum(got, want, [p0[idx].cpu(), p1[idx].cpu()], "fp16", "sum past 2^31", R=2)
    del p0, p1, out
    torch.cuda.empty_cache()


def test_fused_past_2_31_elements():
    H = 8192
    T = N31 // H + 1                      # 262,145 rows: the last row starts at element 2^31
    n = T * H
    if _free_bytes() < 4 * 2 * n + (4 << 30):
        pytest.skip("not enough free device memory")
    p0 = _pattern(n, 509, 254, 128.0, torch.bfloat16).view(T, H)
    res = _pattern(n, 251, 125, 32.0, torch.bfloat16).view(T, H)
    w = (1.0 + _pattern(H, 17, 8, 64.0, torch.float32)).to(torch.bfloat16)
    out, rout = ar.ar_residual_rmsnorm([p0], res, w, 1e-6)
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, T // 2, T - 3, T - 2, T - 1], device="cuda")
    sub_p, sub_r = p0[rows].cpu().contiguous(), res[rows].cpu().contiguous()
    ro, rr, inv = oracle.residual_rmsnorm([sub_p], None, sub_r, w.cpu(), 1e-6, "bf16")
    terms = [sub_p, sub_r]
    tol.check_sum(rout[rows].cpu(), rr, terms, "bf16", "residual_out past 2^31", R=1, hidden=H)
    tol.check_fused_out(out[rows].cpu(), ro, terms, w.cpu(), inv, "bf16", H, "out past 2^31", R=1)
    del p0, res, out, rout
    torch.cuda.empty_cache()
