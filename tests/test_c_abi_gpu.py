"""The library from plain C: tests/c_abi_example.c is compiled with gcc
against include/ar.h, linked with libar.so and the CUDA runtime, and run; its
fused output, residual_out, plain sum and Lamport-style outputs are checked
against the oracle.
Nothing on that path goes through Python or torch."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads
from tensor_allreduce_residual_gb300 import _build
from tests import tolerance as tol

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
R, T, H, EPS = 4, 3, 1000, 1e-5


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_c_program_through_the_abi(tmp_path):
    lib = _build.build()
    cuda = _cuda_home()
    exe = tmp_path / "c_abi_example"
    subprocess.run(["gcc", "-std=c11", "-O2", os.path.join(HERE, "c_abi_example.c"), f"-I{_build.INCLUDE}",
                    f"-I{cuda}/include", f"-L{os.path.dirname(lib)}", "-lar", f"-L{cuda}/lib64", "-lcudart",
                    f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{cuda}/lib64", "-o", str(exe)], check=True)

    f = workloads.fused_inputs(R, T, H, "fp32", partial_dist=("N", 0.0, 0.25), residual_dist=("N", 0.0, 1.0),
                               bias_dist=("N", 0.0, 0.1), weight_dist=("N", 1.0, 0.1), eps=EPS, seed=5)
    blob = torch.cat([p.reshape(-1) for p in f.partials] + [f.residual.reshape(-1), f.bias, f.weight])
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    blob.numpy().astype(np.float32).tofile(inp)
    res = subprocess.run([str(exe), str(inp), str(outp)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and "c_abi_example: ok" in res.stdout, res.stdout + res.stderr

    got = torch.from_numpy(np.fromfile(outp, dtype=np.float32)).reshape(5, T, H)
    ref_out, ref_res, inv = oracle.residual_rmsnorm(f.partials, f.bias, f.residual, f.weight, EPS, "fp32")
    terms = [p.reshape(T, H) for p in f.partials] + [f.bias.expand(T, H).contiguous(), f.residual]
    tol.check_sum(got[1], ref_res, terms, "fp32", "residual_out", R=f.R, hidden=H)
    tol.check_fused_out(got[0], ref_out, terms, f.weight, inv, "fp32", H, "out", R=f.R)
    tol.check_sum(got[2], oracle.sum(f.partials, "fp32"), f.partials, "fp32", "sum", R=f.R)
    tol.check_sum(got[4], ref_res, terms, "fp32", "Lamport residual_out", R=f.R, hidden=H)
    tol.check_fused_out(got[3], ref_out, terms, f.weight, inv, "fp32", H, "Lamport out", R=f.R)
