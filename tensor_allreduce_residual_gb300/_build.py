"""Builds libar.so (the C-ABI library) in-tree with nvcc for sm_103a.

The translation units compile in parallel, then link into one shared
library next to this file.  Nothing is installed anywhere else.

A second library, libar_test.so, is the same code with the test hooks
compiled in (AR_TEST_HOOKS: the launch-shape override, the fault injection
of the bounded-wait tests and the programmatic-launch switch, each read from
the environment, and a communicator over local buffers for the peer
barrier's timeout test).  Only ar_api.cu and ar_peer.cu differ, so only
they are compiled twice.
The tests of forced launch shapes and of bounded waits, and the shape sweeps
that build the AUTO table, load it; everything else loads libar.so, which
reads no environment variable.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libar.so")
TEST_LIB = os.path.join(PKG, "libar_test.so")

SOURCES = ["ar_api.cu", "ar_kern_f32.cu", "ar_kern_f16.cu", "ar_kern_bf16.cu", "ar_noalloc.cu", "ar_host.cu",
           "ar_peer.cu"]
HEADERS = ["ar_internal.h", "ar_kernels.cuh", "ar_tma.cuh", "ar_lamport.cuh", "ar_launch.cuh", "ar_auto_table.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libar.so")
    return exe


def _stale() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(TEST_LIB)):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(TEST_LIB))
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "ar.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link libar.so and libar_test.so if any source is newer; returns libar.so's path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    units = [(src, os.path.join(BUILD, src.replace(".cu", ".o")), []) for src in SOURCES]
    units.append(("ar_api.cu", os.path.join(BUILD, "ar_api_test.o"), ["-DAR_TEST_HOOKS"]))
    units.append(("ar_peer.cu", os.path.join(BUILD, "ar_peer_test.o"), ["-DAR_TEST_HOOKS"]))
    for src, obj, defs in units:
        cmd = [cc, *ARCH, *FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_info or p.returncode != 0):
            print(out, file=sys.stderr)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    product = objs[:len(SOURCES)]
    swap = {os.path.join(BUILD, "ar_api.o"): objs[-2], os.path.join(BUILD, "ar_peer.o"): objs[-1]}
    test = [swap.get(o, o) for o in product]
    for lib, lib_objs in ((LIB, product), (TEST_LIB, test)):
        tmp = f"{lib}.{os.getpid()}.tmp"
        subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *lib_objs], check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
