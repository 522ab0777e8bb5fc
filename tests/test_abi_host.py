"""Host-only checks of the C-ABI library: it builds, loads and exports every
function include/ar.h declares; argument errors come back as status codes
before anything is launched; the ctypes mirror of ar_params matches the C
layout; workspace sizes and the AUTO choice are what the header states.

No test here reaches a kernel launch: every call below fails validation or is
an empty no-op, so these run the same with or without a GPU.
"""
import ctypes
import os
import re
import subprocess

import pytest

import tensor_allreduce_residual_gb300 as ar
from tensor_allreduce_residual_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ar.h")
FAKE = 0x10000  # never dereferenced: every call using it fails validation first


@pytest.fixture(scope="module")
def L():
    _build.build()
    return ar.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ar_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_expected_entry_points():
    names = _declared_functions()
    for want in ["ar_version", "ar_strerror", "ar_workspace_size", "ar_workspace_size_rows", "ar_sum",
                 "ar_residual_rmsnorm", "ar_allreduce", "ar_query_strategy", "ar_query_launch", "ar_device_status",
                 "ar_rmsnorm", "ar_host_staging_size", "ar_residual_rmsnorm_host", "ar_config_workspace_size",
                 "ar_allreduce_config", "ar_lamport_buffer_size", "ar_lamport_init", "ar_lamport_supported",
                 "ar_residual_rmsnorm_lamport", "ar_comm_buffer_size", "ar_comm_export", "ar_comm_create",
                 "ar_comm_destroy", "ar_allreduce_peer"]:
        assert want in names, names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), f"libar.so does not export {name}"
    nm = subprocess.run(["nm", "-D", "--defined-only", ar.LIB_PATH], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r"\bT (ar_\w+)", nm.stdout))
        assert set(_declared_functions()) <= exported


def test_test_library_exports_the_same_symbols(L):
    exported = {}
    for path in (ar.LIB_PATH, ar.TEST_LIB_PATH):
        nm = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True)
        if nm.returncode != 0:
            pytest.skip("nm unavailable")
        exported[path] = set(re.findall(r"\bT (ar_\w+)", nm.stdout))
    # the test build adds one test-only entry point, the communicator over local buffers
    assert exported[ar.TEST_LIB_PATH] == exported[ar.LIB_PATH] | {"ar_comm_create_local"}


_PLAN_PROBE = """
import ctypes, sys
sys.path.insert(0, {root!r})
import tensor_allreduce_residual_gb300 as ar
if sys.argv[1] == "test":
    ar.use_test_library()
print(ar.ar_query_launch(8, 8192, 8192, ar.AR_BF16, "ONESHOT")["kernel_name"],
      ar.ar_query_launch(8, 8192, 8192, ar.AR_BF16, "ONESHOT")["units_per_thread"])
"""


@pytest.mark.parametrize("which", ["product", "test"])
def test_only_the_test_library_reads_the_shape_override(L, which):
    """libar.so reads no environment variable: a launch-shape override left in the environment changes
    nothing there.  libar_test.so applies it (the shape sweeps and the forced-shape tests rely on that)."""
    env = dict(os.environ, AR_ONESHOT_SHAPE="1:0:1", AR_TEST_STALL_STAGE="1", AR_PDL="0")
    res = subprocess.run(["python", "-c", _PLAN_PROBE.format(root=ROOT), which], env=env, capture_output=True,
                         text=True, check=True)
    kernel, vpt = res.stdout.split()
    plain = subprocess.run(["python", "-c", _PLAN_PROBE.format(root=ROOT), "product"], capture_output=True,
                           text=True, check=True, env={k: v for k, v in os.environ.items() if not k.startswith("AR_")})
    if which == "product":
        assert res.stdout == plain.stdout          # the same plan as with a clean environment
    else:
        assert (kernel, vpt) == ("k_fused_oneshot", "1")   # the forced register shape, one vector a thread


def test_version_and_strerror(L):
    assert ar.ar_version() == 10000
    for code in (ar.AR_OK, ar.AR_ERR_INVALID_ARG, ar.AR_ERR_UNSUPPORTED, ar.AR_ERR_WORKSPACE, ar.AR_ERR_CUDA,
                 ar.AR_ERR_TIMEOUT):
        assert ar.ar_strerror(code) and ar.ar_strerror(code) != "unknown status code"
    assert ar.ar_strerror(12345) == "unknown status code"


def test_params_struct_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(f'''
#include <stdio.h>
#include <stddef.h>
#include "{HEADER}"
int main(void) {{
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(ar_params),
    offsetof(ar_params, partials), offsetof(ar_params, R), offsetof(ar_params, dtype),
    offsetof(ar_params, n), offsetof(ar_params, out), offsetof(ar_params, bias),
    offsetof(ar_params, residual), offsetof(ar_params, weight), offsetof(ar_params, eps),
    offsetof(ar_params, hidden), offsetof(ar_params, residual_out),
    offsetof(ar_params, workspace), offsetof(ar_params, workspace_bytes));
  return 0;
}}''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    P = ar.ArParams
    want = [ctypes.sizeof(P)] + [getattr(P, f).offset for f in
                                 ("partials", "R", "dtype", "n", "out", "bias", "residual", "weight", "eps",
                                  "hidden", "residual_out", "workspace", "workspace_bytes")]
    assert got == want


def _ptrs(n, value=FAKE):
    arr = (ctypes.c_void_p * max(n, 1))()
    for k in range(n):
        arr[k] = value + 256 * k
    return arr


def _sum(L, R, n=1024, dtype=ar.AR_FP16, strategy=ar.AR_ONESHOT, ptrs=None, out=FAKE + 65536):
    return L.ar_sum(ptrs if ptrs is not None else _ptrs(R), R, out, n, dtype, strategy, None)


def test_sum_argument_errors(L):
    assert _sum(L, 0) == ar.AR_ERR_INVALID_ARG
    assert _sum(L, ar.AR_MAX_RANKS + 1) == ar.AR_ERR_INVALID_ARG
    assert _sum(L, -3) == ar.AR_ERR_INVALID_ARG
    assert _sum(L, 2, dtype=7) == ar.AR_ERR_UNSUPPORTED
    assert _sum(L, 2, strategy=ar.AR_NCCL) == ar.AR_ERR_UNSUPPORTED
    assert _sum(L, 2, strategy=9) == ar.AR_ERR_UNSUPPORTED
    assert _sum(L, 2, out=None) == ar.AR_ERR_INVALID_ARG
    bad = _ptrs(2)
    bad[1] = None
    assert _sum(L, 2, ptrs=bad) == ar.AR_ERR_INVALID_ARG
    assert L.ar_sum(None, 2, FAKE, 16, ar.AR_FP16, ar.AR_ONESHOT, None) == ar.AR_ERR_INVALID_ARG


def test_empty_and_in_place_passthrough_launch_nothing(L):
    assert _sum(L, 2, n=0) == ar.AR_OK
    assert _sum(L, 2, n=0, ptrs=_ptrs(2, 0), out=None) == ar.AR_OK
    # R = 1 with out == partials[0]: the tpSize = 1 passthrough, in place
    assert _sum(L, 1, n=4096, ptrs=_ptrs(1), out=FAKE) == ar.AR_OK


def _fused(L, R=2, bias=FAKE + 1 << 20, residual=FAKE + 2 << 20, weight=FAKE + 3 << 20, eps=1e-6,
           hidden=64, tokens=4, out=FAKE + 4 << 20, residual_out=FAKE + 5 << 20, ws=None, ws_bytes=0,
           dtype=ar.AR_FP32, strategy=ar.AR_TWOSHOT, ptrs=None):
    return L.ar_residual_rmsnorm(ptrs if ptrs is not None else _ptrs(R), R, bias, residual, weight,
                                 ctypes.c_float(eps), hidden, tokens, out, residual_out, ws, ws_bytes,
                                 dtype, strategy, None)


def test_fused_argument_errors(L):
    assert _fused(L, R=0) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, R=17) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, hidden=0) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, tokens=-1) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, eps=-1e-6) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, eps=float("nan")) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, eps=float("inf")) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, residual=None) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, weight=None) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, out=None) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, residual_out=None) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, out=FAKE + 4 << 20, residual_out=FAKE + 4 << 20) == ar.AR_ERR_INVALID_ARG
    assert _fused(L, dtype=5) == ar.AR_ERR_UNSUPPORTED
    assert _fused(L, strategy=ar.AR_NCCL) == ar.AR_ERR_UNSUPPORTED
    bad = _ptrs(2)
    bad[0] = None
    assert _fused(L, ptrs=bad) == ar.AR_ERR_INVALID_ARG


def test_twoshot_workspace_errors(L):
    need = L.ar_workspace_size_rows(2, 64, 4, ar.AR_FP32)
    assert need > 0
    assert _fused(L, strategy=ar.AR_TWOSHOT, ws=None) == ar.AR_ERR_WORKSPACE
    assert _fused(L, strategy=ar.AR_TWOSHOT, ws=FAKE + 6 << 20, ws_bytes=0) == ar.AR_ERR_WORKSPACE
    assert _fused(L, strategy=ar.AR_TWOSHOT, ws=FAKE + (6 << 20) + 2, ws_bytes=need) == ar.AR_ERR_WORKSPACE
    # a row too long for every one-shot kernel at 64 tokens (the row-split cluster kernel
    # takes long rows only for a few tokens): ONESHOT is unsupported, AUTO needs a workspace
    long_row = 8 * 4096 * 2  # fp32 lanes * units per thread * threads, beyond the register budget
    assert _fused(L, hidden=long_row, tokens=64, strategy=ar.AR_ONESHOT) == ar.AR_ERR_UNSUPPORTED
    assert _fused(L, hidden=long_row, tokens=64, strategy=ar.AR_AUTO) == ar.AR_ERR_WORKSPACE


def test_fused_empty_is_noop(L):
    assert _fused(L, tokens=0, strategy=ar.AR_TWOSHOT) == ar.AR_OK
    assert _fused(L, tokens=0, residual=None, out=None, residual_out=None, ptrs=_ptrs(2, 0)) == ar.AR_OK


def test_allreduce_dispatch_errors(L):
    assert L.ar_allreduce(None, 0, ar.AR_ONESHOT, None) == ar.AR_ERR_INVALID_ARG
    p = ar.ArParams()
    p.R, p.dtype, p.n = 2, ar.AR_FP16, 0
    assert L.ar_allreduce(ctypes.byref(p), ar.AR_FUSION_NONE, ar.AR_ONESHOT, None) == ar.AR_OK
    assert L.ar_allreduce(ctypes.byref(p), 7, ar.AR_ONESHOT, None) == ar.AR_ERR_UNSUPPORTED
    p.n, p.hidden = 100, 64   # not a whole number of rows
    assert L.ar_allreduce(ctypes.byref(p), ar.AR_FUSION_RESIDUAL_RMS_NORM, ar.AR_ONESHOT, None) == ar.AR_ERR_INVALID_ARG
    p.hidden = 0
    assert L.ar_allreduce(ctypes.byref(p), ar.AR_FUSION_RESIDUAL_RMS_NORM, ar.AR_ONESHOT, None) == ar.AR_ERR_INVALID_ARG


def test_workspace_sizes(L):
    assert L.ar_workspace_size(0, 100, ar.AR_FP16) == 0
    assert L.ar_workspace_size(2, 0, ar.AR_FP16) == 0
    assert L.ar_workspace_size(2, 100, 9) == 0
    assert L.ar_workspace_size(2, 100, ar.AR_FP16) == 512        # 4 bytes per element, rounded to 256
    for R, H, T, dt in [(8, 8192, 8192, ar.AR_BF16), (2, 4096, 32, ar.AR_FP16), (2, 64, 4, ar.AR_FP32),
                        (3, 100, 7, ar.AR_FP16), (1, 1, 5, ar.AR_FP32)]:
        rows = L.ar_workspace_size_rows(R, H, T, dt)
        assert rows % 256 == 0 and rows >= T * 4
        assert rows <= L.ar_workspace_size(R, H * T, dt)             # the bound covers every shape
    assert L.ar_workspace_size_rows(8, 8192, 8192, ar.AR_BF16) == 8192 * 16 * 4
    assert L.ar_workspace_size_rows(2, 0, 4, ar.AR_FP32) == 0


def test_query_strategy(L):
    s, w = ar.ar_query_strategy(4, 1 << 20, 0, ar.AR_FP16, ar.AR_FUSION_NONE)
    assert s == ar.AR_ONESHOT and w == 0
    s, w = ar.ar_query_strategy(2, 4096, 4096, ar.AR_FP16)          # TP decode, one token
    assert s == ar.AR_ONESHOT and w >= 1
    s, w = ar.ar_query_strategy(8, 64 * 8192, 8192, ar.AR_BF16)     # R=8 small prefill
    assert s in (ar.AR_ONESHOT, ar.AR_TWOSHOT)
    s, w = ar.ar_query_strategy(2, 4 * 65536 * 2, 65536 * 2, ar.AR_FP32)   # row beyond the one-shot budget
    assert s == ar.AR_TWOSHOT and w == 0
    with pytest.raises(ar.ARError):
        ar.ar_query_strategy(2, 100, 64, ar.AR_FP32)                 # not a whole number of rows
    with pytest.raises(ar.ARError):
        ar.ar_query_strategy(0, 100, 10, ar.AR_FP32)


def test_launch_plan_struct_layout_matches_c(tmp_path):
    src = tmp_path / "plan.c"
    fields = [name for name, _ in ar.ArLaunchPlan._fields_]
    src.write_text(f'''
#include <stdio.h>
#include <stddef.h>
#include "{HEADER}"
int main(void) {{
  printf("%zu{" %zu" * len(fields)}\\n", sizeof(ar_launch_plan){"".join(f", offsetof(ar_launch_plan, {f})" for f in fields)});
  return 0;
}}''')
    exe = tmp_path / "plan"
    subprocess.run(["gcc", "-std=c11", str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    P = ar.ArLaunchPlan
    assert got == [ctypes.sizeof(P)] + [getattr(P, f).offset for f in fields]


def test_query_launch(L):
    # TP prefill, R=8 bf16 8192 x 8192: the measured table picks the bulk-copy-fed persistent kernel
    p = ar.ar_query_launch(8, 8192, 8192, ar.AR_BF16)
    assert p["strategy"] == ar.AR_ONESHOT and p["kernel"] == 4 and p["kernel_name"] == "k_fused_oneshot_tma"
    assert p["threads_per_block"] == p["threads_per_row"] + 32 and p["threads_per_row"] % 32 == 0
    assert p["stages"] >= 2 and p["blocks_per_sm"] >= 1
    assert p["smem_bytes"] * p["blocks_per_sm"] <= 228 * 1024
    # decode: a register-resident one-shot kernel
    p = ar.ar_query_launch(2, 4096, 1, ar.AR_FP16)
    assert p["strategy"] == ar.AR_ONESHOT and p["kernel"] == 1 and p["stages"] == 0
    assert p["threads_per_row"] * p["units_per_thread"] * 8 >= 4096
    # forced two-shot
    p = ar.ar_query_launch(8, 8192, 64, ar.AR_BF16, "TWOSHOT")
    assert p["strategy"] == ar.AR_TWOSHOT and p["kernel"] == 5
    # the AUTO answer agrees with ar_query_strategy
    for R, H, T, dt in [(8, 8192, 1, ar.AR_BF16), (8, 8192, 8192, ar.AR_BF16), (2, 4096, 32, ar.AR_FP16),
                        (2, 64, 4, ar.AR_FP32)]:
        s, w = ar.ar_query_strategy(R, H * T, H, dt)
        p = ar.ar_query_launch(R, H, T, dt)
        assert p["strategy"] == s and (s != ar.AR_ONESHOT or (p["threads_per_row"] + 31) // 32 == w)
    # errors, nothing launched
    plan = ar.ArLaunchPlan()
    assert L.ar_query_launch(0, 64, 4, ar.AR_FP32, ar.AR_AUTO, ctypes.byref(plan)) == ar.AR_ERR_INVALID_ARG
    assert L.ar_query_launch(2, 64, 4, ar.AR_FP32, ar.AR_AUTO, None) == ar.AR_ERR_INVALID_ARG
    assert L.ar_query_launch(2, 64, 4, 9, ar.AR_AUTO, ctypes.byref(plan)) == ar.AR_ERR_UNSUPPORTED
    assert L.ar_query_launch(2, 64, 4, ar.AR_FP32, ar.AR_NCCL, ctypes.byref(plan)) == ar.AR_ERR_UNSUPPORTED
    assert L.ar_query_launch(2, 65536 * 2, 4, ar.AR_FP32, ar.AR_ONESHOT, ctypes.byref(plan)) == ar.AR_ERR_UNSUPPORTED


def test_rmsnorm_argument_errors(L):
    def call(x=FAKE, w=FAKE + 4096, eps=1e-6, H=64, T=4, out=FAKE + 8192, dtype=ar.AR_FP32):
        return L.ar_rmsnorm(x, w, ctypes.c_float(eps), H, T, out, dtype, None)
    assert call(H=0) == ar.AR_ERR_INVALID_ARG
    assert call(T=-1) == ar.AR_ERR_INVALID_ARG
    assert call(eps=-1.0) == ar.AR_ERR_INVALID_ARG
    assert call(eps=float("nan")) == ar.AR_ERR_INVALID_ARG
    assert call(x=None) == ar.AR_ERR_INVALID_ARG
    assert call(w=None) == ar.AR_ERR_INVALID_ARG
    assert call(out=None) == ar.AR_ERR_INVALID_ARG
    assert call(dtype=4) == ar.AR_ERR_UNSUPPORTED
    assert call(H=16385, dtype=ar.AR_BF16) == ar.AR_ERR_UNSUPPORTED      # beyond the register-resident row
    assert call(H=16385 * 4, dtype=ar.AR_FP32) == ar.AR_ERR_UNSUPPORTED
    assert call(T=0, x=None, out=None) == ar.AR_OK                       # empty: nothing launched


def test_host_staging_size_and_errors(L):
    # two buffers of (R + 3) chunk tensors + a workspace each, then weight and bias
    R, H, C = 8, 8192, 512
    chunk = C * H * 2
    ws = L.ar_workspace_size_rows(R, H, C, ar.AR_BF16)
    assert L.ar_host_staging_size(R, H, C, ar.AR_BF16) == 2 * ((R + 3) * chunk + ws) + 2 * H * 2
    assert L.ar_host_staging_size(0, H, C, ar.AR_BF16) == 0
    assert L.ar_host_staging_size(R, H, 0, ar.AR_BF16) == 0
    assert L.ar_host_staging_size(R, H, C, 7) == 0

    def call(R=2, T=4, H=64, chunk=2, staging=FAKE, nbytes=1 << 30, residual=FAKE + 1, ptrs=None, dtype=ar.AR_FP32):
        return L.ar_residual_rmsnorm_host(ptrs if ptrs is not None else _ptrs(R), R, None, residual, FAKE + 2,
                                          ctypes.c_float(1e-6), H, T, FAKE + 3, FAKE + 4, staging, nbytes, chunk,
                                          dtype, ar.AR_AUTO, None)
    assert call(R=0) == ar.AR_ERR_INVALID_ARG
    assert call(chunk=0) == ar.AR_ERR_INVALID_ARG
    assert call(staging=None) == ar.AR_ERR_INVALID_ARG
    assert call(residual=None) == ar.AR_ERR_INVALID_ARG
    assert call(dtype=9) == ar.AR_ERR_UNSUPPORTED
    assert call(nbytes=100) == ar.AR_ERR_WORKSPACE
    assert call(staging=FAKE + 16) == ar.AR_ERR_WORKSPACE        # not 256-byte aligned
    assert call(T=0) == ar.AR_OK


def test_allreduce_config_errors_and_sizes(L):
    assert L.ar_config_workspace_size(4, 1000, 0, ar.AR_FP16) == 4 * 2048          # 2000 B -> 2048 per slot
    assert L.ar_config_workspace_size(2, 64 * 4, 64, ar.AR_FP32) == 2 * 1024 + L.ar_workspace_size_rows(2, 64, 4, ar.AR_FP32)
    assert L.ar_config_workspace_size(0, 100, 0, ar.AR_FP16) == 0
    assert L.ar_config_workspace_size(2, 100, 64, ar.AR_FP16) == 0                 # not a whole number of rows
    assert L.ar_allreduce_config(None, 0, ar.AR_ONESHOT, 1, None) == ar.AR_ERR_INVALID_ARG
    p = ar.ArParams()
    p.R, p.dtype, p.n = 2, ar.AR_FP16, 1024
    p.partials[0], p.partials[1], p.out = FAKE, FAKE + 4096, FAKE + 8192
    assert L.ar_allreduce_config(ctypes.byref(p), 0, ar.AR_ONESHOT, 4, None) == ar.AR_ERR_UNSUPPORTED
    assert L.ar_allreduce_config(ctypes.byref(p), 0, ar.AR_ONESHOT, 1, None) == ar.AR_ERR_WORKSPACE   # no workspace
    p.workspace, p.workspace_bytes = FAKE + 16, 1 << 20
    assert L.ar_allreduce_config(ctypes.byref(p), 0, ar.AR_ONESHOT, 1, None) == ar.AR_ERR_WORKSPACE   # misaligned
    p.workspace, p.workspace_bytes = FAKE, 100
    assert L.ar_allreduce_config(ctypes.byref(p), 0, ar.AR_ONESHOT, 1, None) == ar.AR_ERR_WORKSPACE   # too small
    p.partials[1] = None
    assert L.ar_allreduce_config(ctypes.byref(p), 0, ar.AR_ONESHOT, 1, None) == ar.AR_ERR_INVALID_ARG
    p.n = 0
    assert L.ar_allreduce_config(ctypes.byref(p), 0, ar.AR_ONESHOT, 1, None) == ar.AR_OK


def _lamport(L, R=2, bias=FAKE + 1 << 20, residual=FAKE + 2 << 20, weight=FAKE + 3 << 20, eps=1e-6,
             hidden=64, tokens=4, out=FAKE + 4 << 20, residual_out=FAKE + 5 << 20, buf=FAKE + 7 << 20,
             buf_bytes=1 << 20, dtype=ar.AR_FP32, ptrs=None):
    return L.ar_residual_rmsnorm_lamport(ptrs if ptrs is not None else _ptrs(R), R, bias, residual, weight,
                                         ctypes.c_float(eps), hidden, tokens, out, residual_out, buf, buf_bytes,
                                         dtype, None)


def test_lamport_argument_errors(L):
    assert _lamport(L, R=0) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, R=17) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, hidden=0) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, tokens=-1) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, eps=-1.0) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, eps=float("nan")) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, residual=None) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, weight=None) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, out=None) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, residual_out=FAKE + 4 << 20) == ar.AR_ERR_INVALID_ARG      # out == residual_out
    bad = _ptrs(2)
    bad[1] = None
    assert _lamport(L, ptrs=bad) == ar.AR_ERR_INVALID_ARG
    assert _lamport(L, dtype=5) == ar.AR_ERR_UNSUPPORTED
    # only the 16-byte packed path: misaligned pointers, a hidden that is not a multiple of the
    # lane count, and rows longer than the kernel holds are refused
    assert _lamport(L, residual=(FAKE + 2 << 20) + 4) == ar.AR_ERR_UNSUPPORTED
    assert _lamport(L, ptrs=_ptrs(2, FAKE + 8)) == ar.AR_ERR_UNSUPPORTED
    assert _lamport(L, hidden=66) == ar.AR_ERR_UNSUPPORTED
    assert _lamport(L, hidden=8192 + 4, tokens=4096, buf_bytes=1 << 30) == ar.AR_ERR_UNSUPPORTED
    # the buffer: missing, misaligned or short
    assert _lamport(L, buf=None) == ar.AR_ERR_WORKSPACE
    assert _lamport(L, buf=(FAKE + 7 << 20) + 8) == ar.AR_ERR_WORKSPACE
    need = L.ar_lamport_buffer_size(2, 64, 4, ar.AR_FP32)
    assert need == 2 * 4 * 64 * 4 + 4 * 64 + 4096   # the slots, 64 bytes of exchange area a row, progress words
    assert _lamport(L, buf_bytes=need - 1) == ar.AR_ERR_WORKSPACE
    assert _lamport(L, buf_bytes=2 * 4 * 64 * 4 + 4 * 64) == ar.AR_ERR_WORKSPACE
    # nothing to do
    assert _lamport(L, tokens=0, buf=None, residual=None, out=None) == ar.AR_OK


def test_lamport_buffer_size_support_and_init(L):
    P = 512 * 8                                    # the progress words, one a block
    assert L.ar_lamport_buffer_size(8, 8192, 1, ar.AR_BF16) == (8 * 8192 * 2 + 64 + P + 255) // 256 * 256
    assert L.ar_lamport_buffer_size(3, 16, 1, ar.AR_FP16) == (96 + 64 + P + 255) // 256 * 256
    assert L.ar_lamport_buffer_size(3, 10, 1, ar.AR_FP16) == 0                 # a shape the call cannot take
    # the slots are a ring of at most 1024 row groups: 1024 rows of 8192 (one row a group) ...
    assert L.ar_lamport_buffer_size(8, 8192, 8192, ar.AR_BF16) == 8 * 1024 * 8192 * 2 + 8192 * 64 + P
    # ... or 8192 rows of 64 fp32 (16 vectors a row: 8 rows a group), then 64 bytes a token
    assert L.ar_lamport_buffer_size(2, 64, 20000, ar.AR_FP32) == (2 * 8192 * 64 * 4 + 20000 * 64 + P + 255) // 256 * 256
    assert L.ar_lamport_buffer_size(2, 64, 5000, ar.AR_FP32) == 2 * 5000 * 64 * 4 + 5000 * 64 + P
    for bad in [(0, 64, 1, ar.AR_FP32), (17, 64, 1, ar.AR_FP32), (2, 0, 1, ar.AR_FP32), (2, 64, -1, ar.AR_FP32),
                (2, 64, 1, 9)]:
        assert L.ar_lamport_buffer_size(*bad) == 0
    w = ctypes.c_int(-1)
    # up to 8 rows of many vectors: a row split over 4 blocks; else one block a row, 16 warps up to 512 rows;
    # from 1024 rows separate push and reduce warps, the reduce side 16 warps a row of two vectors a thread
    assert L.ar_lamport_supported(8, 8192, 1, ar.AR_BF16, ctypes.byref(w)) == ar.AR_OK and w.value == 32
    assert L.ar_lamport_supported(2, 4096, 32, ar.AR_FP16, ctypes.byref(w)) == ar.AR_OK and w.value == 16
    assert L.ar_lamport_supported(8, 8192, 256, ar.AR_BF16, ctypes.byref(w)) == ar.AR_OK and w.value == 16
    assert L.ar_lamport_supported(8, 8192, 4096, ar.AR_BF16, ctypes.byref(w)) == ar.AR_OK and w.value == 16
    assert L.ar_lamport_supported(2, 16384, 1, ar.AR_BF16, ctypes.byref(w)) == ar.AR_OK and w.value == 8
    assert L.ar_lamport_supported(2, 16384, 100, ar.AR_BF16, ctypes.byref(w)) == ar.AR_OK and w.value == 8
    assert L.ar_lamport_supported(2, 64, 4, ar.AR_FP32, ctypes.byref(w)) == ar.AR_OK and w.value == 1
    assert L.ar_lamport_supported(2, 8192, 1, ar.AR_FP32, None) == ar.AR_OK
    assert L.ar_lamport_supported(2, 32768, 1000, ar.AR_BF16, None) == ar.AR_ERR_UNSUPPORTED   # row too long
    assert L.ar_lamport_supported(2, 32768, 1, ar.AR_BF16, ctypes.byref(w)) == ar.AR_OK and w.value == 64
    assert L.ar_lamport_supported(2, 8 * 32768, 1, ar.AR_BF16, None) == ar.AR_ERR_UNSUPPORTED
    assert L.ar_lamport_supported(2, 100, 1, ar.AR_BF16, None) == ar.AR_ERR_UNSUPPORTED     # not 8-lane
    assert L.ar_lamport_supported(0, 64, 1, ar.AR_FP32, None) == ar.AR_ERR_INVALID_ARG
    assert L.ar_lamport_supported(2, 64, 1, 9, None) == ar.AR_ERR_UNSUPPORTED
    assert L.ar_lamport_init(None, 16, ar.AR_BF16, None) == ar.AR_ERR_INVALID_ARG
    assert L.ar_lamport_init(FAKE + 8, 16, ar.AR_BF16, None) == ar.AR_ERR_INVALID_ARG
    assert L.ar_lamport_init(FAKE, 15, ar.AR_BF16, None) == ar.AR_ERR_INVALID_ARG
    assert L.ar_lamport_init(FAKE, 16, 9, None) == ar.AR_ERR_UNSUPPORTED
    assert L.ar_lamport_init(FAKE, 0, ar.AR_BF16, None) == ar.AR_OK


def test_launch_plans_are_launchable_for_random_shapes(L):
    """Every plan the host logic accepts, over random shapes, fits the device's launch limits and
    covers its row; shapes it cannot serve are refused with a status, never a bad plan."""
    import random
    rng = random.Random(1234)
    lanes_of = {ar.AR_FP32: 4, ar.AR_FP16: 8, ar.AR_BF16: 8}
    seen = set()
    for _ in range(3000):
        R = rng.randint(1, 16)
        dt = rng.choice([ar.AR_FP32, ar.AR_FP16, ar.AR_BF16])
        hidden = rng.choice([rng.randint(1, 300), rng.randint(1, 70000), 8 * rng.randint(1, 8192)])
        tokens = rng.choice([rng.randint(1, 40), rng.randint(1, 20000)])
        strategy = rng.choice([ar.AR_ONESHOT, ar.AR_TWOSHOT, ar.AR_AUTO])
        plan = ar.ArLaunchPlan()
        st = L.ar_query_launch(R, hidden, tokens, dt, strategy, ctypes.byref(plan))
        if st != ar.AR_OK:
            assert st == ar.AR_ERR_UNSUPPORTED and strategy == ar.AR_ONESHOT, (R, hidden, tokens, dt, strategy, st)
            continue
        p = {k: getattr(plan, k) for k, _ in ar.ArLaunchPlan._fields_}
        seen.add(p["kernel"])
        assert p["strategy"] in (ar.AR_ONESHOT, ar.AR_TWOSHOT)
        assert strategy == ar.AR_AUTO or p["strategy"] == strategy
        assert 32 <= p["threads_per_block"] <= 1024, p
        assert p["smem_bytes"] <= 227 * 1024, p
        units = hidden // lanes_of[dt] if hidden % lanes_of[dt] == 0 else hidden
        if p["kernel"] == 4:       # bulk-copy ring: consumers + producer warp, whole chunks, two stages at least
            nc, cpr, stages = p["threads_per_row"], p["units_per_thread"], p["stages"]
            assert p["threads_per_block"] == nc + 32 and nc % 32 == 0
            assert nc * cpr >= units and stages >= 2
            assert -(-units // nc) <= cpr              # the row's chunks fit the compiled chunk count
            # ring layout: per stage the R partials' and the residual's chunk tiles (16-byte vectors),
            # then a full and an empty mbarrier per stage, then the [2][32] fp32 row-reduction scratch
            tiles = stages * (R + 1) * nc * 16
            assert tiles % 16 == 0 and p["smem_bytes"] == tiles + stages * 16 + 2 * 32 * 4
            last = units - (-(-units // nc) - 1) * nc  # vectors in a row's last (ragged) chunk
            assert 0 < last <= nc
            assert p["smem_bytes"] * p["blocks_per_sm"] <= 228 * 1024 - 1024 * p["blocks_per_sm"]
        elif p["kernel"] == 6:     # row split over a cluster
            assert p["cluster"] in (2, 4, 8) and p["threads_per_row"] == p["threads_per_block"] * p["cluster"]
            assert p["threads_per_row"] * p["units_per_thread"] >= units
        elif p["kernel"] in (1, 2, 3):
            assert p["threads_per_row"] * p["units_per_thread"] >= units
            assert p["threads_per_row"] & (p["threads_per_row"] - 1) == 0
    assert {1, 4, 5, 6} <= seen, seen      # the draw reached the main kernels


def test_binding_rejects_mismatched_tensors_before_any_call():
    """The Python binding checks every tensor's size, dtype, device and layout against the call's shape
    before it reaches the library (which trusts its pointers).  Host tensors exercise the checks without
    a GPU: the host-buffer call takes them, the device calls refuse them."""
    import torch
    T, H = 4, 64
    bf = torch.bfloat16
    parts = [torch.zeros(T, H, dtype=bf) for _ in range(2)]
    res, w, b = torch.zeros(T, H, dtype=bf), torch.ones(H, dtype=bf), torch.zeros(H, dtype=bf)
    out, rout = torch.zeros(T, H, dtype=bf), torch.zeros(T, H, dtype=bf)
    staging = torch.zeros(16, dtype=torch.uint8)

    def host(**kw):
        args = dict(partials=parts, residual=res, weight=w, eps=1e-6, staging=staging, out=out, residual_out=rout,
                    bias=b)
        args.update(kw)
        return ar.ar_residual_rmsnorm_host(**args)

    bad_cases = [
        dict(weight=torch.ones(H - 8, dtype=bf)),                      # short weight
        dict(weight=torch.ones(H, dtype=torch.float16)),               # wrong dtype
        dict(bias=torch.zeros(2 * H, dtype=bf)),                       # long bias
        dict(out=torch.zeros(T - 1, H, dtype=bf)),                     # short output
        dict(residual_out=torch.zeros(T, H, dtype=torch.float32)),     # wrong dtype
        dict(partials=[parts[0], torch.zeros(T, H + 8, dtype=bf)]),    # partial of another shape
        dict(partials=[parts[0], torch.zeros(H, T, dtype=bf).t()]),    # not contiguous
        dict(partials=[]),                                             # no partials
        dict(residual=torch.zeros(T * H, dtype=bf)),                   # not [tokens, hidden]
        dict(out=None),                                                # host outputs are required
    ]
    for kw in bad_cases:
        with pytest.raises(ValueError):
            host(**kw)
    # device calls refuse host tensors outright
    for call in (lambda: ar.ar_residual_rmsnorm(parts, res, w, 1e-6, bias=b, out=out, residual_out=rout),
                 lambda: ar.ar_residual_rmsnorm_lamport(parts, res, w, 1e-6, bias=b, out=out, residual_out=rout),
                 lambda: ar.ar_residual_rmsnorm_noalloc(parts, res, w, 1e-6, bias=b, out=out, residual_out=rout),
                 lambda: ar.ar_rmsnorm(res, w, 1e-6, out=out),
                 lambda: ar.ar_sum(parts, out=out)):
        with pytest.raises(ValueError):
            call()
    with pytest.raises(ValueError):
        ar.ar_rmsnorm(res, torch.ones(H + 8, dtype=bf), 1e-6)


def test_peer_comm_sizes_and_argument_errors(L):
    """The multi-GPU communicator's calls reject bad arguments before any CUDA call."""
    assert L.ar_comm_buffer_size(1, 1) == 16384 + 2 * 256                  # flag words, two data areas
    assert L.ar_comm_buffer_size(8, 1 << 20) == 16384 + 2 * (1 << 20)
    for bad in [(0, 1024), (17, 1024), (2, 0)]:
        assert L.ar_comm_buffer_size(*bad) == 0
    comm = ctypes.c_void_p(0)
    size = L.ar_comm_buffer_size(2, 4096)
    handles = ctypes.create_string_buffer(2 * ar.AR_IPC_HANDLE_BYTES)
    for rank, world, buf, nbytes, maxb, h in [
            (2, 2, FAKE, size, 4096, handles),          # rank out of range
            (-1, 2, FAKE, size, 4096, handles),
            (0, 17, FAKE, size, 4096, handles),         # world beyond AR_MAX_RANKS
            (0, 2, None, size, 4096, handles),          # no buffer
            (0, 2, FAKE + 8, size, 4096, handles),      # misaligned buffer
            (0, 2, FAKE, size, 0, handles),             # nothing to reduce
            (0, 2, FAKE, size, 4096, None)]:            # two ranks and no handles
        assert L.ar_comm_create(rank, world, buf, nbytes, maxb, h, ctypes.byref(comm)) == ar.AR_ERR_INVALID_ARG
    assert L.ar_comm_create(0, 2, FAKE, size - 1, 4096, handles, ctypes.byref(comm)) == ar.AR_ERR_WORKSPACE
    assert L.ar_comm_create(0, 1, FAKE, size, 4096, None, None) == ar.AR_ERR_INVALID_ARG
    assert L.ar_comm_destroy(None) == ar.AR_ERR_INVALID_ARG
    assert L.ar_comm_export(None, handles) == ar.AR_ERR_INVALID_ARG
    assert L.ar_allreduce_peer(None, FAKE, FAKE, 16, ar.AR_FP16, ar.AR_AUTO, None) == ar.AR_ERR_INVALID_ARG


def test_gather_handles_orders_by_rank():
    """The handle exchange concatenates every rank's handle in rank order and refuses short ones."""
    hs = [bytes([r]) * ar.AR_IPC_HANDLE_BYTES for r in range(3)]

    def fake_all_gather(out, obj):
        out[:] = hs
    assert ar.gather_handles(hs[1], fake_all_gather, 3) == b"".join(hs)
    with pytest.raises(ValueError):
        ar.gather_handles(b"short", fake_all_gather, 3)

    def broken(out, obj):
        out[:] = [hs[0], None, hs[2]]
    with pytest.raises(ValueError):
        ar.gather_handles(hs[0], broken, 3)
