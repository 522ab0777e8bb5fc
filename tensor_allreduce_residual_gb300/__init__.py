"""GB300-native R-way all-reduce (sum) and fused sum + residual + RMSNorm.

Thin Python binding of the C-ABI library ``libar.so`` (declared in
``include/ar.h``).  Every function here only marshals torch tensors into
pointers and sizes and calls the library function of the same name; all
arithmetic runs in the library's CUDA kernels.  There is no fallback: if the
library has not been built, or no CUDA device is present, calls raise.

The R partials are R CUDA tensors on the same device: the tensor-parallel
ranks' partial outputs of a row-parallel linear layer, kept in one GPU's HBM.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libar.so")
# The same library with its test hooks compiled in (launch-shape override,
# bounded-wait fault injection, programmatic-launch switch, read from the
# environment); only tests and shape sweeps load it, by use_test_library().
TEST_LIB_PATH = os.path.join(_PKG, "libar_test.so")

# ar_dtype
AR_FP32, AR_FP16, AR_BF16 = 0, 1, 2
# ar_strategy (AllReduceStrategyType values)
AR_NCCL, AR_ONESHOT, AR_TWOSHOT, AR_AUTO = 0, 1, 2, 3
# ar_fusion_op (AllReduceFusionOp values)
AR_FUSION_NONE, AR_FUSION_RESIDUAL_RMS_NORM = 0, 1
# status codes
AR_OK, AR_ERR_INVALID_ARG, AR_ERR_UNSUPPORTED, AR_ERR_WORKSPACE, AR_ERR_CUDA, AR_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
AR_MAX_RANKS = 16
# AllReduceStrategyConfig bit flags
AR_CONFIG_USE_MEMCPY, AR_CONFIG_RESIDUAL_RMS_NORM = 1, 2
AR_NOALLOC_SCRATCH_BYTES = 1 << 20
AR_IPC_HANDLE_BYTES = 64

STRATEGIES = {"NCCL": AR_NCCL, "ONESHOT": AR_ONESHOT, "TWOSHOT": AR_TWOSHOT, "AUTO": AR_AUTO}
STRATEGY_NAMES = {v: k for k, v in STRATEGIES.items()}
_TORCH_TO_AR = {torch.float32: AR_FP32, torch.float16: AR_FP16, torch.bfloat16: AR_BF16}


class ARError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: {status} ({ar_strerror(status)})")


class ArParams(ctypes.Structure):
    """Mirror of the C struct ar_params."""
    _fields_ = [
        ("partials", ctypes.c_void_p * AR_MAX_RANKS),
        ("R", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("n", ctypes.c_size_t),
        ("out", ctypes.c_void_p),
        ("bias", ctypes.c_void_p),
        ("residual", ctypes.c_void_p),
        ("weight", ctypes.c_void_p),
        ("eps", ctypes.c_float),
        ("hidden", ctypes.c_int),
        ("residual_out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class ArLaunchPlan(ctypes.Structure):
    """Mirror of the C struct ar_launch_plan."""
    _fields_ = [(name, ctypes.c_int) for name in (
        "strategy", "kernel", "threads_per_row", "units_per_thread", "rows_per_block", "threads_per_block",
        "blocks_per_sm", "stages", "smem_bytes", "early_residual", "cluster")]


# ar_kernel codes and the kernel names they stand for
KERNEL_NAMES = {1: "k_fused_oneshot", 2: "k_fused_oneshot", 3: "k_fused_oneshot_persist",
                4: "k_fused_oneshot_tma", 5: "k_twoshot_phase1+k_twoshot_phase2", 6: "k_fused_oneshot_cluster"}

_lib: Optional[ctypes.CDLL] = None
_lib_path = LIB_PATH


def use_test_library() -> None:
    """Load libar_test.so instead of libar.so in this process (tests and shape sweeps only: its launch
    shapes and fault injection follow AR_ONESHOT_SHAPE, AR_TEST_STALL_STAGE, AR_TEST_LAMPORT_SKIP_RANK
    and AR_PDL).  Must come before the first call into the library."""
    global _lib_path
    if _lib is not None and _lib_path != TEST_LIB_PATH:
        raise RuntimeError("libar.so is already loaded in this process")
    _lib_path = TEST_LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libar.so (or libar_test.so) with its C signatures declared.  Raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_lib_path):
        raise RuntimeError(f"{_lib_path} is missing: build it first (tensor_allreduce_residual_gb300._build.build())")
    L = ctypes.CDLL(_lib_path)
    vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pvp = ctypes.POINTER(ctypes.c_void_p)
    L.ar_version.argtypes, L.ar_version.restype = [], i
    L.ar_strerror.argtypes, L.ar_strerror.restype = [i], ctypes.c_char_p
    L.ar_workspace_size.argtypes, L.ar_workspace_size.restype = [i, sz, i], sz
    L.ar_workspace_size_rows.argtypes, L.ar_workspace_size_rows.restype = [i, i, i, i], sz
    L.ar_sum.argtypes, L.ar_sum.restype = [pvp, i, vp, sz, i, i, vp], i
    L.ar_residual_rmsnorm.argtypes = [pvp, i, vp, vp, vp, ctypes.c_float, i, i, vp, vp, vp, sz, i, i, vp]
    L.ar_residual_rmsnorm.restype = i
    L.ar_allreduce.argtypes, L.ar_allreduce.restype = [ctypes.POINTER(ArParams), i, i, vp], i
    L.ar_query_strategy.argtypes = [i, sz, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
    L.ar_query_strategy.restype = i
    L.ar_residual_rmsnorm_noalloc.argtypes = [pvp, i, vp, vp, vp, ctypes.c_float, i, i, vp, vp, i, vp]
    L.ar_residual_rmsnorm_noalloc.restype = i
    L.ar_device_status.argtypes, L.ar_device_status.restype = [], i
    L.ar_rmsnorm.argtypes, L.ar_rmsnorm.restype = [vp, vp, ctypes.c_float, i, i, vp, i, vp], i
    L.ar_host_staging_size.argtypes, L.ar_host_staging_size.restype = [i, i, i, i], sz
    L.ar_config_workspace_size.argtypes, L.ar_config_workspace_size.restype = [i, sz, i, i], sz
    L.ar_allreduce_config.argtypes = [ctypes.POINTER(ArParams), i, i, i, vp]
    L.ar_allreduce_config.restype = i
    L.ar_residual_rmsnorm_host.argtypes = [pvp, i, vp, vp, vp, ctypes.c_float, i, i, vp, vp, vp, sz, i, i, i, vp]
    L.ar_residual_rmsnorm_host.restype = i
    L.ar_query_launch.argtypes = [i, i, i, i, i, ctypes.POINTER(ArLaunchPlan)]
    L.ar_query_launch.restype = i
    L.ar_lamport_buffer_size.argtypes, L.ar_lamport_buffer_size.restype = [i, i, i, i], sz
    L.ar_lamport_init.argtypes, L.ar_lamport_init.restype = [vp, sz, i, vp], i
    L.ar_lamport_supported.argtypes = [i, i, i, i, ctypes.POINTER(i)]
    L.ar_lamport_supported.restype = i
    L.ar_residual_rmsnorm_lamport.argtypes = [pvp, i, vp, vp, vp, ctypes.c_float, i, i, vp, vp, vp, sz, i, vp]
    L.ar_residual_rmsnorm_lamport.restype = i
    L.ar_comm_buffer_size.argtypes, L.ar_comm_buffer_size.restype = [i, sz], sz
    L.ar_comm_export.argtypes, L.ar_comm_export.restype = [vp, vp], i
    L.ar_comm_create.argtypes = [i, i, vp, sz, sz, vp, ctypes.POINTER(vp)]
    L.ar_comm_create.restype = i
    L.ar_comm_destroy.argtypes, L.ar_comm_destroy.restype = [vp], i
    L.ar_allreduce_peer.argtypes, L.ar_allreduce_peer.restype = [vp, vp, vp, sz, i, i, vp], i
    if hasattr(L, "ar_comm_create_local"):   # the test build only
        L.ar_comm_create_local.argtypes = [i, i, pvp, sz, sz, ctypes.POINTER(vp)]
        L.ar_comm_create_local.restype = i
    _lib = L
    return L


# ------------------------------------------------------------------ helpers

def dtype_code(dtype: torch.dtype) -> int:
    try:
        return _TORCH_TO_AR[dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {dtype}; expected float32, float16 or bfloat16") from None


def _code(dtype) -> int:
    """An ar_dtype code, given as one or as a torch dtype."""
    return dtype if isinstance(dtype, int) else dtype_code(dtype)


_STRATEGY_CODES = {**STRATEGIES, **{k.lower(): v for k, v in STRATEGIES.items()}}


def _strategy(s) -> int:
    if isinstance(s, str):
        code = _STRATEGY_CODES.get(s)
        return code if code is not None else STRATEGIES[s.upper()]
    return int(s)


def _ptr_array(ptrs):
    return (ctypes.c_void_p * max(1, len(ptrs)))(*ptrs)


def _dev_ptr(t: Optional[torch.Tensor], what: str) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


# The raw handle of the current device's current stream, without building a
# torch.cuda.Stream object (the public route costs a few microseconds a call).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_get_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        if _raw_stream is not None and _get_device is not None:
            return _raw_stream(_get_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(func: str, status: int):
    if status != AR_OK:
        raise ARError(func, status)


def _fused_pointers(partials, residual, weight, bias, out, residual_out, host=False):
    """Pointers of a fused call's tensors, in one pass that checks each: the size and dtype the call
    reads or writes (the library trusts its pointers, so a short or wrongly typed tensor would be
    read or written past its end), contiguity, and the device (residual's GPU; the host for host
    calls).  Names are built only for an error message.

    Returns (tokens, hidden, partial pointer array, bias, residual, weight, out, residual_out)."""
    if residual.dim() != 2:
        raise ValueError("residual must be [tokens, hidden]")
    if len(partials) == 0:
        raise ValueError("at least one partial is needed")
    tokens, hidden = residual.shape
    n = tokens * hidden
    dt = residual.dtype
    dev = residual.get_device()
    if host != (dev < 0):
        raise ValueError("residual must be a host (CPU) tensor" if host else "residual must be a CUDA tensor")

    def fail(name, numel):
        where = "the host" if host else f"cuda:{dev}"
        raise ValueError(f"{name} must be a contiguous tensor of {numel} {dt} elements on {where}")

    addrs = []
    for p in partials:
        if p.numel() != n or p.dtype != dt or p.get_device() != dev or not p.is_contiguous():
            fail(f"partials[{len(addrs)}]", n)
        addrs.append(p.data_ptr())
    got = [None] * 5
    for i, (t, numel) in enumerate(((bias, hidden), (residual, n), (weight, hidden), (out, n), (residual_out, n))):
        if t is not None:
            if t.numel() != numel or t.dtype != dt or t.get_device() != dev or not t.is_contiguous():
                fail(("bias", "residual", "weight", "out", "residual_out")[i], numel)
            got[i] = t.data_ptr()
    return (tokens, hidden, _ptr_array(addrs), *got)


# ------------------------------------------------------------------ the ABI

def ar_version() -> int:
    return lib().ar_version()


def ar_strerror(code: int) -> str:
    return lib().ar_strerror(code).decode()


def ar_device_status() -> int:
    """AR_OK, or AR_ERR_TIMEOUT if a kernel gave up a bounded wait since the last call (synchronous)."""
    return lib().ar_device_status()


def ar_workspace_size(R: int, n: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return int(lib().ar_workspace_size(R, n, code))


def ar_workspace_size_rows(R: int, hidden: int, tokens: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return int(lib().ar_workspace_size_rows(R, hidden, tokens, code))


def ar_query_strategy(R: int, n: int, hidden: int, dtype, fusion_op: int = AR_FUSION_RESIDUAL_RMS_NORM):
    """(strategy code, warps per token) that AR_AUTO picks for this shape."""
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    chosen, warps = ctypes.c_int(0), ctypes.c_int(0)
    _check("ar_query_strategy",
           lib().ar_query_strategy(R, n, hidden, code, fusion_op, ctypes.byref(chosen), ctypes.byref(warps)))
    return chosen.value, warps.value


def ar_query_launch(R: int, hidden: int, tokens: int, dtype, strategy="AUTO") -> dict:
    """The kernel and launch shape ar_residual_rmsnorm would use (aligned pointers, workspace given)."""
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    plan = ArLaunchPlan()
    _check("ar_query_launch", lib().ar_query_launch(R, hidden, tokens, code, _strategy(strategy), ctypes.byref(plan)))
    d = {name: getattr(plan, name) for name, _ in ArLaunchPlan._fields_}
    d["kernel_name"] = KERNEL_NAMES.get(plan.kernel, "?")
    return d


def ar_sum(partials: Sequence[torch.Tensor], out: Optional[torch.Tensor] = None,
           strategy="AUTO", stream=None) -> torch.Tensor:
    """out = sum of the R partial tensors (same shape, dtype and device)."""
    if len(partials) == 0:
        raise ValueError("ar_sum needs at least one partial")
    p0 = partials[0]
    shape, dt, device = p0.shape, p0.dtype, p0.device
    for k, p in enumerate(partials):
        if p.shape != shape or p.dtype != dt or p.device != device:
            raise ValueError(f"partials[{k}] does not match partials[0] in shape, dtype or device")
    if out is None:
        out = torch.empty_like(p0)
    elif out.numel() != p0.numel() or out.dtype != p0.dtype or out.device != device:
        raise ValueError("out must match the partials in size, dtype and device")
    ptrs = _ptr_array([_dev_ptr(p, f"partials[{k}]") for k, p in enumerate(partials)])
    status = lib().ar_sum(ptrs, len(partials), _dev_ptr(out, "out"), p0.numel(), dtype_code(p0.dtype),
                          _strategy(strategy), _stream_handle(stream))
    _check("ar_sum", status)
    return out


def ar_residual_rmsnorm(partials: Sequence[torch.Tensor], residual: torch.Tensor, weight: torch.Tensor,
                        eps: float, bias: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None, residual_out: Optional[torch.Tensor] = None,
                        intermediate: Optional[torch.Tensor] = None, strategy="AUTO", stream=None):
    """(out, residual_out) of the fused sum + bias + residual + RMSNorm over [tokens, hidden] rows.

    ``intermediate`` is the two-shot workspace (any CUDA tensor of at least
    ar_workspace_size_rows(...) bytes); when it is None and the strategy may
    take the two-shot path, one is allocated with torch.
    """
    if out is None:
        out = torch.empty_like(residual)
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    tokens, hidden, ptrs, p_bias, p_res, p_w, p_out, p_rout = _fused_pointers(
        partials, residual, weight, bias, out, residual_out)
    code = dtype_code(residual.dtype)
    st = _strategy(strategy)
    if intermediate is None and st in (AR_TWOSHOT, AR_AUTO):
        need = ar_workspace_size_rows(len(partials), hidden, tokens, code)
        if need:
            intermediate = torch.empty(need, dtype=torch.uint8, device=residual.device)
    ws_ptr = _dev_ptr(intermediate, "intermediate")
    ws_bytes = 0 if intermediate is None else intermediate.numel() * intermediate.element_size()
    status = lib().ar_residual_rmsnorm(ptrs, len(partials), p_bias, p_res, p_w, eps, hidden, tokens, p_out, p_rout,
                                       ws_ptr, ws_bytes, code, st, _stream_handle(stream))
    _check("ar_residual_rmsnorm", status)
    return out, residual_out


def ar_residual_rmsnorm_noalloc(partials: Sequence[torch.Tensor], residual: torch.Tensor, weight: torch.Tensor,
                                eps: float, bias: Optional[torch.Tensor] = None,
                                out: torch.Tensor = None, residual_out: torch.Tensor = None, stream=None):
    """(out, residual_out) of the two-shot fused call whose scratch is the library's own array.

    For callers that must not allocate device memory during the call: ``out``
    and ``residual_out`` are required (this wrapper creates no tensor either).
    Accepts shapes with ar_workspace_size_rows(...) <= AR_NOALLOC_SCRATCH_BYTES.
    """
    if out is None or residual_out is None:
        raise ValueError("out and residual_out must be given: this call allocates nothing")
    tokens, hidden, ptrs, p_bias, p_res, p_w, p_out, p_rout = _fused_pointers(
        partials, residual, weight, bias, out, residual_out)
    status = lib().ar_residual_rmsnorm_noalloc(ptrs, len(partials), p_bias, p_res, p_w, ctypes.c_float(eps), hidden,
                                               tokens, p_out, p_rout, dtype_code(residual.dtype),
                                               _stream_handle(stream))
    _check("ar_residual_rmsnorm_noalloc", status)
    return out, residual_out


def ar_rmsnorm(x: torch.Tensor, weight: torch.Tensor, eps: float, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """out = RMSNorm of the [tokens, hidden] rows of x, times weight (out may be x)."""
    if x.dim() != 2:
        raise ValueError("x must be [tokens, hidden]")
    tokens, hidden = x.shape
    if weight.numel() != hidden or weight.dtype != x.dtype or weight.device != x.device:
        raise ValueError("weight must be [hidden] of x's dtype, on x's device")
    if out is None:
        out = torch.empty_like(x)
    elif out.numel() != x.numel() or out.dtype != x.dtype or out.device != x.device:
        raise ValueError("out must match x in size, dtype and device")
    _check("ar_rmsnorm", lib().ar_rmsnorm(_dev_ptr(x, "x"), _dev_ptr(weight, "weight"), ctypes.c_float(eps), hidden,
                                          tokens, _dev_ptr(out, "out"), dtype_code(x.dtype), _stream_handle(stream)))
    return out


def ar_host_staging_size(R: int, hidden: int, chunk_tokens: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return int(lib().ar_host_staging_size(R, hidden, chunk_tokens, code))


def _host_ptr(t: Optional[torch.Tensor], what: str) -> Optional[int]:
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError(f"{what} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def ar_residual_rmsnorm_host(partials: Sequence[torch.Tensor], residual: torch.Tensor, weight: torch.Tensor,
                             eps: float, staging: torch.Tensor, out: torch.Tensor, residual_out: torch.Tensor,
                             bias: Optional[torch.Tensor] = None, chunk_tokens: int = 512, strategy="AUTO",
                             stream=None):
    """The fused call on host (preferably pinned) tensors, copies pipelined through device `staging`.

    Asynchronous: synchronise `stream` before reading out / residual_out.
    """
    if out is None or residual_out is None:
        raise ValueError("out and residual_out must be given (host tensors)")
    tokens, hidden, ptrs, p_bias, p_res, p_w, p_out, p_rout = _fused_pointers(
        partials, residual, weight, bias, out, residual_out, host=True)
    status = lib().ar_residual_rmsnorm_host(
        ptrs, len(partials), p_bias, p_res, p_w, ctypes.c_float(eps), hidden, tokens, p_out, p_rout,
        _dev_ptr(staging, "staging"), staging.numel() * staging.element_size(), chunk_tokens,
        dtype_code(residual.dtype), _strategy(strategy), _stream_handle(stream))
    _check("ar_residual_rmsnorm_host", status)
    return out, residual_out


def ar_allreduce(params: ArParams, fusion_op: int, strategy="AUTO", stream=None) -> None:
    """Calls ar_allreduce with a filled ArParams structure (raw device pointers)."""
    _check("ar_allreduce", lib().ar_allreduce(ctypes.byref(params), fusion_op, _strategy(strategy),
                                              _stream_handle(stream)))


def ar_config_workspace_size(R: int, n: int, hidden: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else dtype_code(dtype)
    return int(lib().ar_config_workspace_size(R, n, hidden, code))


def ar_allreduce_config(params: ArParams, fusion_op: int, strategy="AUTO", config: int = 0, stream=None) -> None:
    """Calls ar_allreduce_config (AllReduceStrategyConfig flags in `config`) with a filled ArParams."""
    _check("ar_allreduce_config", lib().ar_allreduce_config(ctypes.byref(params), fusion_op, _strategy(strategy),
                                                            config, _stream_handle(stream)))


def make_params(partials, out, *, bias=None, residual=None, weight=None, eps=0.0, hidden=0,
                residual_out=None, workspace=None) -> ArParams:
    """Fills an ArParams from tensors (marshalling only)."""
    p = ArParams()
    for k, t in enumerate(partials):
        p.partials[k] = _dev_ptr(t, f"partials[{k}]")
    p.R = len(partials)
    p.dtype = dtype_code(partials[0].dtype)
    p.n = partials[0].numel()
    p.out = _dev_ptr(out, "out")
    p.bias = _dev_ptr(bias, "bias")
    p.residual = _dev_ptr(residual, "residual")
    p.weight = _dev_ptr(weight, "weight")
    p.eps = eps
    p.hidden = hidden
    p.residual_out = _dev_ptr(residual_out, "residual_out")
    p.workspace = _dev_ptr(workspace, "workspace")
    p.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return p


def ar_lamport_buffer_size(R: int, hidden: int, tokens: int, dtype) -> int:
    """Bytes of the Lamport buffer for R partials of [tokens, hidden] (0 for bad arguments)."""
    return int(lib().ar_lamport_buffer_size(R, hidden, tokens, _code(dtype)))


def ar_lamport_init(buffer: torch.Tensor, dtype, stream=None) -> torch.Tensor:
    """Fills the whole CUDA tensor ``buffer`` with the empty marker of ``dtype`` (negative zero)."""
    nbytes = buffer.numel() * buffer.element_size()
    _check("ar_lamport_init", lib().ar_lamport_init(_dev_ptr(buffer, "buffer"), nbytes, _code(dtype),
                                                    _stream_handle(stream)))
    return buffer


def ar_lamport_supported(R: int, hidden: int, tokens: int, dtype) -> Optional[int]:
    """Warps per row of the Lamport call for this shape, or None if it cannot take the shape."""
    w = ctypes.c_int(0)
    status = lib().ar_lamport_supported(R, hidden, tokens, _code(dtype), ctypes.byref(w))
    if status == AR_ERR_UNSUPPORTED:
        return None
    _check("ar_lamport_supported", status)
    return w.value


def lamport_buffer(R: int, hidden: int, tokens: int, dtype: torch.dtype, device=None) -> torch.Tensor:
    """A new device buffer for ar_residual_rmsnorm_lamport, filled with the empty marker."""
    nbytes = ar_lamport_buffer_size(R, hidden, tokens, dtype)
    if nbytes == 0:
        raise ValueError("no Lamport buffer for this shape")
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device if device is not None else "cuda")
    return ar_lamport_init(buf, dtype)


def ar_residual_rmsnorm_lamport(partials: Sequence[torch.Tensor], residual: torch.Tensor, weight: torch.Tensor,
                                eps: float, bias: Optional[torch.Tensor] = None,
                                out: Optional[torch.Tensor] = None, residual_out: Optional[torch.Tensor] = None,
                                buffer: Optional[torch.Tensor] = None, stream=None):
    """(out, residual_out) of the fused op through the Lamport protocol.

    ``buffer`` is the marker-filled Lamport buffer (see lamport_buffer); every
    completed call leaves it filled again, so one buffer serves a sequence of
    calls on one stream.  When it is None a new one is made for this call.
    """
    if out is None:
        out = torch.empty_like(residual)
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    tokens, hidden, ptrs, p_bias, p_res, p_w, p_out, p_rout = _fused_pointers(
        partials, residual, weight, bias, out, residual_out)
    if buffer is None:
        buffer = lamport_buffer(len(partials), hidden, tokens, residual.dtype, residual.device)
    status = lib().ar_residual_rmsnorm_lamport(
        ptrs, len(partials), p_bias, p_res, p_w, ctypes.c_float(eps), hidden, tokens, p_out, p_rout,
        _dev_ptr(buffer, "buffer"), buffer.numel() * buffer.element_size(), dtype_code(residual.dtype),
        _stream_handle(stream))
    _check("ar_residual_rmsnorm_lamport", status)
    return out, residual_out


# ------------------------------------------------------------ the all-reduce across GPUs (one process per GPU)

def ar_comm_buffer_size(world: int, max_bytes: int) -> int:
    """Bytes each rank registers for an all-reduce of up to max_bytes (0 for bad arguments)."""
    return int(lib().ar_comm_buffer_size(world, max_bytes))


def ar_comm_export(buffer: torch.Tensor) -> bytes:
    """The CUDA IPC handle of a registered buffer, as AR_IPC_HANDLE_BYTES bytes."""
    h = ctypes.create_string_buffer(AR_IPC_HANDLE_BYTES)
    _check("ar_comm_export", lib().ar_comm_export(_dev_ptr(buffer, "buffer"), h))
    return h.raw


def gather_handles(handle: bytes, all_gather_object, world: int) -> bytes:
    """Every rank's handle, in rank order, as one byte string of world * AR_IPC_HANDLE_BYTES bytes.

    ``all_gather_object(out_list, obj)`` is the collective that fills out_list with every rank's obj
    in rank order (torch.distributed.all_gather_object, or any equivalent)."""
    if len(handle) != AR_IPC_HANDLE_BYTES:
        raise ValueError("an IPC handle has AR_IPC_HANDLE_BYTES bytes")
    got = [None] * world
    all_gather_object(got, handle)
    if any(not isinstance(h, (bytes, bytearray)) or len(h) != AR_IPC_HANDLE_BYTES for h in got):
        raise ValueError("a rank sent no valid handle")
    return b"".join(bytes(h) for h in got)


class PeerComm:
    """This rank's side of the all-reduce across the GPUs of one node (one process per GPU).

    Registers a device buffer, exchanges its IPC handle with the other ranks
    through ``all_gather_object`` and ``barrier`` (torch.distributed's by
    default), and maps the peers' buffers (ar_comm_create).  allreduce(x)
    then returns the sum over the ranks of every rank's x, on every rank.
    """

    def __init__(self, rank: int, world: int, max_bytes: int, device=None, all_gather_object=None, barrier=None):
        self.rank, self.world, self.max_bytes = rank, world, max_bytes
        nbytes = ar_comm_buffer_size(world, max_bytes)
        if nbytes == 0:
            raise ValueError("bad world size or max_bytes")
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=device if device is not None else "cuda")
        handles = None
        if world > 1:
            if all_gather_object is None or barrier is None:
                import torch.distributed as dist
                all_gather_object = all_gather_object or dist.all_gather_object
                barrier = barrier or dist.barrier
            handles = gather_handles(ar_comm_export(self.buffer), all_gather_object, world)
        comm = ctypes.c_void_p(0)
        _check("ar_comm_create", lib().ar_comm_create(rank, world, _dev_ptr(self.buffer, "buffer"), nbytes,
                                                      max_bytes, handles, ctypes.byref(comm)))
        self._comm = comm
        if world > 1:
            barrier()   # every rank's flag words are zeroed before any rank signals into them

    def allreduce(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, strategy="AUTO",
                  stream=None) -> torch.Tensor:
        if self._comm is None:
            raise RuntimeError("the communicator is closed")
        if out is None:
            out = torch.empty_like(x)
        if out.numel() != x.numel() or out.dtype != x.dtype or not x.is_contiguous() or not out.is_contiguous():
            raise ValueError("out must be a contiguous tensor of x's size and dtype")
        _check("ar_allreduce_peer", lib().ar_allreduce_peer(self._comm, _dev_ptr(x, "x"), _dev_ptr(out, "out"),
                                                            x.numel(), dtype_code(x.dtype), _strategy(strategy),
                                                            _stream_handle(stream)))
        return out

    def close(self) -> None:
        if self._comm is not None:
            _check("ar_comm_destroy", lib().ar_comm_destroy(self._comm))
            self._comm = None

    def __del__(self):
        try:
            self.close()
        except Exception:   # pragma: no cover - interpreter teardown
            pass
