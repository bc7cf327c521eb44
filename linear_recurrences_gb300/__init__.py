"""Python binding of the GB300 selective-scan library (libss.so, include/ss.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI. PyTorch provides device memory and streams.
There is no CPU fallback: if the library was not built, or no CUDA device is
present, the calls raise.

Functions keep the C names:
  ss_affine_scan(a, b, h=None, workspace=None, stream=None) -> h
  ss_selective_scan_fwd(x, delta, Bt, Ct, A, Dskip=None, delta_softplus=False, y=None, ...)
  ss_selective_scan_bidir(...same...)
  ss_get_device_status(workspace, stream=None) -> status code
plus workspace helpers. Tensors must be contiguous CUDA tensors: fp32 for the
affine scan; fp32 or bf16 (all of x, delta, Bt, Ct, y alike) for S6, with A
and Dskip fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "SS_OK", "SS_ERR_INVALID", "SS_ERR_UNSUPPORTED", "SS_ERR_WORKSPACE", "SS_ERR_CUDA",
    "SS_ERR_TIMEOUT", "SS_ERR_BOUNDS", "SS_F32", "SS_BF16", "SSError", "lib", "library_path",
    "ss_status_string", "ss_abi_version", "ss_affine_scan_workspace_bytes", "ss_affine_scan",
    "ss_selective_scan_workspace_bytes", "ss_selective_scan_fwd", "ss_selective_scan_bidir",
    "ss_get_device_status", "ss_set_spin_timeout_ns", "ss_testing_skip_publish_once",
    "ss_testing_s6_plan", "ss_testing_s6_describe_plan", "ss_testing_proj_gemm",
    "ss_testing_proj_gemm_describe_plan",
    "ss_probe_mufu_ex2", "ss_affine_scan_noalloc", "ss_affine_scan_noalloc_status",
    "SS_AFFINE_NOALLOC_MAX_N",
    "ss_selective_scan_fwd_state", "ss_selective_scan_bwd", "ss_selective_scan_bwd_workspace_bytes",
    "ss_selective_scan_layer_fwd", "ss_selective_scan_layer_workspace_bytes",
    "ss_affine_scan_log_step", "ss_affine_scan_state", "ss_affine_scan_host",
    "ss_affine_scan_host_workspace_bytes", "new_workspace", "EXPORTED_SYMBOLS",
]

SS_OK, SS_ERR_INVALID, SS_ERR_UNSUPPORTED, SS_ERR_WORKSPACE = 0, 1, 2, 3
SS_ERR_CUDA, SS_ERR_TIMEOUT, SS_ERR_BOUNDS = 4, 5, 6
SS_F32, SS_BF16 = 0, 1

EXPORTED_SYMBOLS = (
    "ss_status_string", "ss_abi_version", "ss_affine_scan_workspace_bytes", "ss_affine_scan",
    "ss_selective_scan_workspace_bytes", "ss_selective_scan_fwd", "ss_selective_scan_bidir",
    "ss_get_device_status", "ss_set_spin_timeout_ns", "ss_testing_skip_publish_once",
    "ss_testing_s6_plan", "ss_testing_s6_describe_plan", "ss_testing_proj_gemm",
    "ss_testing_proj_gemm_describe_plan",
    "ss_probe_mufu_ex2", "ss_affine_scan_noalloc", "ss_affine_scan_noalloc_status",
    "ss_selective_scan_fwd_state",
    "ss_selective_scan_bwd_workspace_bytes", "ss_selective_scan_bwd",
    "ss_selective_scan_layer_workspace_bytes", "ss_selective_scan_layer_fwd",
    "ss_affine_scan_log_step", "ss_affine_scan_state", "ss_affine_scan_host_workspace_bytes",
    "ss_affine_scan_host",
)

_PKG = os.path.dirname(os.path.abspath(__file__))
_DEFAULT_LIB = os.path.join(_PKG, "_build", "libss.so")
_lock = threading.Lock()
_lib = None
_plan_generation = 0  # bumped by ss_testing_s6_plan: cached S6 workspaces are keyed on it


class SSError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {ss_status_string(status)} ({status})")


def library_path() -> str:
    return os.environ.get("SS_LIBRARY", _DEFAULT_LIB)


def lib() -> ctypes.CDLL:
    """The loaded libss.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libss.so not found at {path}; build it with "
                    "`python -m linear_recurrences_gb300.build`")
            _lib = _bind(ctypes.CDLL(path))
        return _lib


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    vp, i64, sz, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
    L.ss_status_string.argtypes = [ci]
    L.ss_status_string.restype = ctypes.c_char_p
    L.ss_abi_version.argtypes = []
    L.ss_abi_version.restype = ci
    L.ss_affine_scan_workspace_bytes.argtypes = [i64]
    L.ss_affine_scan_workspace_bytes.restype = sz
    L.ss_affine_scan.argtypes = [vp, vp, vp, i64, vp, sz, vp]
    L.ss_affine_scan.restype = ci
    L.ss_selective_scan_workspace_bytes.argtypes = [i64, i64, i64, i64, ci, ci]
    L.ss_selective_scan_workspace_bytes.restype = sz
    s6 = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, ci, ci, vp, sz, vp]
    L.ss_selective_scan_fwd.argtypes = s6
    L.ss_selective_scan_fwd.restype = ci
    L.ss_selective_scan_bidir.argtypes = s6
    L.ss_selective_scan_bidir.restype = ci
    L.ss_get_device_status.argtypes = [vp, vp]
    L.ss_get_device_status.restype = ci
    L.ss_set_spin_timeout_ns.argtypes = [ctypes.c_uint64]
    L.ss_set_spin_timeout_ns.restype = ci
    L.ss_testing_skip_publish_once.argtypes = [i64]
    L.ss_testing_skip_publish_once.restype = None
    L.ss_testing_s6_plan.argtypes = [ci, ci, ci, ci]
    L.ss_testing_s6_plan.restype = None
    L.ss_testing_s6_describe_plan.argtypes = [i64, i64, i64, i64, ci, ci,
                                              ctypes.POINTER(ctypes.c_int64)]
    L.ss_testing_s6_describe_plan.restype = ci
    L.ss_testing_proj_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, vp]
    L.ss_testing_proj_gemm.restype = ci
    L.ss_testing_proj_gemm_describe_plan.argtypes = [i64, i64, i64, ctypes.POINTER(ctypes.c_int64)]
    L.ss_testing_proj_gemm_describe_plan.restype = ci
    L.ss_probe_mufu_ex2.argtypes = [vp, ci, ci, vp]
    L.ss_probe_mufu_ex2.restype = ci
    L.ss_affine_scan_noalloc.argtypes = [vp, vp, vp, i64, vp]
    L.ss_affine_scan_noalloc.restype = ci
    L.ss_affine_scan_noalloc_status.argtypes = [vp]
    L.ss_affine_scan_noalloc_status.restype = ci
    L.ss_selective_scan_fwd_state.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                              i64, ci, ci, vp, sz, vp]
    L.ss_selective_scan_fwd_state.restype = ci
    L.ss_selective_scan_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64]
    L.ss_selective_scan_bwd_workspace_bytes.restype = sz
    L.ss_selective_scan_bwd.argtypes = [vp] * 16 + [i64, i64, i64, i64, ci, ci, vp, sz, vp]
    L.ss_selective_scan_bwd.restype = ci
    L.ss_selective_scan_layer_workspace_bytes.argtypes = [i64, i64, i64, i64, ci]
    L.ss_selective_scan_layer_workspace_bytes.restype = sz
    L.ss_selective_scan_layer_fwd.argtypes = [vp] * 6 + [i64, i64, i64, i64, ci, vp, sz, vp]
    L.ss_selective_scan_layer_fwd.restype = ci
    L.ss_affine_scan_log_step.argtypes = [vp, vp, vp, i64, vp, sz, vp]
    L.ss_affine_scan_log_step.restype = ci
    L.ss_affine_scan_state.argtypes = [vp, vp, vp, i64, vp, vp, sz, vp]
    L.ss_affine_scan_state.restype = ci
    L.ss_affine_scan_host_workspace_bytes.argtypes = [i64]
    L.ss_affine_scan_host_workspace_bytes.restype = sz
    L.ss_affine_scan_host.argtypes = [vp, vp, vp, i64, vp, sz, vp]
    L.ss_affine_scan_host.restype = ci
    return L


def ss_status_string(status: int) -> str:
    try:
        return lib().ss_status_string(int(status)).decode()
    except RuntimeError:
        return str(status)


def ss_abi_version() -> int:
    return lib().ss_abi_version()


def ss_set_spin_timeout_ns(ns: int) -> None:
    st = lib().ss_set_spin_timeout_ns(int(ns))
    if st != SS_OK:
        raise SSError(st, "ss_set_spin_timeout_ns")


def ss_testing_skip_publish_once(unit: int) -> None:
    """Test hook (include/ss_testing.h): the next launch lets work unit `unit`
    skip publishing its look-back descriptors, so waits on it time out."""
    lib().ss_testing_skip_publish_once(int(unit))


def ss_testing_s6_plan(kind: int = 0, a: int = 0, b: int = 0, c: int = 0) -> None:
    """Test hook (include/ss_testing.h): forces the S6 plan for later calls;
    kind 0 restores the planner's choice, 1 = chunked (warps per CTA,
    timesteps per warp, lanes per channel), 2 = time-parallel (channels per
    warp, steps per lane, warps per CTA), 3 = wavefront (steps per slice,
    slices per CTA)."""
    global _plan_generation
    lib().ss_testing_s6_plan(int(kind), int(a), int(b), int(c))
    _plan_generation += 1


def ss_testing_s6_describe_plan(B, L, D, N, io_dtype=SS_F32, bidir=False):
    """(kind, six parameters) of the plan an S6 call of this shape would use:
    kind 2 = wavefront (steps per slice, slices, channels per CTA, blocks per
    sequence, CTAs, steps per block), 1 = time-parallel (channels per warp, steps per lane, warps per CTA,
    blocks per sequence, CTAs, steps per block), 0 = chunked (lanes per
    channel, warps per CTA, timesteps per warp, chunks, CTAs, states per
    lane)."""
    out = (ctypes.c_int64 * 6)()
    k = lib().ss_testing_s6_describe_plan(int(B), int(L), int(D), int(N), int(io_dtype),
                                          int(bool(bidir)), out)
    return k, tuple(out)


def ss_testing_proj_gemm_describe_plan(M, K, Nout):
    """Launch plan of the projection GEMM for an M x K by Nout x K product,
    computed on the host: (N-tile width, N-tiles, K-columns per stage,
    K-blocks, stages, pair (1/0), work units, dynamic shared memory bytes),
    or None for an invalid shape."""
    out = (ctypes.c_int64 * 8)()
    if lib().ss_testing_proj_gemm_describe_plan(int(M), int(K), int(Nout), out) != 0:
        return None
    return tuple(out)


def ss_testing_proj_gemm(x, W, bias=None, out=None, ld_out=None, workspace=None, stream=None):
    """Test hook (include/ss_testing.h): the layer's projection GEMM alone.
    x (M, K) and W (Nout, K) bf16 CUDA tensors; bias fp32 (n_bias,) added to
    the first n_bias columns; returns out (M, ld_out) bf16 (columns from the
    multiple of 8 at or above Nout are left untouched)."""
    torch = _torch()
    _check_cuda(x, "x", (torch.bfloat16,))
    _check_cuda(W, "W", (torch.bfloat16,))
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1] or x.device != W.device:
        raise ValueError("x must be (M, K) and W (Nout, K) on one device")
    M, K = x.shape
    Nout = W.shape[0]
    ld = int(ld_out) if ld_out is not None else Nout
    if out is None:
        out = torch.zeros((M, ld), dtype=torch.bfloat16, device=x.device)
    _check_cuda(out, "out", (torch.bfloat16,))
    if bias is not None:
        _check_cuda(bias, "bias", (torch.float32,))
    if workspace is None:
        workspace = new_workspace(256, x.device)
    with torch.cuda.device(x.device):
        st = lib().ss_testing_proj_gemm(_ptr(x), _ptr(W), _ptr(out), _ptr(bias),
                                        0 if bias is None else bias.numel(), M, K, Nout, ld,
                                        _ptr(workspace), _stream_handle(stream, x.device))
    if st != SS_OK:
        raise SSError(st, "ss_testing_proj_gemm")
    return out


def ss_probe_mufu_ex2(out, blocks: int, iters: int, stream=None) -> None:
    """Measurement kernel (include/ss_probe.h): blocks*256*8*iters MUFU ex2 ops."""
    sh = _stream_handle(stream, out.device)
    st = lib().ss_probe_mufu_ex2(_ptr(out), int(blocks), int(iters), sh)
    if st != SS_OK:
        raise SSError(st, "ss_probe_mufu_ex2")


# ---------------------------------------------------------------- torch glue
def _torch():
    import torch
    return torch


def _stream_handle(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(t, name, dtypes):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None and t.numel() > 0 else 0)


_ws_cache: dict = {}


def new_workspace(nbytes: int, device):
    """A zero-filled, 256-byte aligned device workspace of at least nbytes."""
    torch = _torch()
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _cached_workspace(key, nbytes, device, stream_handle):
    """One zeroed workspace per (entry point, shape, device, stream), reused
    across calls as the C ABI allows."""
    full = (key, str(device), stream_handle.value)
    ws = _ws_cache.get(full)
    if ws is None or ws.numel() < nbytes:
        ws = new_workspace(nbytes, device)
        _ws_cache[full] = ws
    return ws


def ss_affine_scan_workspace_bytes(n: int) -> int:
    return lib().ss_affine_scan_workspace_bytes(int(n))


def ss_affine_scan(a, b, h=None, workspace=None, stream=None, _fn="ss_affine_scan"):
    """h[t] = a[t]*h[t-1] + b[t] (fp32, 1-D, on the GPU). Returns h."""
    torch = _torch()
    _check_cuda(a, "a", (torch.float32,))
    _check_cuda(b, "b", (torch.float32,))
    if a.dim() != 1 or a.shape != b.shape or a.device != b.device:
        raise ValueError("a and b must be 1-D, same length, same device")
    n = a.numel()
    if h is None:
        h = torch.empty_like(a)
    _check_cuda(h, "h", (torch.float32,))
    if h.shape != a.shape:
        raise ValueError("h must match a")
    sh = _stream_handle(stream, a.device)
    need = ss_affine_scan_workspace_bytes(n)
    if workspace is None and need:
        workspace = _cached_workspace(("affine",), need, a.device, sh)
    wsb = workspace.numel() if workspace is not None else 0
    st = getattr(lib(), _fn)(_ptr(a), _ptr(b), _ptr(h), n, _ptr(workspace), wsb, sh)
    if st != SS_OK:
        raise SSError(st, _fn)
    return h


def ss_affine_scan_log_step(a, b, h=None, workspace=None, stream=None):
    """The affine scan with a log-step (Hillis-Steele) scan of each tile: a
    comparison kernel for the work-efficient ss_affine_scan."""
    return ss_affine_scan(a, b, h, workspace, stream, _fn="ss_affine_scan_log_step")


def ss_affine_scan_state(a, b, h0=None, h=None, workspace=None, stream=None):
    """The affine scan from h[-1] = h0: h0 is a 1-element fp32 CUDA tensor
    (read when the kernel runs) or None for 0. Returns h."""
    torch = _torch()
    _check_cuda(a, "a", (torch.float32,))
    _check_cuda(b, "b", (torch.float32,))
    if a.dim() != 1 or a.shape != b.shape or a.device != b.device:
        raise ValueError("a and b must be 1-D, same length, same device")
    if h0 is not None:
        _check_cuda(h0, "h0", (torch.float32,))
        if h0.numel() != 1 or h0.device != a.device:
            raise ValueError("h0 must hold one float on a's device")
    n = a.numel()
    if h is None:
        h = torch.empty_like(a)
    _check_cuda(h, "h", (torch.float32,))
    if h.shape != a.shape:
        raise ValueError("h must match a")
    sh = _stream_handle(stream, a.device)
    need = ss_affine_scan_workspace_bytes(n)
    if workspace is None and need:
        workspace = _cached_workspace(("affine_state",), need, a.device, sh)
    wsb = workspace.numel() if workspace is not None else 0
    st = lib().ss_affine_scan_state(_ptr(a), _ptr(b), _ptr(h), n, _ptr(h0), _ptr(workspace),
                                    wsb, sh)
    if st != SS_OK:
        raise SSError(st, "ss_affine_scan_state")
    return h


def ss_affine_scan_host_workspace_bytes(n: int) -> int:
    return lib().ss_affine_scan_host_workspace_bytes(int(n))


def _check_host(t, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32 or t.dim() != 1:
        raise ValueError(f"{name} must be a contiguous 1-D float32 host tensor")


def ss_affine_scan_host(a, b, h=None, workspace=None, stream=None, device=None):
    """The affine scan of HOST tensors (best pinned: torch's pin_memory()),
    streamed through the GPU in chunks with copies in both directions
    overlapping the scans. Returns h (a host tensor); it is complete once
    `stream` (default: the current stream of `device`) is."""
    torch = _torch()
    _check_host(a, "a")
    _check_host(b, "b")
    if a.shape != b.shape:
        raise ValueError("a and b must have the same length")
    n = a.numel()
    if h is None:
        h = torch.empty(n, dtype=torch.float32, pin_memory=True)
    _check_host(h, "h")
    if h.shape != a.shape:
        raise ValueError("h must match a")
    dev = torch.device(device) if device is not None else (
        workspace.device if workspace is not None else torch.device("cuda", torch.cuda.current_device()))
    sh = _stream_handle(stream, dev)
    need = ss_affine_scan_host_workspace_bytes(n)
    if workspace is None and need:
        workspace = _cached_workspace(("affine_host",), need, dev, sh)
    wsb = workspace.numel() if workspace is not None else 0
    with torch.cuda.device(dev):
        st = lib().ss_affine_scan_host(_ptr(a), _ptr(b), _ptr(h), n, _ptr(workspace), wsb, sh)
    if st != SS_OK:
        raise SSError(st, "ss_affine_scan_host")
    return h


SS_AFFINE_NOALLOC_MAX_N = 1 << 24


def ss_affine_scan_noalloc(a, b, h=None, stream=None):
    """ss_affine_scan with the library's static scratch array instead of a
    workspace (for callers that must not allocate device memory; see
    include/ss.h). n <= SS_AFFINE_NOALLOC_MAX_N."""
    torch = _torch()
    _check_cuda(a, "a", (torch.float32,))
    _check_cuda(b, "b", (torch.float32,))
    if a.dim() != 1 or a.shape != b.shape or a.device != b.device:
        raise ValueError("a and b must be 1-D, same length, same device")
    if h is None:
        h = torch.empty_like(a)
    _check_cuda(h, "h", (torch.float32,))
    with torch.cuda.device(a.device):
        st = lib().ss_affine_scan_noalloc(_ptr(a), _ptr(b), _ptr(h), a.numel(),
                                          _stream_handle(stream, a.device))
    if st != SS_OK:
        raise SSError(st, "ss_affine_scan_noalloc")
    return h


def ss_affine_scan_noalloc_status(stream=None, device=None) -> int:
    """Synchronises `stream`, then reads and clears the device-side error word
    of the static scratch used by ss_affine_scan_noalloc on `device` (the
    current CUDA device by default): SS_OK or SS_ERR_TIMEOUT."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    with torch.cuda.device(dev):
        return lib().ss_affine_scan_noalloc_status(_stream_handle(stream, dev))


def ss_selective_scan_workspace_bytes(B, L, D, N, io_dtype=SS_F32, bidir=False) -> int:
    return lib().ss_selective_scan_workspace_bytes(int(B), int(L), int(D), int(N),
                                                   int(io_dtype), int(bool(bidir)))


def _s6(fn_name, x, delta, Bt, Ct, A, Dskip, delta_softplus, y, workspace, stream, bidir,
        state=None):
    torch = _torch()
    io = (torch.float32, torch.bfloat16)
    for t, nm in ((x, "x"), (delta, "delta"), (Bt, "Bt"), (Ct, "Ct")):
        _check_cuda(t, nm, io)
    if not (x.dtype == delta.dtype == Bt.dtype == Ct.dtype):
        raise TypeError("x, delta, Bt, Ct must share one dtype")
    _check_cuda(A, "A", (torch.float32,))
    if Dskip is not None:
        _check_cuda(Dskip, "Dskip", (torch.float32,))
    if x.dim() != 3 or A.dim() != 2:
        raise ValueError("x must be (B, L, D) and A (D, N)")
    B, L, D = x.shape
    N = A.shape[1]
    if delta.shape != x.shape or Bt.shape != (B, L, N) or Ct.shape != (B, L, N) or A.shape[0] != D:
        raise ValueError("shape mismatch between x, delta, Bt, Ct, A")
    if Dskip is not None and Dskip.shape != (D,):
        raise ValueError("Dskip must be (D,)")
    if y is None:
        y = torch.empty_like(x)
    _check_cuda(y, "y", (x.dtype,))
    if y.shape != x.shape:
        raise ValueError("y must match x")
    io_dtype = SS_BF16 if x.dtype == torch.bfloat16 else SS_F32
    sh = _stream_handle(stream, x.device)
    need = ss_selective_scan_workspace_bytes(B, L, D, N, io_dtype, bidir)
    if workspace is None and need:
        key = (fn_name, B, L, D, N, io_dtype, need, _plan_generation)
        workspace = _cached_workspace(key, need, x.device, sh)
    wsb = workspace.numel() if workspace is not None else 0
    if state is not None:  # (h0, h_last) of the forward-with-state call
        h0, h_last = state
        for t, nm in ((h0, "h0"), (h_last, "h_last")):
            if t is not None:
                _check_cuda(t, nm, (torch.float32,))
                if tuple(t.shape) != (B, D, N):
                    raise ValueError(f"{nm} must be (B, D, N) = {(B, D, N)}")
        st = lib().ss_selective_scan_fwd_state(
            _ptr(x), _ptr(delta), _ptr(Bt), _ptr(Ct), _ptr(A), _ptr(Dskip), _ptr(h0), _ptr(y),
            _ptr(h_last), B, L, D, N, io_dtype, int(bool(delta_softplus)), _ptr(workspace), wsb, sh)
    else:
        st = getattr(lib(), fn_name)(_ptr(x), _ptr(delta), _ptr(Bt), _ptr(Ct), _ptr(A),
                                     _ptr(Dskip), _ptr(y), B, L, D, N, io_dtype,
                                     int(bool(delta_softplus)), _ptr(workspace), wsb, sh)
    if st != SS_OK:
        raise SSError(st, fn_name)
    return y


def ss_selective_scan_fwd(x, delta, Bt, Ct, A, Dskip=None, delta_softplus=False, y=None,
                          workspace=None, stream=None):
    """S6 selective-scan forward; returns y (B, L, D) in x's dtype."""
    return _s6("ss_selective_scan_fwd", x, delta, Bt, Ct, A, Dskip, delta_softplus, y,
               workspace, stream, False)


def ss_selective_scan_fwd_state(x, delta, Bt, Ct, A, Dskip=None, h0=None, delta_softplus=False,
                                y=None, h_last=None, workspace=None, stream=None):
    """S6 forward from the state h0 ((B, D, N) fp32, zeros if None); returns
    (y, h_last) with h_last (B, D, N) fp32 the state after the last step."""
    torch = _torch()
    if h_last is None:
        B, _, D = x.shape
        h_last = torch.empty((B, D, A.shape[1]), dtype=torch.float32, device=x.device)
    y = _s6("ss_selective_scan_fwd", x, delta, Bt, Ct, A, Dskip, delta_softplus, y,
            workspace, stream, False, state=(h0, h_last))
    return y, h_last


def ss_selective_scan_bidir(x, delta, Bt, Ct, A, Dskip=None, delta_softplus=False, y=None,
                            workspace=None, stream=None):
    """Bidirectional S6 (forward + time-reversed over shared dA, dBx)."""
    return _s6("ss_selective_scan_bidir", x, delta, Bt, Ct, A, Dskip, delta_softplus, y,
               workspace, stream, True)


def ss_get_device_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns (then clears) the device error word."""
    dev = workspace.device if workspace is not None else None
    sh = _stream_handle(stream, dev)
    return lib().ss_get_device_status(_ptr(workspace), sh)


def ss_selective_scan_bwd_workspace_bytes(B, L, D, N) -> int:
    return lib().ss_selective_scan_bwd_workspace_bytes(int(B), int(L), int(D), int(N))


def ss_selective_scan_bwd(x, delta, Bt, Ct, A, Dskip, dy, h0=None, dh_last=None,
                          delta_softplus=False, workspace=None, stream=None) -> dict:
    """Gradients of sum(dy * y) + sum(dh_last * h_last) for
    ss_selective_scan_fwd_state: dict with dx, ddelta (x's dtype), dA, dBt,
    dCt, dDskip, dh0 (fp32)."""
    torch = _torch()
    io = (torch.float32, torch.bfloat16)
    for t, nm in ((x, "x"), (delta, "delta"), (Bt, "Bt"), (Ct, "Ct"), (dy, "dy")):
        _check_cuda(t, nm, io)
    if not (x.dtype == delta.dtype == Bt.dtype == Ct.dtype == dy.dtype):
        raise TypeError("x, delta, Bt, Ct, dy must share one dtype")
    _check_cuda(A, "A", (torch.float32,))
    B, L, D = x.shape
    N = A.shape[1]
    if delta.shape != x.shape or dy.shape != x.shape or Bt.shape != (B, L, N) or \
            Ct.shape != (B, L, N) or A.shape != (D, N):
        raise ValueError("shape mismatch between x, delta, dy, Bt, Ct, A")
    for t, nm, shape in ((Dskip, "Dskip", (D,)), (h0, "h0", (B, D, N)),
                         (dh_last, "dh_last", (B, D, N))):
        if t is not None:
            _check_cuda(t, nm, (torch.float32,))
            if tuple(t.shape) != shape:
                raise ValueError(f"{nm} must be {shape}")
    dev = x.device
    f32 = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)
    out = {"dx": torch.empty_like(x), "ddelta": torch.empty_like(x), "dA": f32(D, N),
           "dBt": f32(B, L, N), "dCt": f32(B, L, N), "dDskip": f32(D), "dh0": f32(B, D, N)}
    io_dtype = SS_BF16 if x.dtype == torch.bfloat16 else SS_F32
    sh = _stream_handle(stream, dev)
    need = ss_selective_scan_bwd_workspace_bytes(B, L, D, N)
    if workspace is None and need:
        workspace = _cached_workspace(("ss_selective_scan_bwd", B, L, D, N, need), need, dev, sh)
    wsb = workspace.numel() if workspace is not None else 0
    st = lib().ss_selective_scan_bwd(
        _ptr(x), _ptr(delta), _ptr(Bt), _ptr(Ct), _ptr(A), _ptr(Dskip), _ptr(h0), _ptr(dy),
        _ptr(dh_last), _ptr(out["dx"]), _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dBt"]),
        _ptr(out["dCt"]), _ptr(out["dDskip"]), _ptr(out["dh0"]), B, L, D, N, io_dtype,
        int(bool(delta_softplus)), _ptr(workspace), wsb, sh)
    if st != SS_OK:
        raise SSError(st, "ss_selective_scan_bwd")
    return out


def ss_selective_scan_layer_workspace_bytes(B, L, D, N, io_dtype=SS_F32) -> int:
    return lib().ss_selective_scan_layer_workspace_bytes(int(B), int(L), int(D), int(N),
                                                         int(io_dtype))


def ss_selective_scan_layer_fwd(x, W_proj, b_delta, A, Dskip=None, y=None, workspace=None,
                                stream=None):
    """Selective-scan layer forward: delta = softplus(x W_delta^T + b_delta),
    B_t = x W_B^T, C_t = x W_C^T (W_proj (D + 2N, D), rows proj_delta |
    proj_B | proj_C), then the scan; returns y (B, L, D) in x's dtype."""
    torch = _torch()
    _check_cuda(x, "x", (torch.float32, torch.bfloat16))
    _check_cuda(W_proj, "W_proj", (x.dtype,))
    _check_cuda(b_delta, "b_delta", (torch.float32,))
    _check_cuda(A, "A", (torch.float32,))
    if Dskip is not None:
        _check_cuda(Dskip, "Dskip", (torch.float32,))
    B, L, D = x.shape
    N = A.shape[1]
    if W_proj.shape != (D + 2 * N, D) or A.shape != (D, N) or b_delta.shape != (D,):
        raise ValueError("W_proj must be (D + 2N, D), A (D, N), b_delta (D,)")
    if y is None:
        y = torch.empty_like(x)
    _check_cuda(y, "y", (x.dtype,))
    io_dtype = SS_BF16 if x.dtype == torch.bfloat16 else SS_F32
    sh = _stream_handle(stream, x.device)
    need = ss_selective_scan_layer_workspace_bytes(B, L, D, N, io_dtype)
    if workspace is None and need:
        key = ("ss_selective_scan_layer_fwd", B, L, D, N, io_dtype, need, _plan_generation)
        workspace = _cached_workspace(key, need, x.device, sh)
    wsb = workspace.numel() if workspace is not None else 0
    st = lib().ss_selective_scan_layer_fwd(_ptr(x), _ptr(W_proj), _ptr(b_delta), _ptr(A),
                                           _ptr(Dskip), _ptr(y), B, L, D, N, io_dtype,
                                           _ptr(workspace), wsb, sh)
    if st != SS_OK:
        raise SSError(st, "ss_selective_scan_layer_fwd")
    return y
